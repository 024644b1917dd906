// Decode attention on the tensor cores, d = 64 or 128: the split kernel for one new query
// token per sequence over its key/value cache with grouped key/value heads (course page
// "Week 13. GPU and FlashAttention", step 1, the bullet on attention in decode; step 2's
// online softmax).  For every key range of every (sequence, key/value head) it writes the
// unnormalised output of each query head with its running maximum and sum; the combine
// kernel of fa_decode.cu merges the ranges.
//
// Why tensor cores for a stream.  Per key the step does 2 G d multiply-adds on 4 d bytes of
// K and V; on CUDA cores that means converting every bf16 element to fp32 and about two
// FMAs per byte, which keeps the issue slots busy before HBM is.  Here the two products run
// as tcgen05 MMAs on tiles of 128 keys, with the G query heads padded to N = 16:
//   S^T = K Q^T     A = K tile [128 keys][d] (K-major, TMA 128B swizzle),
//                   B = Q rows of the group [16][d] (K-major)        -> TMEM, lane = key
//   O^T += V^T P^T  A = V tile read MN-major (the same TMA layout),
//                   B = P^T [16][128 keys] bf16 (K-major)           -> TMEM, lane = d
// and the CUDA cores only run the softmax of 128 x G scores per tile.  The second product
// always has M = 128: with d = 64 the second 64-row group of its A operand is a zeroed
// shared-memory block, and the rows of O^T it produces are never read.
//
// Work and roles.  A unit is (sequence b, key/value head g, key range of `chunk` keys); a
// persistent grid of at most one CTA per SM takes units blockIdx.x, + gridDim.x, ... and
// streams their tiles through one pipeline:
//   warp 0      TMA producer: the unit's 16 query rows (rows past the group are other heads'
//               or zero and only feed ignored columns), then K and V tiles through 3 (d =
//               128) or 4 (d = 64) stages;
//   warp 1      MMA issuer: S^T(n+1) is issued before O^T += V^T P^T(n) so that the scores of
//               the next tile form while the softmax works on this one;
//   warp 2      tensor-memory allocation (S^T x 2 [0,32), O^T x 2 [32,64));
//   warps 4-7   softmax, thread = key row: a CTA-wide maximum per head through an mbarrier
//               exchange, P = 2^(s c - m) as bf16 into the P^T tile, running sums per thread;
//               rows past the range (which may hold anything, even NaN) are masked in S and
//               zeroed in the V tile before the product reads it; O^T is rescaled in TMEM
//               only when a head's maximum grows by more than 2^8.
// Every wait is bounded; on expiry the CTA records FA_ERR_TIMEOUT and leaves.
#include <atomic>

#include <cuda.h>
#include <math.h>

#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kKeys = 128;                    // keys per tile
constexpr int kN = 16;                        // query heads padded to the MMA's N
constexpr int kMaxStages = 4;
constexpr int kSub = kKeys * 128;             // [128 rows][64 bf16] swizzled subtile, 16 KB
constexpr int kPBytes = 2 * kN * 128;         // [16][128 keys] bf16
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

struct Bars {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t p_free[2];
  uint64_t o_full[2];
  uint64_t xmax[2];
  uint64_t xsum[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: the drain wait must not be cut short by an abort
};

template <int D>
struct TC {
  static constexpr int NSUB = D / 64;                  // 64-column subtiles of a K or V tile
  static constexpr int STAGES = D == 128 ? 3 : 4;
  static constexpr int STAGE = 2 * NSUB * kSub;        // K tile then V tile
  static constexpr int PAD = D == 128 ? 0 : kSub;      // zero rows d = 64..127 of V^T
  static constexpr int QBYTES = NSUB * kN * 128;       // [16][d] bf16
  static constexpr int PSTRIDE = D + 4;                // floats per (split, head) partial row
  static constexpr int SMEM = 1024 + STAGES * STAGE + PAD + 2 * QBYTES + 2 * kPBytes +
                              2 * 4 * 8 * 4 * 2 + static_cast<int>(sizeof(Bars));
  static_assert(STAGES <= kMaxStages && SMEM <= 227 * 1024, "shared memory");
};

// The sequence of units and tiles every role walks in the same order.
struct Cursor {
  int bg, split;  // (sequence, key/value head) pair and key range of the unit
  int k0, k1;     // the unit's keys [k0, k1)
  int ntiles;
};

__device__ __forceinline__ void load_unit(Cursor& c, int u, int splits, int chunk, int Hkv,
                                          int Lmax, const int32_t* cache_len) {
  c.bg = u / splits;
  c.split = u % splits;
  const int b = c.bg / Hkv;
  int L = Lmax;
  if (cache_len) {
    L = cache_len[b];
    L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
  }
  c.k0 = c.split * chunk;
  c.k1 = min(c.k0 + chunk, L);
  c.ntiles = c.k1 > c.k0 ? (c.k1 - c.k0 + kKeys - 1) / kKeys : 0;
}

// Byte offset of element (row h, column r) in a [16][128] bf16 K-major operand tile stored as
// two 128B-swizzled [16][64] subtiles.
__device__ __forceinline__ uint32_t nk_offset(int h, int r) {
  return static_cast<uint32_t>((r >> 6) * (kN * 128) + (h >> 3) * 1024 + (h & 7) * 128 +
                               ((((r & 63) >> 3) ^ (h & 7)) << 4) + (r & 7) * 2);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                 const __grid_constant__ CUtensorMap mq, const int32_t* __restrict__ cache_len,
                 int Hq, int Hkv, int Lmax, int splits, int chunk, int units, float c,
                 float* __restrict__ part, int* err, unsigned long long wait_ns) {
  using C = TC<D>;
  constexpr int kStages = C::STAGES, kStage = C::STAGE, kQBytes = C::QBYTES;
  constexpr int kPStride = C::PSTRIDE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sKV = base;                                   // [kStages][K subtiles, V subtiles]
  uint8_t* sPad = sKV + kStages * kStage;                // d = 64: [128 keys][64] zeros
  uint8_t* sQ = sPad + C::PAD;                           // [2][kQBytes]
  uint8_t* sP = sQ + 2 * kQBytes;                        // [2][kPBytes]
  float* red_m = reinterpret_cast<float*>(sP + 2 * kPBytes);   // [2][4 warps][8 heads]
  float* red_l = red_m + 2 * 4 * 8;                            // [2][4 warps][8 heads]
  Bars* bars = reinterpret_cast<Bars*>(red_l + 2 * 4 * 8);
  volatile int* abort_flag = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
      mbar_init(&bars->p_free[i], 1);
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->xmax[i], 128);
      mbar_init(&bars->xsum[i], 128);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->never = 0;
    fence_mbar_init();
  }
  if constexpr (C::PAD > 0) {
    for (int i = tid; i < C::PAD / 16; i += kThreads)
      reinterpret_cast<uint4*>(sPad)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();   // read by the tensor cores
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      tma_prefetch_desc(&mq);
      bool ok = true;
      int n = 0, nu = 0;
      Cursor cu;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        load_unit(cu, u, splits, chunk, Hkv, Lmax, cache_len);
        if (cu.ntiles == 0) continue;
        const int qb = nu & 1;
        if (nu >= 2) {
          ok = mbar_wait(&bars->q_empty[qb], ((nu >> 1) - 1) & 1, abort_flag, err, wait_ns);
          if (!ok) break;
        }
        const int b = cu.bg / Hkv, g = cu.bg % Hkv;
        mbar_arrive_expect_tx(&bars->q_full[qb], kQBytes);
        for (int s = 0; s < C::NSUB; ++s)
          tma_load_3d(sQ + qb * kQBytes + s * (kN * 128), &mq, &bars->q_full[qb], 64 * s,
                      b * Hq + g * G, 0);
        for (int t = 0; t < cu.ntiles; ++t, ++n) {
          const int st = n % kStages;
          if (n >= kStages) {
            ok = mbar_wait(&bars->empty[st], ((n / kStages) - 1) & 1, abort_flag, err, wait_ns);
            if (!ok) break;
          }
          uint8_t* dst = sKV + st * kStage;
          mbar_arrive_expect_tx(&bars->full[st], kStage);
          const int row = cu.k0 + t * kKeys;
          for (int s = 0; s < C::NSUB; ++s) {
            tma_load_3d(dst + s * kSub, &mk, &bars->full[st], 64 * s, row, cu.bg);
            tma_load_3d(dst + (C::NSUB + s) * kSub, &mv, &bars->full[st], 64 * s, row, cu.bg);
          }
        }
        ++nu;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, kN, false, false);
      constexpr uint32_t idO = idesc_bf16(128, kN, true, false);
      bool ok = true;
      // The flattened tile sequence, with the unit of each tile.
      Cursor cur, nxt;
      int cur_t = 0, nxt_t = 0, n = 0, nu_cur = -1, nu_nxt = -1;
      int u_next = blockIdx.x;
      auto next_tile = [&](Cursor& cc, int& t, int& nu) -> bool {
        // Advance (cc, t) to the next tile; false at the end.  nu counts units with tiles.
        if (nu >= 0 && t + 1 < cc.ntiles) {
          ++t;
          return true;
        }
        for (; u_next < units; u_next += gridDim.x) {
          load_unit(cc, u_next, splits, chunk, Hkv, Lmax, cache_len);
          if (cc.ntiles > 0) {
            u_next += gridDim.x;
            t = 0;
            ++nu;
            return true;
          }
        }
        return false;
      };
      // S^T of tile m (unit cursor cc, tile t of it, unit ordinal nu) into S buffer m & 1.
      auto issue_s = [&](const Cursor& cc, int t, int nu, int m) -> bool {
        const int st = m % kStages;
        if (t == 0) {
          if (!mbar_wait(&bars->q_full[nu & 1], (nu >> 1) & 1, abort_flag, err, wait_ns))
            return false;
        }
        if (!mbar_wait(&bars->full[st], (m / kStages) & 1, abort_flag, err, wait_ns)) return false;
        tc_fence_after();
        const uint64_t dK = sw128_desc(smem_u32(sKV + st * kStage), 16, 1024);
        const uint64_t dQ = sw128_desc(smem_u32(sQ + (nu & 1) * kQBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t offA = static_cast<uint64_t>(((kk >> 2) * kSub + (kk & 3) * 32) >> 4);
          const uint64_t offB = static_cast<uint64_t>(((kk >> 2) * (kN * 128) + (kk & 3) * 32) >> 4);
          mma_ss(tb + (m & 1) * kN, dK + offA, dQ + offB, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[m & 1]);
        if (t == cc.ntiles - 1) mma_commit(&bars->q_empty[nu & 1]);
        return true;
      };
      bool have = next_tile(cur, cur_t, nu_cur);
      if (have) ok = issue_s(cur, cur_t, nu_cur, 0);
      while (ok && have) {
        nxt = cur;
        nxt_t = cur_t;
        nu_nxt = nu_cur;
        const bool have_next = next_tile(nxt, nxt_t, nu_nxt);
        if (have_next) {
          ok = issue_s(nxt, nxt_t, nu_nxt, n + 1);
          if (!ok) break;
        }
        ok = mbar_wait(&bars->p_full[n & 1], (n >> 1) & 1, abort_flag, err, wait_ns);
        if (!ok) break;
        tc_fence_after();
        const int st = n % kStages;
        // A = V^T, M = 128: the second group of 64 rows is the next 64 columns of V (d =
        // 128) or the zero block (d = 64), LBO bytes further on.
        const uint32_t aV = smem_u32(sKV + st * kStage + C::NSUB * kSub);
        const uint32_t lbo = C::PAD > 0 ? smem_u32(sPad) - aV : static_cast<uint32_t>(kSub);
        const uint64_t dV = sw128_desc(aV, lbo, 1024);
        const uint64_t dP = sw128_desc(smem_u32(sP + (n & 1) * kPBytes), 16, 1024);
        const uint32_t tO = tb + 32 + (nu_cur & 1) * kN;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t offA = static_cast<uint64_t>((2048 * kk) >> 4);
          const uint64_t offB = static_cast<uint64_t>(((kk >> 2) * (kN * 128) + (kk & 3) * 32) >> 4);
          mma_ss(tO, dV + offA, dP + offB, idO, (cur_t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->p_free[n & 1]);
        mma_commit(&bars->empty[st]);
        if (cur_t == cur.ntiles - 1) mma_commit(&bars->o_full[nu_cur & 1]);
        cur = nxt;
        cur_t = nxt_t;
        nu_cur = nu_nxt;
        have = have_next;
        ++n;
      }
      // Every MMA issued has completed before tensor memory is released.
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, &bars->never, nullptr, wait_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax (thread = key row)
    const int w4 = warp & 3;
    const int r = 32 * w4 + lane;
    const uint32_t lane_base = tb + (static_cast<uint32_t>(32 * w4) << 16);
    bool ok = true;
    int n = 0, nu = 0;
    Cursor cu;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      load_unit(cu, u, splits, chunk, Hkv, Lmax, cache_len);
      float* out = part + (static_cast<size_t>(cu.bg) * splits + cu.split) * G * kPStride;
      if (cu.ntiles == 0) {  // a range past the sequence's cache: an empty partial
        for (int i = r; i < G * kPStride; i += 128) {
          const int col = i % kPStride;
          out[i] = col == D ? -INFINITY : 0.f;
        }
        continue;
      }
      float m_run[G], l_run[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
      }
      for (int t = 0; t < cu.ntiles; ++t, ++n) {
        const int valid = min(kKeys, cu.k1 - (cu.k0 + t * kKeys));
        ok = mbar_wait_warp(&bars->s_full[n & 1], (n >> 1) & 1, abort_flag, err, wait_ns);
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[16];
        tmem_ld16(lane_base + (n & 1) * kN, sv);
        tmem_wait_ld();
        float x[G];
#pragma unroll
        for (int h = 0; h < G; ++h) x[h] = r < valid ? __uint_as_float(sv[h]) * c : -INFINITY;
        // CTA-wide maximum per head: warp maxima through shared memory and an mbarrier.
        float* rm = red_m + (n & 1) * 32;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float v = x[h];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
          if (lane == 0) rm[w4 * 8 + h] = v;
        }
        mbar_arrive(&bars->xmax[n & 1]);
        ok = mbar_wait_warp(&bars->xmax[n & 1], (n >> 1) & 1, abort_flag, err, wait_ns);
        if (!ok) break;
        float alpha[G], muse[G];
        bool grow = false;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mt = fmaxf(fmaxf(rm[h], rm[8 + h]), fmaxf(rm[16 + h], rm[24 + h]));
          const float mn = mt > m_run[h] + kRescaleThreshold ? mt : m_run[h];
          const bool ch = mn != m_run[h];
          alpha[h] = ch ? ex2(m_run[h] - mn) : 1.f;   // m_run = -inf gives 0
          grow |= ch;
          m_run[h] = mn;
          muse[h] = mn == -INFINITY ? 0.f : mn;
        }
        // P^T into this tile's P buffer once the product two tiles back has read it.
        if (n >= 2) {
          ok = mbar_wait_warp(&bars->p_free[n & 1], ((n >> 1) - 1) & 1, abort_flag, err, wait_ns);
          if (!ok) break;
        }
        uint8_t* pt = sP + (n & 1) * kPBytes;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = ex2(x[h] - muse[h]);   // x = -inf gives 0
          l_run[h] = l_run[h] * alpha[h] + p;
          *reinterpret_cast<__nv_bfloat16*>(pt + nk_offset(h, r)) = __float2bfloat16_rn(p);
        }
        if (r >= valid) {  // a row past the range: zero its V so that 0 x (anything) stays 0
          uint8_t* vt = sKV + (n % kStages) * kStage + C::NSUB * kSub;
#pragma unroll
          for (int s = 0; s < C::NSUB; ++s)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(vt + s * kSub + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
        // Rescale the running O^T (lane = d) when a maximum moved after the first tile; the
        // product of the previous tile must have completed.
        if (grow && t > 0) {
          ok = mbar_wait_warp(&bars->p_free[(n - 1) & 1], ((n - 1) >> 1) & 1, abort_flag, err,
                              wait_ns);
          if (!ok) break;
          tc_fence_after();
          uint32_t ov[16];
          const uint32_t oaddr = lane_base + 32 + (nu & 1) * kN;
          tmem_ld16(oaddr, ov);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < G; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
          tmem_st16(oaddr, ov);
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[n & 1]);
      }
      if (!ok) break;
      // ---- the unit's partial: O^T columns of the group's heads (lane = d), then (m, l)
      ok = mbar_wait_warp(&bars->o_full[nu & 1], (nu >> 1) & 1, abort_flag, err, wait_ns);
      if (!ok) break;
      tc_fence_after();
      uint32_t ov[16];
      tmem_ld16(lane_base + 32 + (nu & 1) * kN, ov);
      tmem_wait_ld();
      tc_fence_before();
      if (r < D) {
#pragma unroll
        for (int h = 0; h < G; ++h) out[h * kPStride + r] = __uint_as_float(ov[h]);
      }
      float* rl = red_l + (nu & 1) * 32;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float v = l_run[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) rl[w4 * 8 + h] = v;
      }
      mbar_arrive(&bars->xsum[nu & 1]);
      ok = mbar_wait_warp(&bars->xsum[nu & 1], (nu >> 1) & 1, abort_flag, err, wait_ns);
      if (!ok) break;
      if (r == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          out[h * kPStride + D] = m_run[h];
          out[h * kPStride + D + 1] = rl[h] + rl[8 + h] + rl[16 + h] + rl[24 + h];
        }
      }
      ++nu;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (bars->abort && tid == 0) {
    // Let any copy still in flight land before the CTA's shared memory is released.
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) {
    }
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tb, 64);
  }
}

template <int D, int G>
cudaError_t launch_g(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq,
                     const int32_t* cache_len, int Hq, int Hkv, int Lmax, int splits, int chunk,
                     int units, float c, float* part, int* err, unsigned long long wait_ns,
                     cudaStream_t s) {
  static std::atomic<bool> attr_set[64];  // per device; a race repeats the same call
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TC<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true);
  }
  const int grid = units < sm_count() ? units : sm_count();
  decode_tc_kernel<D, G><<<grid, kThreads, TC<D>::SMEM, s>>>(mk, mv, mq, cache_len, Hq, Hkv, Lmax, splits,
                                                    chunk, units, c, part, err, wait_ns);
  return cudaGetLastError();
}

}  // namespace

int decode_tc_splits(int B, int Hkv, int Lmax) {
  // About 48 units per SM over the grid, key ranges of whole 128-key tiles.
  const long long pairs = static_cast<long long>(B) * Hkv;
  const long long tiles = (Lmax + kKeys - 1) / kKeys;
  long long splits = (48ll * sm_count() + pairs - 1) / pairs;
  if (splits > tiles) splits = tiles;
  if (splits < 1) splits = 1;
  const long long per = (tiles + splits - 1) / splits;
  return static_cast<int>((tiles + per - 1) / per);
}

namespace {

template <int D>
cudaError_t launch_tc_d(const void* q, const void* k, const void* v, int B, int Hq, int Hkv,
                        int Lmax, const int32_t* cache_len, float scale, float* part, int splits,
                        int* err, unsigned long long wait_ns, cudaStream_t s) {
  CUtensorMap mk, mv, mq;
  if (!make_head_map_rows(&mk, k, B * Hkv, Lmax, D, kKeys) ||
      !make_head_map_rows(&mv, v, B * Hkv, Lmax, D, kKeys) ||
      !make_head_map_rows(&mq, q, 1, B * Hq, D, kN))
    return cudaErrorInvalidValue;
  const long long tiles = (Lmax + kKeys - 1) / kKeys;
  const int chunk = static_cast<int>((tiles + splits - 1) / splits) * kKeys;
  const int units = B * Hkv * splits;
  const float c = scale * kLog2e;
  switch (Hq / Hkv) {
    case 1: return launch_g<D, 1>(mk, mv, mq, cache_len, Hq, Hkv, Lmax, splits, chunk, units, c, part, err, wait_ns, s);
    case 2: return launch_g<D, 2>(mk, mv, mq, cache_len, Hq, Hkv, Lmax, splits, chunk, units, c, part, err, wait_ns, s);
    case 4: return launch_g<D, 4>(mk, mv, mq, cache_len, Hq, Hkv, Lmax, splits, chunk, units, c, part, err, wait_ns, s);
    case 8: return launch_g<D, 8>(mk, mv, mq, cache_len, Hq, Hkv, Lmax, splits, chunk, units, c, part, err, wait_ns, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_tc(const void* q, const void* k, const void* v, int B, int Hq,
                             int Hkv, int Lmax, int d, const int32_t* cache_len, float scale,
                             float* part, int splits, int* err, unsigned long long wait_ns,
                             cudaStream_t s) {
  return d == 64 ? launch_tc_d<64>(q, k, v, B, Hq, Hkv, Lmax, cache_len, scale, part, splits,
                                   err, wait_ns, s)
                 : launch_tc_d<128>(q, k, v, B, Hq, Hkv, Lmax, cache_len, scale, part, splits,
                                    err, wait_ns, s);
}

}  // namespace fa
