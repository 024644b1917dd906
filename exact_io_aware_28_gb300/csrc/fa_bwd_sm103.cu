// Backward attention on sm_103a tensor cores (tcgen05 + TMA), key-outer.
//
// The backward recomputes the scores and probabilities block by block from Q, K and the
// saved logsumexp instead of reading a stored P (answer page "How FlashAttention works
// for training", sections 3 and 3.1; course week 13, step 2), and forms the gradients
// by the chain rule (the answer page's printed formulas for dQ and dK are garbled; these
// are the standard ones):
//   P_ij  = exp(scale q_i.k_j - lse_i)          dV_j += sum_i P_ij dO_i
//   dP_ij = dO_i . v_j                           dS_ij = P_ij (dP_ij - D_i)
//   dK_j += scale sum_i dS_ij q_i                dQ_i += scale sum_j dS_ij k_j
// with D_i = rowsum(dO_i o O_i) precomputed by the preprocess kernel.  The scale of dQ is
// applied by the dQ-convert kernel.
//
// GB300 mapping: one CTA owns a block of 128 keys of one (batch, head) and keeps K_j, V_j
// in shared memory; it walks the 128-row query blocks i that see those keys (i >= j under
// the causal mask, mask[i][j] = 1 under a block mask), accumulating dK_j, dV_j in tensor
// memory and adding each dQ_i partial to an fp32 accumulator in global memory.
// Per query block the tensor pipe runs five MMAs (all M = 128, bf16 in, fp32 out):
//   S^T  = K_j Q_i^T   (A: K_j K-major smem,   B: Q_i K-major smem)     -> TMEM [0,128)
//   dP^T = V_j dO_i^T  (A: V_j K-major smem,   B: dO_i K-major smem)    -> TMEM [128,256)
//   dV  += P^T dO_i    (A: P^T bf16 in TMEM,   B: dO_i MN-major smem)   -> TMEM [256,256+d)
//   dK  += dS^T Q_i    (A: dS^T K-major smem,  B: Q_i MN-major smem)    -> TMEM [384,384+d)
//   dQ_i = dS K_j      (A: dS^T MN-major smem, B: K_j MN-major smem)    -> TMEM [128,128+d)
// Warps: 0 TMA producer (K_j, V_j once; Q_i, dO_i through a two-stage ring), 1 MMA issuer,
// 2 tensor-memory allocation, 4-7 one thread per key row forming P^T and dS^T, 8-11 one
// thread per query row adding dQ_i to the accumulator with vector atomics.
// Every mbarrier wait is bounded; on expiry the CTA records FA_ERR_TIMEOUT and exits.
#include <cuda.h>
#include <math.h>

#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kBlk = 128;
constexpr int kSub = 128 * 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 384;

template <int D>
struct Cfg {
  static constexpr int NSUB = D / 64;
  static constexpr int TILE = NSUB * kSub;         // one 128 x d bf16 tile
  static constexpr int NSTAGE = 2;                 // Q_i / dO_i ring
  static constexpr int DS = 2 * kSub;              // dS^T, 128 x 128 bf16
  static constexpr int SMEM = 1024 + 2 * TILE + NSTAGE * 2 * TILE + DS + 1024 + 256;
};

struct Bars {
  uint64_t kv_full;
  uint64_t qdo_full[2];
  uint64_t qdo_empty[2];
  uint64_t s_full;
  uint64_t ps_ready;
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t ds_free;
  uint64_t acc_done;
  uint64_t stats_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: waits that must not be cut short by an abort
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Unit {
  int bh, j, L, nb, nq;
};

__device__ __forceinline__ bool need(const Problem& p, const Unit& u, int i) {
  if (u.j * kBlk >= u.L) return false;
  if (p.causal && i < u.j) return false;
  if (p.blockmask && !p.blockmask[i * u.nb + u.j]) return false;
  return true;
}

__device__ __forceinline__ int next_q(const Problem& p, const Unit& u, int i) {
  for (++i; i < u.nq; ++i)
    if (need(p, u, i)) return i;
  return -1;
}

// Byte offset of bf16 element (row, col) in a [rows][128] tile stored as two 128B-swizzled
// [rows][64] subtiles (16-byte chunk c of row r lands in chunk c ^ (r % 8)).
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  const int sub = col >> 6, chunk = (col & 63) >> 3;
  return sub * kSub + (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4) +
         ((col & 7) << 1);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_sm103_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                 const float* __restrict__ lse, const float* __restrict__ Dsum,
                 float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dk,
                 __nv_bfloat16* __restrict__ dv, Problem p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = base;
  uint8_t* sV = sK + C::TILE;
  uint8_t* sQ = sV + C::TILE;                  // [NSTAGE][Q tile, dO tile]
  uint8_t* sDS = sQ + C::NSTAGE * 2 * C::TILE;
  float* sL = reinterpret_cast<float*>(sDS + C::DS);   // [128] lse * log2(e) (or +inf)
  float* sD = sL + kBlk;                               // [128] D
  Bars* bars = reinterpret_cast<Bars*>(sD + kBlk);
  volatile int* abort_flag = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bhs = p.B * p.H;
  Unit u;
  u.bh = blockIdx.x % bhs;
  u.j = blockIdx.x / bhs;           // key block; small j first (most query blocks under causal)
  u.nb = (p.N + kBlk - 1) / kBlk;
  u.nq = u.nb;
  {
    int L = p.N;
    if (p.kv_len) {
      L = p.kv_len[u.bh / p.H];
      L = L < 0 ? 0 : (L > p.N ? p.N : L);
    }
    u.L = L;
  }

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->qdo_full[s], 1);
      mbar_init(&bars->qdo_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->ps_ready, kBlk);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, kBlk);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->stats_full, kBlk);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->never = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = bars->tmem_base;
  const int first = next_q(p, u, -1);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && first >= 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mdo);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::TILE);
      for (int s = 0; s < C::NSUB; ++s) {
        tma_load_3d(sK + s * kSub, &mk, &bars->kv_full, 64 * s, u.j * kBlk, u.bh);
        tma_load_3d(sV + s * kSub, &mv, &bars->kv_full, 64 * s, u.j * kBlk, u.bh);
      }
      int stage = 0, round = 0;
      for (int i = first; i >= 0; i = next_q(p, u, i)) {
        if (!mbar_wait(&bars->qdo_empty[stage], (round & 1) ^ 1, abort_flag, p.err, p.wait_ns))
          break;
        mbar_arrive_expect_tx(&bars->qdo_full[stage], 2 * C::TILE);
        uint8_t* dst = sQ + stage * 2 * C::TILE;
        for (int s = 0; s < C::NSUB; ++s) {
          tma_load_3d(dst + s * kSub, &mq, &bars->qdo_full[stage], 64 * s, i * kBlk, u.bh);
          tma_load_3d(dst + C::TILE + s * kSub, &mdo, &bars->qdo_full[stage], 64 * s, i * kBlk,
                      u.bh);
        }
        if (++stage == C::NSTAGE) {
          stage = 0;
          ++round;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && first >= 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t idKN = idesc_bf16(128, D, false, true);     // dV, dK (B MN-major)
      constexpr uint32_t idMN = idesc_bf16(128, D, true, true);      // dQ (A, B MN-major)
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aDS = smem_u32(sDS);
      bool ok = mbar_wait(&bars->kv_full, 0, abort_flag, p.err, p.wait_ns);
      tc_fence_after();
      int stage = 0, round = 0, n = 0;
      for (int i = first; ok && i >= 0; i = next_q(p, u, i)) {
        ok = mbar_wait(&bars->qdo_full[stage], round & 1, abort_flag, p.err, p.wait_ns);
        tc_fence_after();
        if (!ok) break;
        const uint32_t aQ = smem_u32(sQ + stage * 2 * C::TILE);
        const uint32_t aDO = aQ + C::TILE;
        // S^T = K_j Q_i^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSub + (kk & 3) * 32;
          mma_ss(tb, sw128_desc(aK + off, 16, 1024), sw128_desc(aQ + off, 16, 1024), idSS, kk > 0);
        }
        // dP^T = V_j dO_i^T into the columns the previous dQ partial occupied.
        if (n > 0) {
          ok = mbar_wait(&bars->dq_free, (n - 1) & 1, abort_flag, p.err, p.wait_ns);
          tc_fence_after();
          if (!ok) break;
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSub + (kk & 3) * 32;
          mma_ss(tb + 128, sw128_desc(aV + off, 16, 1024), sw128_desc(aDO + off, 16, 1024), idSS,
                 kk > 0);
        }
        mma_commit(&bars->s_full);
        ok = mbar_wait(&bars->ps_ready, n & 1, abort_flag, p.err, p.wait_ns);
        tc_fence_after();
        if (!ok) break;
        // dV += P^T dO_i ; dK += dS^T Q_i ; dQ_i = dS K_j
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ts(tb + 256, tb + 8 * kk, sw128_desc(aDO + 2048 * kk, kSub, 1024), idKN,
                 (n > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ss(tb + 384, sw128_desc(aDS + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024),
                 sw128_desc(aQ + 2048 * kk, kSub, 1024), idKN, (n > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ss(tb + 128, sw128_desc(aDS + 2048 * kk, kSub, 1024),
                 sw128_desc(aK + 2048 * kk, kSub, 1024), idMN, kk > 0);
        mma_commit(&bars->dq_full);
        mma_commit(&bars->ds_free);
        mma_commit(&bars->qdo_empty[stage]);
        if (++stage == C::NSTAGE) {
          stage = 0;
          ++round;
        }
        ++n;
      }
      mma_commit(&bars->acc_done);
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, &bars->never, nullptr, p.wait_ns);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ P^T and dS^T (key rows)
    const int r = ((warp & 3) << 5) + lane;     // key row within the block = TMEM lane
    const int key = u.j * kBlk + r;
    const bool key_live = key < u.L;
    const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) << 5) << 16);
    const float c = p.scale * kLog2e;
    const size_t row_off = static_cast<size_t>(u.bh) * p.N;
    bool ok = true;
    int n = 0;
    for (int i = first; ok && i >= 0; i = next_q(p, u, i)) {
      // The previous dS^T has been read by its dK and dQ MMAs; that also means every
      // thread of this warpgroup has finished with the previous block's statistics.
      if (n > 0) {
        ok = mbar_wait_warp(&bars->ds_free, (n - 1) & 1, abort_flag, p.err, p.wait_ns);
        if (!ok) break;
      }
      // Column statistics of this query block: lse * log2(e) (+inf where the row is
      // outside the sequence or sees no key, so that P = 0 there) and D.
      {
        const int qrow = i * kBlk + r;
        float l2 = INFINITY, dd = 0.f;
        if (qrow < p.N) {
          const float lv = lse[row_off + qrow];
          l2 = lv == -INFINITY ? INFINITY : lv * kLog2e;
          dd = Dsum[row_off + qrow];
        }
        sL[r] = l2;
        sD[r] = dd;
        mbar_arrive(&bars->stats_full);
        ok = mbar_wait_warp(&bars->stats_full, n & 1, abort_flag, p.err, p.wait_ns);
        if (!ok) break;
      }
      ok = mbar_wait_warp(&bars->s_full, n & 1, abort_flag, p.err, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const bool diag = p.causal && i == u.j;
      const int lim = diag ? r : 0;   // diagonal block: query column q sees key r iff q >= r
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sv[32], dpv[32];
        tmem_ld32(lane_base + cc * 32, sv);
        tmem_ld32(lane_base + 128 + cc * 32, dpv);
        tmem_wait_ld();
        uint32_t pp[16], dsp[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int q0 = cc * 32 + e;
          float pa = ex2(fmaf(__uint_as_float(sv[e]), c, -sL[q0]));
          float pb = ex2(fmaf(__uint_as_float(sv[e + 1]), c, -sL[q0 + 1]));
          if (!key_live || q0 < lim) pa = 0.f;
          if (!key_live || q0 + 1 < lim) pb = 0.f;
          const float da = pa * (__uint_as_float(dpv[e]) - sD[q0]);
          const float db = pb * (__uint_as_float(dpv[e + 1]) - sD[q0 + 1]);
          pp[e >> 1] = pack_bf16x2(pa, pb);
          dsp[e >> 1] = pack_bf16x2(da, db);
        }
        // P^T over the already-read S^T columns [16cc, 16cc + 16).
        tmem_st16(lane_base + cc * 16, pp);
        // dS^T row r, columns 32cc .. 32cc + 31, into the swizzled shared tile.
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 w = make_uint4(dsp[4 * g], dsp[4 * g + 1], dsp[4 * g + 2], dsp[4 * g + 3]);
          *reinterpret_cast<uint4*>(sDS + sw128_offset(r, cc * 32 + 8 * g)) = w;
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->ps_ready);
      ++n;
    }
    // ------------------------------------------------------------ dK, dV epilogue
    if (ok && n > 0) {
      ok = mbar_wait_warp(&bars->acc_done, 0, abort_flag, p.err, p.wait_ns);
      tc_fence_after();
    }
    // TMEM loads are warp-collective: every lane loads, only rows inside the sequence store.
    if (ok) {
      const bool store = key < p.N;
      __nv_bfloat16* dkrow = dk + (row_off + key) * D;
      __nv_bfloat16* dvrow = dv + (row_off + key) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t a[32], b[32];
        if (n > 0) {
          tmem_ld32(lane_base + 384 + cc * 32, a);
          tmem_ld32(lane_base + 256 + cc * 32, b);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = b[e] = 0u;
        }
        if (!store) continue;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 wk, wv;
          wk.x = pack_bf16x2(__uint_as_float(a[8 * g]) * p.scale, __uint_as_float(a[8 * g + 1]) * p.scale);
          wk.y = pack_bf16x2(__uint_as_float(a[8 * g + 2]) * p.scale, __uint_as_float(a[8 * g + 3]) * p.scale);
          wk.z = pack_bf16x2(__uint_as_float(a[8 * g + 4]) * p.scale, __uint_as_float(a[8 * g + 5]) * p.scale);
          wk.w = pack_bf16x2(__uint_as_float(a[8 * g + 6]) * p.scale, __uint_as_float(a[8 * g + 7]) * p.scale);
          wv.x = pack_bf16x2(__uint_as_float(b[8 * g]), __uint_as_float(b[8 * g + 1]));
          wv.y = pack_bf16x2(__uint_as_float(b[8 * g + 2]), __uint_as_float(b[8 * g + 3]));
          wv.z = pack_bf16x2(__uint_as_float(b[8 * g + 4]), __uint_as_float(b[8 * g + 5]));
          wv.w = pack_bf16x2(__uint_as_float(b[8 * g + 6]), __uint_as_float(b[8 * g + 7]));
          *reinterpret_cast<uint4*>(dkrow + cc * 32 + 8 * g) = wk;
          *reinterpret_cast<uint4*>(dvrow + cc * 32 + 8 * g) = wv;
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ partials (query rows)
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) << 5) << 16);
    bool ok = true;
    int n = 0;
    for (int i = first; ok && i >= 0; i = next_q(p, u, i)) {
      ok = mbar_wait_warp(&bars->dq_full, n & 1, abort_flag, p.err, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const int qrow = i * kBlk + r;
      float* dst = dq_acc + (static_cast<size_t>(u.bh) * p.N + qrow) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(lane_base + 128 + cc * 32, v);
        tmem_wait_ld();
        if (qrow < p.N) {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            atomicAdd(reinterpret_cast<float4*>(dst + cc * 32 + 4 * g),
                      make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                  __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3])));
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      ++n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (bars->abort && tid == 0) {
    // Let any bulk copy still in flight land before the CTA's shared memory is released.
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) {
    }
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

template <int D>
cudaError_t bwd_launch(const Problem& p, const void* q, const void* k, const void* v,
                       const float* lse, const void* dO, const float* Dsum, float* dq_acc,
                       void* dk, void* dv, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mdo;
  const int BH = p.B * p.H;
  if (!make_head_map(&mq, q, BH, p.N, D) || !make_head_map(&mk, k, BH, p.N, D) ||
      !make_head_map(&mv, v, BH, p.N, D) || !make_head_map(&mdo, dO, BH, p.N, D))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bwd_sm103_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int nkb = (p.N + kBlk - 1) / kBlk;
  dim3 grid(static_cast<unsigned>(BH) * nkb);
  bwd_sm103_kernel<D><<<grid, kThreads, Cfg<D>::SMEM, s>>>(
      mq, mk, mv, mdo, lse, Dsum, dq_acc, static_cast<__nv_bfloat16*>(dk),
      static_cast<__nv_bfloat16*>(dv), p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_sm103(const Problem& p, const void* q, const void* k, const void* v,
                             const float* lse, const void* dO, const float* Dsum, float* dq_acc,
                             void* dk, void* dv, cudaStream_t s) {
  return p.d == 64 ? bwd_launch<64>(p, q, k, v, lse, dO, Dsum, dq_acc, dk, dv, s)
                   : bwd_launch<128>(p, q, k, v, lse, dO, Dsum, dq_acc, dk, dv, s);
}

}  // namespace fa
