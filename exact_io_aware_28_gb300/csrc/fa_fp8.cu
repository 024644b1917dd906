// FP8 (e4m3) forward on sm_103a tensor cores, d = 128: the input encoders and the kernel.
//
// What it computes.  FP8 operands are what the third FlashAttention adds on Hopper (answer
// page "How FlashAttention works for training", section 7; course week 13, step 2); the
// pages give nothing beyond that.  Here both products, S = Q K^T and O += P V, take e4m3
// operands (tcgen05.mma kind::f8f6f4, fp32 accumulation in tensor memory); everything else
// is the forward of fa_fwd_sm103.cu: the running (max, sum) state per query row, O kept
// unnormalised and divided by the row sum once, the per-row logsumexp, causal / padding /
// block-mask skipping (reading guide arXiv 2205.14135, "Method", steps 1-4).
//
// Encoding.  A bf16 tensor becomes e4m3 codes and power-of-two scales s = 2^k, k the
// smallest integer with amax <= 448 * 2^k: x / s is then exact and rounding (to nearest,
// ties to even, saturating) is the only error.  Q and K carry one scale per 128-row block,
// which folds into the exponent's multiplier per score tile for free; V carries one scale
// per (b, h), applied once in the epilogue (a scale per key block would have to multiply P
// before its own rounding).
//
// V layout.  The second product needs V as a K-major operand (keys contiguous), so the V
// encoder writes V^T: [B, H, 128, Np] bytes, Np = N rounded up to 128, zero past N.  Within
// each block of 128 keys the columns are permuted: column k of the block holds key
//   pi(k) = 32 (k >> 5) + 16 ((k >> 2) & 1) + 8 ((k >> 1) & 1) + 2 ((k >> 3) & 3) + (k & 1).
// That is where the softmax threads' probabilities land when they store them with the
// 16-lane tensor-memory shape: thread t of a warp holds keys 8c + 2(t % 4) + {0, 1} of its
// two rows (c = 0..15) and packs the e4m3 pairs of chunks 2m, 2m+1 into one 32-bit word m,
// which .16x256b puts in column 8(m >> 1) + 2(t % 4) + (m & 1).  Reading byte b of column
// C as contraction index 4C + b gives exactly pi; permuting V's keys the same way keeps
// sum_k P[row, pi(k)] V[pi(k), :] = P V, with no shuffles in the softmax.
//
// Kernel roles (384 threads, one CTA = 256 query rows of one (b, h), two 128-row tiles):
//   warp 0      TMA producer: Q0, Q1 once, then K_j and V^T_j (16 KB each) through 6 stages;
//   warps 1, 3  MMA issuers for tile 0 / tile 1 (S_t = Q_t K_j^T, then O_t += P_t V_j with
//               P read from tensor memory; in-order issue keeps S_t(j+1) from overwriting
//               P_t(j) before the product has read it);
//   warp 2      tensor-memory allocation (S0 [0,128), S1 [128,256), O0 [256,384), O1
//               [384,512));
//   warps 4-11  softmax on each tile in turn, then the epilogue: O * s_v / l staged as bf16
//               in shared memory and stored with the TMA; logsumexp per row.
// O is rescaled only when a row's maximum grows by more than 2^8, so P <= 256 < 448 always
// fits e4m3.  Every mbarrier wait is bounded; on expiry the CTA records FA_ERR_TIMEOUT.
#include <atomic>

#include <cuda.h>
#include <cuda_fp8.h>
#include <math.h>

#include "fa_fwd_units.cuh"
#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;
using namespace units;

constexpr int kD = 128;
constexpr int kTile = kBlk * kD;    // bytes of a 128 x 128 e4m3 tile: one 128B-swizzled block
constexpr int kOSub = 128 * 128;    // bytes of a 128-row x 64-column bf16 output subtile
constexpr int kStages = 6;
constexpr int kThreads = 384;
constexpr int kSmem = 1024 + 2 * kTile + kStages * kTile + 2 * 2 * kOSub + 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

// ------------------------------------------------------------------ encoders

// k of the scale 2^k for a block whose largest magnitude is `amax` (finite, >= 0): the
// smallest k with amax <= 448 * 2^k, clamped to [-126, 127]; 0 for amax = 0.  With
// amax = (1 + f) 2^e and 448 = 1.75 * 2^8, k = e - 8 when 1 + f <= 1.75, else e - 7.
__device__ __forceinline__ int scale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  if (amax < 1.17549435e-38f) return -126;
  const uint32_t b = __float_as_uint(amax);
  const int e = static_cast<int>((b >> 23) & 0xFFu) - 127;
  const int k = e - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return max(-126, min(127, k));
}

__device__ __forceinline__ float pow2f(int k) {  // 2^k for k in [-126, 127]
  return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float amax8(const uint4& v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

// Largest value over the CTA (256 threads).
__device__ __forceinline__ float block_max(float m, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
  return m;
}

// Loads one 128-row x 128-column bf16 block: 2048 vectors of 8, eight per thread; rows past
// the end read as zero.
__device__ __forceinline__ void load_block(const __nv_bfloat16* head, int r0, int rows,
                                           uint4 (&v)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int idx = threadIdx.x + 256 * i, row = idx >> 4, cv = idx & 15;
    v[i] = row < rows ? __ldg(reinterpret_cast<const uint4*>(head + (size_t)(r0 + row) * kD) + cv)
                      : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Q, K: one scale per 128-row block; codes keep the [B, H, N, 128] layout.
__global__ void __launch_bounds__(256)
quant_rows_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ x8,
                  float* __restrict__ scale, int N, int nb) {
  __shared__ float red[8];
  const int blk = blockIdx.x, bh = blockIdx.y, r0 = blk * kBlk;
  const int rows = min(kBlk, N - r0);
  const size_t head = static_cast<size_t>(bh) * N * kD;
  uint4 v[8];
  load_block(x + head, r0, rows, v);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, amax8(v[i]));
  const int k = scale_exponent(block_max(m, red));
  const float inv = pow2f(-k);
  if (threadIdx.x == 0) scale[static_cast<size_t>(bh) * nb + blk] = pow2f(k);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int idx = threadIdx.x + 256 * i, row = idx >> 4, cv = idx & 15;
    if (row >= rows) continue;
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
    uint32_t w[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float2 a = __bfloat1622float2(h[2 * j]), b = __bfloat1622float2(h[2 * j + 1]);
      w[j] = e4m3x2(a.x * inv, a.y * inv) | (e4m3x2(b.x * inv, b.y * inv) << 16);
    }
    *reinterpret_cast<uint2*>(x8 + head + static_cast<size_t>(r0 + row) * kD + cv * 8) =
        make_uint2(w[0], w[1]);
  }
}

// V, pass 1: the largest magnitude of each (b, h), as the bit pattern of a non-negative
// float (ordered like unsigned integers) combined with atomicMax into amax_bits[bh] (zeroed
// by the caller).
__global__ void __launch_bounds__(256)
v_amax_kernel(const __nv_bfloat16* __restrict__ v, unsigned* __restrict__ amax_bits, int N) {
  __shared__ float red[8];
  const int blk = blockIdx.x, bh = blockIdx.y, r0 = blk * kBlk;
  const int rows = min(kBlk, N - r0);
  uint4 x[8];
  load_block(v + static_cast<size_t>(bh) * N * kD, r0, rows, x);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, amax8(x[i]));
  m = block_max(m, red);
  if (threadIdx.x == 0) atomicMax(amax_bits + bh, __float_as_uint(m));
}

// Key held by column k (0..127) of a V^T block (see the header comment).
__device__ __forceinline__ int vt_key(int k) {
  return 32 * (k >> 5) + 16 * ((k >> 2) & 1) + 8 * ((k >> 1) & 1) + 2 * ((k >> 3) & 3) + (k & 1);
}

// V, pass 2: codes of V^T with the per-head scale.  The 128 x 128 block is read with
// coalesced 16-byte loads and staged in shared memory as it lies in V ([key][dim]); thread
// task (dim, group) then reads 16 columns 16g .. 16g+15 of row `dim` of the V^T block,
// gathered from rows vt_key(column) (neighbouring lanes read neighbouring dims of one key:
// no bank conflicts), and stores them as one 16-byte word.
__global__ void __launch_bounds__(256)
v_quant_kernel(const __nv_bfloat16* __restrict__ v, uint8_t* __restrict__ vt8,
               const unsigned* __restrict__ amax_bits, int N, int Np) {
  __shared__ __align__(16) __nv_bfloat16 sv[kBlk * kD];
  const int blk = blockIdx.x, bh = blockIdx.y, r0 = blk * kBlk;
  const int rows = min(kBlk, N - r0);
  const float inv = pow2f(-scale_exponent(__uint_as_float(amax_bits[bh])));
  {
    uint4 x[8];
    load_block(v + static_cast<size_t>(bh) * N * kD, r0, rows, x);   // rows past N: zero
#pragma unroll
    for (int i = 0; i < 8; ++i)
      reinterpret_cast<uint4*>(sv)[threadIdx.x + 256 * i] = x[i];
  }
  __syncthreads();
  uint8_t* out = vt8 + static_cast<size_t>(bh) * kD * Np + static_cast<size_t>(blk) * kBlk;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int task = threadIdx.x + 256 * i, dim = task & 127, g = task >> 7;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[4];
#pragma unroll
      for (int b = 0; b < 4; ++b)
        f[b] = __bfloat162float(sv[vt_key(16 * g + 4 * q + b) * kD + dim]) * inv;
      w[q] = e4m3x2(f[0], f[1]) | (e4m3x2(f[2], f[3]) << 16);
    }
    *reinterpret_cast<uint4*>(out + static_cast<size_t>(dim) * Np + 16 * g) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// V, pass 3: the per-head scales 2^k replace the amax bit patterns.
__global__ void v_scale_kernel(float* __restrict__ scale, int BH) {
  const int bh = blockIdx.x * blockDim.x + threadIdx.x;
  if (bh < BH) scale[bh] = pow2f(scale_exponent(scale[bh]));  // amax (as a float) -> 2^k
}

// ------------------------------------------------------------------ forward kernel

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t o_staged[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

__global__ void __launch_bounds__(kThreads, 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mvt, const __grid_constant__ CUtensorMap mo,
               const float* __restrict__ q_scale, const float* __restrict__ k_scale,
               const float* __restrict__ v_scale, float* __restrict__ lse, Problem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = base;                          // [2][kTile]
  uint8_t* sKV = sQ + 2 * kTile;               // [kStages][kTile]: K_j and V^T_j alternately
  uint8_t* sO = sKV + kStages * kTile;         // [2][2][kOSub]: bf16 output staging
  Bars* bars = reinterpret_cast<Bars*>(sO + 4 * kOSub);
  volatile int* abort_flag = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Unit u = make_unit(p);
  const int jend = key_blocks(p, u);

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 2 * kBlk);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_staged[t], 2 * kBlk);
    }
    mbar_init(&bars->drain, 2);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mvt);
      mbar_arrive_expect_tx(&bars->q_full, 2 * kTile);
      for (int t = 0; t < 2; ++t)
        tma_load_3d(sQ + t * kTile, &mq, &bars->q_full, 0, u.q0 + t * kBlk, u.bh);
      int stage = 0, round = 0;
      bool ok = true;
      for (int j = next_any(p, u, -1, jend); ok && j >= 0; j = next_any(p, u, j, jend)) {
        for (int which = 0; which < 2 && ok; ++which) {
          ok = mbar_wait(&bars->kv_empty[stage], (round & 1) ^ 1, abort_flag, p.err, p.wait_ns);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars->kv_full[stage], kTile);
          if (which == 0)
            tma_load_3d(sKV + stage * kTile, &mk, &bars->kv_full[stage], 0, j * kBlk, u.bh);
          else
            tma_load_3d(sKV + stage * kTile, &mvt, &bars->kv_full[stage], j * kBlk, 0, u.bh);
          if (++stage == kStages) {
            stage = 0;
            ++round;
          }
        }
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      const int t = warp == 1 ? 0 : 1;
      constexpr uint32_t idS = idesc_e4m3(128, 128);
      constexpr uint32_t idO = idesc_e4m3(128, kD);
      constexpr uint64_t kTileD = kTile >> 4;
      // Every operand in shared memory is K-major with 128-byte rows (Q_t, K_j: a query or
      // key per row; V^T_j: a dimension per row); a K step of 32 bytes adds 2 to the start
      // address field.
      const uint64_t dQ = sw128_desc(smem_u32(sQ + t * kTile), 16, 1024);
      const uint64_t dKV = sw128_desc(smem_u32(sKV), 16, 1024);
      const uint32_t tS = tb + t * 128, tO = tb + 256 + t * 128;
      int last = -1;
      for (int j = jend - 1; j >= 0 && last < 0; --j)
        if (need(p, u, t, j)) last = j;
      int cs = 0;
      uint32_t cr = 0;
      int npv = 0;
      bool ok = mbar_wait(&bars->q_full, 0, abort_flag, p.err, p.wait_ns);
      tc_fence_after();
      auto issue_s = [&](int slot) {
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk)
          mma_ss_f8(tS, dQ + 2 * kk, dKV + slot * kTileD + 2 * kk, idS, kk > 0);
        mma_commit(&bars->s_full[t]);
      };
      int j = next_any(p, u, -1, jend);
      if (ok && j >= 0) {
        const int ks = cs;
        ok = mbar_wait(&bars->kv_full[ks], cr & 1, abort_flag, p.err, p.wait_ns);
        if (++cs == kStages) { cs = 0; ++cr; }
        tc_fence_after();
        if (ok) {
          if (need(p, u, t, j)) issue_s(ks);
          mma_commit(&bars->kv_empty[ks]);
        }
      }
      while (ok && j >= 0) {
        const int jn = next_any(p, u, j, jend);
        const int vs = cs;
        ok = mbar_wait(&bars->kv_full[vs], cr & 1, abort_flag, p.err, p.wait_ns);
        if (++cs == kStages) { cs = 0; ++cr; }
        int ks = -1;
        if (ok && jn >= 0) {
          ks = cs;
          ok = mbar_wait(&bars->kv_full[ks], cr & 1, abort_flag, p.err, p.wait_ns);
          if (++cs == kStages) { cs = 0; ++cr; }
        }
        if (!ok) break;
        tc_fence_after();
        if (need(p, u, t, j)) {
          ok = mbar_wait(&bars->p_full[t], npv & 1, abort_flag, p.err, p.wait_ns);
          tc_fence_after();
          if (!ok) break;
          // P: 32 columns of e4m3 quadruples at the start of this tile's S region.
#pragma unroll
          for (int kk = 0; kk < kBlk / 32; ++kk)
            mma_ts_f8(tO, tS + 8 * kk, dKV + vs * kTileD + 2 * kk, idO,
                      (npv > 0 || kk > 0) ? 1u : 0u);
          ++npv;
          if (j == last) mma_commit(&bars->o_done[t]);
        }
        mma_commit(&bars->kv_empty[vs]);
        if (jn >= 0) {
          if (need(p, u, t, jn)) issue_s(ks);
          mma_commit(&bars->kv_empty[ks]);
        }
        j = jn;
      }
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, &bars->never, nullptr, p.wait_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax warps
    // Warp 4 + q + 4h owns rows 32q + 16h + [0, 16) of both tiles: thread t holds rows
    // A = 32q + 16h + t/4 and B = A + 8, keys 8c + 2(t%4) + {0, 1}, c = 0..15.
    const int q4 = warp & 3, h = (warp - 4) >> 2, t4 = lane & 3;
    const int rA = 32 * q4 + 16 * h + (lane >> 2), rB = rA + 8;
    const uint32_t lane_base = tb + (static_cast<uint32_t>(32 * q4 + 16 * h) << 16);
    const float* ksc = k_scale + static_cast<size_t>(u.bh) * u.nb;
    float cq[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r0 = u.q0 + t * kBlk;
      cq[t] = r0 < p.N ? p.scale * kLog2e * q_scale[static_cast<size_t>(u.bh) * u.nb + r0 / kBlk]
                       : 0.f;
    }
    float m_run[2][2] = {{-INFINITY, -INFINITY}, {-INFINITY, -INFINITY}};
    float l_part[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    int n_t[2] = {0, 0};
    bool ok = true;
    for (int j = 0; j < jend && ok; ++j) {
      const float kj = (need(p, u, 0, j) || need(p, u, 1, j)) ? __ldg(ksc + j) : 0.f;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok || !need(p, u, t, j)) continue;
        const float c = cq[t] * kj;  // scale * log2(e) * s_q * s_k: exact powers of two apart
        const uint64_t c2 = f2_pack(c, c);
        ok = mbar_wait_warp(&bars->s_full[t], n_t[t] & 1, abort_flag, p.err, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        uint32_t v[64];
        tmem_ld_16x256b_x16_wait(lane_base + t * 128, v);
        float sv[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) sv[i] = __uint_as_float(v[i]);
        const int k0 = j * kBlk;
        const int row0 = u.q0 + t * kBlk;
        const bool edge = (p.causal && k0 + kBlk - 1 > row0) || (k0 + kBlk > u.L);
        if (edge) {
          const int lim_len = u.L - 1 - k0;
          const int limA = min(p.causal ? row0 + rA - k0 : kBlk - 1, lim_len);
          const int limB = min(p.causal ? row0 + rB - k0 : kBlk - 1, lim_len);
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const int key = 8 * cc + 2 * t4;
            if (key > limA) sv[4 * cc] = -INFINITY;
            if (key + 1 > limA) sv[4 * cc + 1] = -INFINITY;
            if (key > limB) sv[4 * cc + 2] = -INFINITY;
            if (key + 1 > limB) sv[4 * cc + 3] = -INFINITY;
          }
        }
        float ma0 = fmaxf(sv[0], sv[1]), ma1 = fmaxf(sv[4], sv[5]);
        float mb0 = fmaxf(sv[2], sv[3]), mb1 = fmaxf(sv[6], sv[7]);
#pragma unroll
        for (int cc = 2; cc < 16; cc += 2) {
          ma0 = fmax3(ma0, sv[4 * cc], sv[4 * cc + 1]);
          mb0 = fmax3(mb0, sv[4 * cc + 2], sv[4 * cc + 3]);
          ma1 = fmax3(ma1, sv[4 * cc + 4], sv[4 * cc + 5]);
          mb1 = fmax3(mb1, sv[4 * cc + 6], sv[4 * cc + 7]);
        }
        float mA = fmaxf(ma0, ma1), mB = fmaxf(mb0, mb1);
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 1));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 1));
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 2));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 2));
        mA *= c;
        mB *= c;
        const float oldA = m_run[t][0], oldB = m_run[t][1];
        const float newA = mA > oldA + kRescaleThreshold ? mA : oldA;
        const float newB = mB > oldB + kRescaleThreshold ? mB : oldB;
        const bool chA = newA != oldA, chB = newB != oldB;
        const float alphaA = chA ? ex2(oldA - newA) : 1.f;
        const float alphaB = chB ? ex2(oldB - newB) : 1.f;
        const float useA = newA == -INFINITY ? 0.f : newA;
        const float useB = newB == -INFINITY ? 0.f : newB;
        const uint64_t nA = f2_pack(-useA, -useA), nB = f2_pack(-useB, -useB);
        uint64_t accA = f2_pack(0.f, 0.f), accB = accA;
        // P as e4m3: word m of a row packs chunks 2m (low half) and 2m+1 (high half);
        // .16x256b.x4 takes row A's words m = 2r, 2r+1 in registers 4r, 4r+1 and row B's
        // in 4r+2, 4r+3.
        uint32_t pk[16];
        uint32_t wa = 0u, wb = 0u;
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const float2 xa = f2_unpack(ffma2(f2_pack(sv[4 * cc], sv[4 * cc + 1]), c2, nA));
          const float2 xb = f2_unpack(ffma2(f2_pack(sv[4 * cc + 2], sv[4 * cc + 3]), c2, nB));
          const float pa0 = ex2(xa.x), pa1 = ex2(xa.y);
          const float pb0 = ex2(xb.x), pb1 = ex2(xb.y);
          accA = fadd2(accA, f2_pack(pa0, pa1));
          accB = fadd2(accB, f2_pack(pb0, pb1));
          const uint32_t ha = e4m3x2(pa0, pa1), hb = e4m3x2(pb0, pb1);
          if ((cc & 1) == 0) {
            wa = ha;
            wb = hb;
          } else {
            const int r = cc >> 2, w = (cc >> 1) & 1;
            pk[4 * r + w] = wa | (ha << 16);
            pk[4 * r + 2 + w] = wb | (hb << 16);
          }
        }
        tmem_st_16x256b_x4(lane_base + t * 128, pk);
        const float2 sa = f2_unpack(accA), sb = f2_unpack(accB);
        l_part[t][0] = l_part[t][0] * alphaA + (sa.x + sa.y);
        l_part[t][1] = l_part[t][1] * alphaB + (sb.x + sb.y);
        m_run[t][0] = newA;
        m_run[t][1] = newB;
        if (n_t[t] > 0 && __any_sync(0xffffffffu, chA || chB)) {
#pragma unroll
          for (int half = 0; half < kD / 64; ++half) {
            uint32_t o[32];
            const uint32_t oaddr = lane_base + 256 + t * 128 + 64 * half;
            tmem_ld_16x256b_x8_wait(oaddr, o);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * ((i & 2) ? alphaB : alphaA));
            tmem_st_16x256b_x8(oaddr, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
        ++n_t[t];
      }
    }
    // ------------------------------------------------------------ epilogue
    const float s_v = v_scale[u.bh];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (ok && n_t[t] > 0) {
        ok = mbar_wait_warp(&bars->o_done[t], 0, abort_flag, p.err, p.wait_ns);
        tc_fence_after();
      }
      if (!ok) break;
      float lA = l_part[t][0], lB = l_part[t][1];
      lA += __shfl_xor_sync(0xffffffffu, lA, 1);
      lB += __shfl_xor_sync(0xffffffffu, lB, 1);
      lA += __shfl_xor_sync(0xffffffffu, lA, 2);
      lB += __shfl_xor_sync(0xffffffffu, lB, 2);
      const float invA = lA > 0.f ? s_v / lA : 0.f, invB = lB > 0.f ? s_v / lB : 0.f;
      const int rowA = u.q0 + t * kBlk + rA, rowB = rowA + 8;
      uint8_t* stage = sO + t * 2 * kOSub;
#pragma unroll
      for (int half = 0; half < kD / 64; ++half) {
        uint32_t ov[32];
        if (n_t[t] > 0) {
          tmem_ld_16x256b_x8_wait(lane_base + 256 + t * 128 + 64 * half, ov);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0u;
        }
        uint8_t* sub = stage + half * kOSub;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint32_t byte = static_cast<uint32_t>(4 * t4);
          *reinterpret_cast<uint32_t*>(sub + rA * 128 + ((cc ^ (rA & 7)) << 4) + byte) =
              pack_bf16x2(__uint_as_float(ov[4 * cc]) * invA,
                          __uint_as_float(ov[4 * cc + 1]) * invA);
          *reinterpret_cast<uint32_t*>(sub + rB * 128 + ((cc ^ (rB & 7)) << 4) + byte) =
              pack_bf16x2(__uint_as_float(ov[4 * cc + 2]) * invB,
                          __uint_as_float(ov[4 * cc + 3]) * invB);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->o_staged[t]);
      if (warp == 4 && lane == 0 && u.q0 + t * kBlk < p.N) {
        if (mbar_wait(&bars->o_staged[t], 0, abort_flag, p.err, p.wait_ns)) {
#pragma unroll
          for (int half = 0; half < kD / 64; ++half)
            tma_store_3d(&mo, stage + half * kOSub, 64 * half, u.q0 + t * kBlk, u.bh);
          bulk_commit_group();
        }
      }
      if (t4 == 0) {
        float* lrow = lse + static_cast<size_t>(u.bh) * p.N;
        if (rowA < p.N) lrow[rowA] = lA > 0.f ? (m_run[t][0] + __log2f(lA)) * kLn2 : -INFINITY;
        if (rowB < p.N) lrow[rowB] = lB > 0.f ? (m_run[t][1] + __log2f(lB)) * kLn2 : -INFINITY;
      }
    }
  }

  if (warp == 4 && lane == 0) bulk_wait_group_all();
  tc_fence_before();
  __syncthreads();
  if (bars->abort && tid == 0) {
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

}  // namespace

cudaError_t launch_fp8_quantize_rows(const void* x, void* x8, float* scale, int BH, int N,
                                     cudaStream_t s) {
  const int nb = (N + kBlk - 1) / kBlk;
  quant_rows_kernel<<<dim3(nb, BH), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                                 static_cast<uint8_t*>(x8), scale, N, nb);
  return cudaGetLastError();
}

cudaError_t launch_fp8_quantize_v(const void* v, void* vt8, float* scale, int BH, int N,
                                  cudaStream_t s) {
  const int nb = (N + kBlk - 1) / kBlk;
  cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float) * static_cast<size_t>(BH), s);
  if (e != cudaSuccess) return e;
  unsigned* bits = reinterpret_cast<unsigned*>(scale);
  v_amax_kernel<<<dim3(nb, BH), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(v), bits, N);
  v_quant_kernel<<<dim3(nb, BH), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(v),
                                              static_cast<uint8_t*>(vt8), bits, N, nb * kBlk);
  v_scale_kernel<<<(BH + 255) / 256, 256, 0, s>>>(scale, BH);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const Problem& p, const void* q8, const void* k8, const void* vt8,
                           const float* q_scale, const float* k_scale, const float* v_scale,
                           void* o, float* lse, cudaStream_t s) {
  const int BH = p.B * p.H;
  const int Np = (p.N + kBlk - 1) / kBlk * kBlk;
  CUtensorMap mq, mk, mvt, mo;
  if (!make_u8_map(&mq, q8, BH, p.N, kD) || !make_u8_map(&mk, k8, BH, p.N, kD) ||
      !make_u8_map(&mvt, vt8, BH, kD, Np) || !make_head_map(&mo, o, BH, p.N, kD))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];  // per device; a race repeats the same call
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load()) {
    cudaError_t e =
        cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true);
  }
  const int nqb = (p.N + 2 * kBlk - 1) / (2 * kBlk);
  fwd_fp8_kernel<<<dim3(static_cast<unsigned>(BH) * nqb), kThreads, kSmem, s>>>(
      mq, mk, mvt, mo, q_scale, k_scale, v_scale, lse, p);
  return cudaGetLastError();
}

}  // namespace fa
