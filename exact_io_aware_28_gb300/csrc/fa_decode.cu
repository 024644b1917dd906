// Decode attention over a key/value cache with grouped key/value heads: one new query
// token per sequence, split over the cache length, then combined.
//
// What it computes (course page "Week 13. GPU and FlashAttention", step 1, the bullet on
// attention in decode, and step 2's online softmax): query head h of sequence b reads
// key/value head g = h / G (G = Hq / Hkv query heads per key/value head) and the keys
// j < cache_len[b]; o = softmax(scale q K^T) V and lse = logsumexp(scale q K^T).  Each
// sequence has its own cache, so the step reads every cached byte once and does about G
// FLOPs per byte: it is bound by HBM bandwidth, and grouping the heads is what raises the
// work done per byte read.
//
// GB300 mapping.  Split kernel: one CTA per (key range, sequence, key/value head), 256
// threads, two CTAs per SM.  Thread 0 streams 64-key tiles of K and V into a three-stage
// ring with TMA (128-byte swizzle, mbarrier completion, bounded waits; a result that differs
// between threads is settled with a CTA-wide AND before anyone leaves the loop).  Per tile:
//   scores  -- each thread keeps a slice of d of the G queries in registers (fp32, scale *
//              log2(e) folded in) and forms partial dot products for a few keys; the
//              slices of a key are neighbouring lanes, summed by shuffles; then
//   softmax -- one warp per query head: tile maximum and sum by shuffles, running maximum
//              m and sum l, probabilities and the rescale factor into shared memory;
//   P V     -- thread (pair of output columns, group of keys) accumulates all G heads.
// This CUDA-core split kernel serves d = 64; for d = 128 the tensor-core split kernel of
// fa_decode_tc.cu runs instead (on CUDA cores the fp32 conversions and about two FMAs per
// cache byte keep the issue slots busier than HBM).  Each split writes its unnormalised
// output with (m, l) to the caller's fp32 workspace; the combine kernel merges the splits of
// each (b, h) with the same rescaling rule and writes o (bf16) and lse (fp32, natural log).
#include <cuda.h>
#include <math.h>

#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kTile = 64;                   // keys per tile
constexpr int kThreads = 256;
constexpr int kStages = 3;
constexpr int kSubBytes = kTile * 128;      // one [64 keys][64 columns] bf16 swizzled subtile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DCfg {
  static constexpr int NSUB = D / 64;
  static constexpr int TILE = NSUB * kSubBytes;   // bytes of a K (or V) tile
  static constexpr int STAGE = 2 * TILE;          // K tile then V tile
  static constexpr int NDP = D / 2;               // column pairs of the P V phase
  static constexpr int KGROUPS = kThreads / NDP;  // key groups of the P V phase: 4 or 8
  static constexpr int KPER = kTile / KGROUPS;    // keys per P V thread: 16 or 8
  static constexpr int PSTRIDE = D + 4;           // floats per (split, head) partial row
};

// Score-phase split of d: each thread keeps its slice of the G queries in registers (at most
// 64 floats) and serves KPT keys; the NPART slices of a key are neighbouring lanes.
template <int D, int G>
struct SCfg {
  static constexpr int NPART = (D * G / 64) > 4 ? (D * G / 64) : 4;
  static constexpr int DPART = D / NPART;   // 64 .. 8 columns
  static constexpr int KPW = 32 / NPART;    // keys per warp pass
  static constexpr int KPT = NPART / 4;     // keys per thread per 64-key tile
  static_assert(DPART % 8 == 0 && KPW * KPT * 8 == kTile, "score split");
};

struct DBars {
  uint64_t full[kStages];
  int abort;
};

// Byte offset of bf16 element (row, col) in a tile of 128-byte-swizzled [64][64] subtiles.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return static_cast<uint32_t>((col >> 6) * kSubBytes + row * 128 +
                               ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1));
}

// A pair of bf16 (low element first) as two floats.
__device__ __forceinline__ float2 bf2f(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int D, int G>
constexpr int decode_smem_bytes() {
  using C = DCfg<D>;
  return 1024 + kStages * C::STAGE + 4 * (2 * kTile * G + 8) + static_cast<int>(sizeof(DBars));
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2)
decode_split_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ cache_len,
                    int Hq, int Hkv, int Lmax, int splits, int chunk, float c,
                    float* __restrict__ part, int* err, unsigned long long wait_ns) {
  using C = DCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
  float* sp = reinterpret_cast<float*>(stages + kStages * C::STAGE);  // [kTile][G] scores
  float* pb = sp + kTile * G;                                         // [kTile][G]
  float* alpha_s = pb + kTile * G;                                    // [G] (8 slots)
  DBars* bars = reinterpret_cast<DBars*>(alpha_s + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bg = blockIdx.y;
  const int b = bg / Hkv, g = bg % Hkv;
  int L = Lmax;
  if (cache_len) {
    L = cache_len[b];
    L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
  }
  const int k0 = split * chunk;
  const int k1 = min(k0 + chunk, L);
  const int ntiles = k1 > k0 ? (k1 - k0 + kTile - 1) / kTile : 0;

  // This thread's slice of the G queries, scaled by scale * log2(e), kept in registers.
  using S = SCfg<D, G>;
  const int spart = lane % S::NPART;
  float qr[G][S::DPART];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const __nv_bfloat16* qh = q + (static_cast<size_t>(b) * Hq + g * G + h) * D + spart * S::DPART;
#pragma unroll
    for (int i = 0; i < S::DPART; i += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(qh + i);
      const float2 a = bf2f(w.x), bq = bf2f(w.y), cq = bf2f(w.z), dq = bf2f(w.w);
      qr[h][i] = a.x * c;
      qr[h][i + 1] = a.y * c;
      qr[h][i + 2] = bq.x * c;
      qr[h][i + 3] = bq.y * c;
      qr[h][i + 4] = cq.x * c;
      qr[h][i + 5] = cq.y * c;
      qr[h][i + 6] = dq.x * c;
      qr[h][i + 7] = dq.y * c;
    }
  }
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&bars->full[st], 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int t) {  // thread 0 only: tile t into stage t % kStages
    const int st = t % kStages;
    uint8_t* dst = stages + st * C::STAGE;
    mbar_arrive_expect_tx(&bars->full[st], C::STAGE);
    const int row = k0 + t * kTile;
#pragma unroll
    for (int sub = 0; sub < C::NSUB; ++sub) {
      tma_load_3d(dst + sub * kSubBytes, &mk, &bars->full[st], 64 * sub, row, bg);
      tma_load_3d(dst + C::TILE + sub * kSubBytes, &mv, &bars->full[st], 64 * sub, row, bg);
    }
  };
  if (tid == 0) {
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
    for (int t = 0; t < kStages && t < ntiles; ++t) issue(t);
  }

  const int dp = tid % C::NDP, kg = tid / C::NDP;         // P V phase: column pair, key group
  float o_acc[G][2];
#pragma unroll
  for (int h = 0; h < G; ++h) o_acc[h][0] = o_acc[h][1] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // kept by warp h < G for head h
  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int st = t % kStages;
    const bool got = mbar_wait(&bars->full[st], (t / kStages) & 1, &bars->abort, err, wait_ns);
    ok = __syncthreads_and(got ? 1 : 0) != 0;
    if (!ok) break;
    const uint8_t* kt = stages + st * C::STAGE;
    const uint8_t* vt = kt + C::TILE;
    const int valid = min(kTile, k1 - (k0 + t * kTile));  // keys of this tile inside the range
    // ---- scores: partial dot products over this thread's slice of d, summed over the
    // NPART neighbouring lanes that hold the other slices of the same key
#pragma unroll
    for (int kk = 0; kk < S::KPT; ++kk) {
      const int j = (warp * S::KPT + kk) * S::KPW + lane / S::NPART;
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
      for (int cc = 0; cc < S::DPART; cc += 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(kt + swz(j, spart * S::DPART + cc));
        const float2 k01 = bf2f(w.x), k23 = bf2f(w.y), k45 = bf2f(w.z), k67 = bf2f(w.w);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float a = acc[h];
          a = fmaf(qr[h][cc], k01.x, a);
          a = fmaf(qr[h][cc + 1], k01.y, a);
          a = fmaf(qr[h][cc + 2], k23.x, a);
          a = fmaf(qr[h][cc + 3], k23.y, a);
          a = fmaf(qr[h][cc + 4], k45.x, a);
          a = fmaf(qr[h][cc + 5], k45.y, a);
          a = fmaf(qr[h][cc + 6], k67.x, a);
          a = fmaf(qr[h][cc + 7], k67.y, a);
          acc[h] = a;
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int off = S::NPART / 2; off > 0; off >>= 1)
          acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], off);
      }
      if (spart == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) sp[j * G + h] = acc[h];
      }
    }
    __syncthreads();
    // ---- online softmax: warp h handles head h (keys lane and lane + 32)
    if (warp < G) {
      const int h = warp;
      float s2[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = lane + 32 * e;
        s2[e] = j < valid ? sp[j * G + h] : -INFINITY;
      }
      float mx = fmaxf(s2[0], s2[1]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_run, mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m_run - m_use);  // 0 while nothing has been seen
      const float p0 = exp2f(s2[0] - m_use), p1 = exp2f(s2[1] - m_use);
      float sum = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      pb[lane * G + h] = p0;
      pb[(lane + 32) * G + h] = p1;
      if (lane == 0) alpha_s[h] = alpha;
    }
    __syncthreads();
    // ---- O += P V for this thread's column pair and keys, every head of the group
    {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float a = alpha_s[h];
        o_acc[h][0] *= a;
        o_acc[h][1] *= a;
      }
#pragma unroll
      for (int jj = 0; jj < C::KPER; ++jj) {
        const int j = kg * C::KPER + jj;
        if (j < valid) {  // rows past the range may hold anything, even NaN: never read them
          const float2 vv = bf2f(*reinterpret_cast<const uint32_t*>(vt + swz(j, 2 * dp)));
          float pr[G];
          if constexpr (G >= 4) {
#pragma unroll
            for (int h4 = 0; h4 < G; h4 += 4) {
              const float4 p4 = *reinterpret_cast<const float4*>(pb + j * G + h4);
              pr[h4] = p4.x;
              pr[h4 + 1] = p4.y;
              pr[h4 + 2] = p4.z;
              pr[h4 + 3] = p4.w;
            }
          } else if constexpr (G == 2) {
            const float2 p2 = *reinterpret_cast<const float2*>(pb + j * G);
            pr[0] = p2.x;
            pr[1] = p2.y;
          } else {
            pr[0] = pb[j];
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
            o_acc[h][0] = fmaf(pr[h], vv.x, o_acc[h][0]);
            o_acc[h][1] = fmaf(pr[h], vv.y, o_acc[h][1]);
          }
        }
      }
    }
    __syncthreads();  // every thread is done with this stage
    if (tid == 0 && t + kStages < ntiles) issue(t + kStages);
  }

  if (!ok) {
    // Let any tile still in flight land before the CTA's shared memory is released.
    if (tid == 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 1000000ull) {
      }
    }
    __syncthreads();
    return;
  }
  // ---- sum the key groups through shared memory (the ring is idle now) and write the
  // split's unnormalised output with its running maximum and sum
  float* red = reinterpret_cast<float*>(stages);  // [KGROUPS][G][D]
#pragma unroll
  for (int h = 0; h < G; ++h) {
    red[(kg * G + h) * D + 2 * dp] = o_acc[h][0];
    red[(kg * G + h) * D + 2 * dp + 1] = o_acc[h][1];
  }
  __syncthreads();
  float* out = part + (static_cast<size_t>(bg) * gridDim.x + split) * G * C::PSTRIDE;
  for (int i = tid; i < G * D; i += kThreads) {
    const int h = i / D, col = i % D;
    float v = 0.f;
#pragma unroll
    for (int q2 = 0; q2 < C::KGROUPS; ++q2) v += red[(q2 * G + h) * D + col];
    out[h * C::PSTRIDE + col] = v;
  }
  if (warp < G && lane == 0) {
    out[warp * C::PSTRIDE + D] = m_run;
    out[warp * C::PSTRIDE + D + 1] = l_run;
  }
}

// One warp per (b, h): merge the splits (rescale each by 2^(m_s - M)), normalise, write.
// The split statistics are read one split per lane and the weights broadcast by shuffles;
// each lane owns D / 32 consecutive columns and loads them as one vector per split.
template <int D>
__global__ void __launch_bounds__(256)
decode_combine_kernel(const float* __restrict__ part, int B, int Hq, int Hkv, int splits,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  constexpr int PSTRIDE = D + 4;
  constexpr int PER = D / 32;   // 2 or 4 consecutive columns per lane
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B * Hq) return;
  const int b = row / Hq, hq = row % Hq, G = Hq / Hkv;
  const int g = hq / G, h = hq % G;
  const size_t sstride = static_cast<size_t>(G) * PSTRIDE;   // floats between splits
  const float* base = part + ((static_cast<size_t>(b) * Hkv + g) * splits) * sstride +
                      h * PSTRIDE;
  float M = -INFINITY;
  for (int s = lane; s < splits; s += 32) M = fmaxf(M, base[s * sstride + D]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < splits; s0 += 32) {
      const int s = s0 + lane;
      float w = 0.f;
      if (s < splits) {
        const float ms = base[s * sstride + D];
        w = ms == -INFINITY ? 0.f : exp2f(ms - M);   // a split that saw no key weighs 0
        lsum += base[s * sstride + D + 1] * w;
      }
      const int cnt = min(32, splits - s0);
#pragma unroll 4
      for (int j = 0; j < cnt; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, j);
        const float* ps = base + (s0 + j) * sstride + lane * PER;
        if constexpr (PER == 4) {
          const float4 v = *reinterpret_cast<const float4*>(ps);
          acc[0] += wj * v.x;
          acc[1] += wj * v.y;
          acc[2] += wj * v.z;
          acc[3] += wj * v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(ps);
          acc[0] += wj * v.x;
          acc[1] += wj * v.y;
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  __nv_bfloat16* orow = o + static_cast<size_t>(row) * D + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; ++i) orow[i] = __float2bfloat16_rn(acc[i] * inv);
  if (lane == 0) lse[row] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : -INFINITY;
}

template <int D, int G>
cudaError_t launch_split(const CUtensorMap& mk, const CUtensorMap& mv, const void* q,
                         const int32_t* cache_len, int B, int Hq, int Hkv, int Lmax, int splits,
                         int chunk, float c, float* part, int* err, unsigned long long wait_ns,
                         cudaStream_t s) {
  constexpr int smem = decode_smem_bytes<D, G>();
  static_assert(smem <= 113 * 1024, "two CTAs per SM");
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid(static_cast<unsigned>(splits), static_cast<unsigned>(B * Hkv));
  decode_split_kernel<D, G><<<grid, kThreads, smem, s>>>(
      mk, mv, static_cast<const __nv_bfloat16*>(q), cache_len, Hq, Hkv, Lmax, splits, chunk, c,
      part, err, wait_ns);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Lmax, const int32_t* cache_len, float scale,
                     float* part, int splits, int* err, unsigned long long wait_ns,
                     cudaStream_t s) {
  CUtensorMap mk, mv;
  if (!make_head_map_rows(&mk, k, B * Hkv, Lmax, D, kTile) ||
      !make_head_map_rows(&mv, v, B * Hkv, Lmax, D, kTile))
    return cudaErrorInvalidValue;
  const int chunk = ((Lmax + splits - 1) / splits + kTile - 1) / kTile * kTile;
  const float c = scale * kLog2e;
  cudaError_t e;
  switch (Hq / Hkv) {
    case 1: e = launch_split<D, 1>(mk, mv, q, cache_len, B, Hq, Hkv, Lmax, splits, chunk, c, part, err, wait_ns, s); break;
    case 2: e = launch_split<D, 2>(mk, mv, q, cache_len, B, Hq, Hkv, Lmax, splits, chunk, c, part, err, wait_ns, s); break;
    case 4: e = launch_split<D, 4>(mk, mv, q, cache_len, B, Hq, Hkv, Lmax, splits, chunk, c, part, err, wait_ns, s); break;
    case 8: e = launch_split<D, 8>(mk, mv, q, cache_len, B, Hq, Hkv, Lmax, splits, chunk, c, part, err, wait_ns, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  const int rows = B * Hq;
  decode_combine_kernel<D><<<(rows + 7) / 8, 256, 0, s>>>(part, B, Hq, Hkv, splits,
                                                           static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError();
}

}  // namespace

int decode_splits(int B, int Hkv, int Lmax, int d) {
  if (d == 128) return decode_tc_splits(B, Hkv, Lmax);
  // About eight CTAs per SM over the whole grid (two resident at a time), key ranges of at
  // least 256 keys and a whole number of 64-key tiles.
  const long long pairs = static_cast<long long>(B) * Hkv;
  const long long target = 8ll * sm_count();
  long long splits = (target + pairs - 1) / pairs;
  long long chunk = (Lmax + splits - 1) / splits;
  chunk = (chunk + kTile - 1) / kTile * kTile;
  if (chunk < 256) chunk = 256;
  splits = (Lmax + chunk - 1) / chunk;
  if (splits < 1) splits = 1;
  return static_cast<int>(splits);
}

cudaError_t launch_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int Lmax, int d, const int32_t* cache_len,
                          float scale, float* partials, int splits, int* err,
                          unsigned long long wait_ns, cudaStream_t s) {
  if (d == 64)
    return launch_d<64>(q, k, v, o, lse, B, Hq, Hkv, Lmax, cache_len, scale, partials, splits,
                        err, wait_ns, s);
  // d = 128: the tensor-core split kernel (fa_decode_tc.cu), then the same combine.
  cudaError_t e = launch_decode_tc(q, k, v, B, Hq, Hkv, Lmax, cache_len, scale, partials,
                                   splits, err, wait_ns, s);
  if (e != cudaSuccess) return e;
  const int rows = B * Hq;
  decode_combine_kernel<128><<<(rows + 7) / 8, 256, 0, s>>>(partials, B, Hq, Hkv, splits,
                                                             static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError();
}

}  // namespace fa
