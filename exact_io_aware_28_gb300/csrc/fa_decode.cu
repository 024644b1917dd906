// Decode attention over a key/value cache with grouped key/value heads: one new query token
// per sequence, split over the cache length, then combined.
//
// What it computes (course page "Week 13. GPU and FlashAttention", step 1, the bullet on
// attention in decode, and step 2's online softmax): query head h of sequence b reads
// key/value head g = h / G (G = Hq / Hkv query heads per key/value head) and the keys
// j < cache_len[b]; o = softmax(scale q K^T) V and lse = logsumexp(scale q K^T).  Each
// sequence has its own cache, so the step reads every cached byte once and does about G
// FLOPs per byte: it is bound by HBM bandwidth, and grouping the heads is what raises the
// work done per byte read.
//
// Two kernels: the tensor-core split kernel of fa_decode_tc.cu writes, for every key range
// of every (sequence, key/value head), the unnormalised output of each query head with its
// running maximum m (log2 domain) and sum l to the caller's fp32 workspace; the combine
// kernel below merges the ranges of each (b, h) by the same rescaling rule and writes o
// (bf16) and lse (fp32, natural log).
#include <cuda.h>
#include <math.h>

#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

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

}  // namespace

int decode_splits(int B, int Hkv, int Lmax, int d) {
  (void)d;  // both head dimensions split the same way: whole 128-key tiles
  return decode_tc_splits(B, Hkv, Lmax);
}

cudaError_t launch_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int Lmax, int d, const int32_t* cache_len,
                          float scale, float* partials, int splits, int* err,
                          unsigned long long wait_ns, cudaStream_t s) {
  cudaError_t e = launch_decode_tc(q, k, v, B, Hq, Hkv, Lmax, d, cache_len, scale, partials,
                                   splits, err, wait_ns, s);
  if (e != cudaSuccess) return e;
  const int rows = B * Hq;
  if (d == 64)
    decode_combine_kernel<64><<<(rows + 7) / 8, 256, 0, s>>>(partials, B, Hq, Hkv, splits,
                                                              static_cast<__nv_bfloat16*>(o), lse);
  else
    decode_combine_kernel<128><<<(rows + 7) / 8, 256, 0, s>>>(partials, B, Hq, Hkv, splits,
                                                               static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError();
}

}  // namespace fa
