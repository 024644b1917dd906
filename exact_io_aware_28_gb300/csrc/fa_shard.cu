// Kernels of attention split over key/value shards of one sequence.
//
//  * merge: S partial results of the same query rows over disjoint key sets, each a
//    normalised O_k with its logsumexp lse_k, combine into the attention over all keys.
//    This is the merge rule of the FlashAttention reading guide (arXiv 2205.14135,
//    "Method": m = max(m1, m2), l = e^{m1 - m} l1 + e^{m2 - m} l2) written for (O, lse)
//    pairs: lse = ln sum_k e^{lse_k} and O = sum_k e^{lse_k - lse} O_k.  Parts with
//    lse_k = -inf weigh nothing; a row with no visible key anywhere gets O = 0, lse = -inf.
//  * accumulate / finish: fp32 running sums of gradient contributions (acc += x) and the
//    final rounding of a running sum to the output type, for the dK, dV of a key shard
//    that several query shards contribute to.
//
// All three are HBM-bound: 16-byte vector accesses, grid-stride loops over a grid sized to
// the SM count.
#include "fa_internal.cuh"

namespace fa {
namespace {

template <typename T> struct V16;
template <> struct V16<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const __nv_bfloat16* p, float* out) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float* in) {
    uint4 raw;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = raw;
  }
};
template <> struct V16<float> {
  static constexpr int n = 4;
  __device__ static void load(const float* p, float* out) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(p));
    out[0] = f.x; out[1] = f.y; out[2] = f.z; out[3] = f.w;
  }
  __device__ static void store(float* p, const float* in) {
    *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
  }
};

// TPR lanes per row, each owning one 16-byte vector of the row; rows per warp = 32 / TPR.
template <typename T, int D>
__global__ void __launch_bounds__(256)
merge_kernel(const T* __restrict__ o_parts, const float* __restrict__ lse_parts, int S,
             T* __restrict__ o, float* __restrict__ lse, long long rows) {
  constexpr int VEC = V16<T>::n;
  constexpr int TPR = D / VEC;
  constexpr int RPW = 32 / TPR;
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int sub = lane / TPR, part = lane % TPR;
  for (long long r0 = warp * RPW; r0 < rows; r0 += nwarps * RPW) {
    const long long row = r0 + sub;
    if (row >= rows) continue;
    // m = max_k lse_k, then the weights e^{lse_k - m} and their sum; four parts' loads are
    // in flight at a time.
    float m = -INFINITY;
    int k = 0;
    for (; k + 4 <= S; k += 4) {
      float l[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) l[t] = __ldg(lse_parts + (k + t) * rows + row);
      m = fmaxf(m, fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3])));
    }
    for (; k < S; ++k) m = fmaxf(m, __ldg(lse_parts + k * rows + row));
    float acc[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
    float total = 0.f;
    if (m != -INFINITY) {
      k = 0;
      for (; k + 4 <= S; k += 4) {
        float l[4], x[4][VEC];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          l[t] = __ldg(lse_parts + (k + t) * rows + row);
          V16<T>::load(o_parts + ((k + t) * rows + row) * D + part * VEC, x[t]);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          // a part without visible keys (lse = -inf) contributes nothing, whatever its O row
          if (l[t] == -INFINITY) continue;
          const float wk = expf(l[t] - m);
          total += wk;
#pragma unroll
          for (int i = 0; i < VEC; ++i) acc[i] = fmaf(wk, x[t][i], acc[i]);
        }
      }
      for (; k < S; ++k) {
        const float lk = __ldg(lse_parts + k * rows + row);
        if (lk == -INFINITY) continue;
        const float wk = expf(lk - m);
        total += wk;
        float x[VEC];
        V16<T>::load(o_parts + (k * rows + row) * D + part * VEC, x);
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = fmaf(wk, x[i], acc[i]);
      }
    }
    const float inv = total > 0.f ? 1.f / total : 0.f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[i] *= inv;
    V16<T>::store(o + row * D + part * VEC, acc);
    if (part == 0) lse[row] = total > 0.f ? m + logf(total) : -INFINITY;
  }
}

// acc[i] += x[i], four elements per thread and iteration.
template <typename T>
__global__ void __launch_bounds__(256)
accumulate_kernel(float* __restrict__ acc, const T* __restrict__ x, long long n4) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 a = reinterpret_cast<float4*>(acc)[i];
    float v[4];
    if constexpr (sizeof(T) == 2) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x) + i);
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
    } else {
      const float4 f = __ldg(reinterpret_cast<const float4*>(x) + i);
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
    a.x += v[0]; a.y += v[1]; a.z += v[2]; a.w += v[3];
    reinterpret_cast<float4*>(acc)[i] = a;
  }
}

// out[i] = acc[i] rounded to the output type, four elements per thread and iteration.
template <typename T>
__global__ void __launch_bounds__(256)
finish_kernel(T* __restrict__ out, const float* __restrict__ acc, long long n4) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc) + i);
    if constexpr (sizeof(T) == 2) {
      uint2 raw;
      *reinterpret_cast<__nv_bfloat162*>(&raw.x) = __floats2bfloat162_rn(a.x, a.y);
      *reinterpret_cast<__nv_bfloat162*>(&raw.y) = __floats2bfloat162_rn(a.z, a.w);
      reinterpret_cast<uint2*>(out)[i] = raw;
    } else {
      reinterpret_cast<float4*>(out)[i] = a;
    }
  }
}

unsigned grid_for(long long work_items, int per_block) {
  long long blocks = (work_items + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(sm_count()) * 8;  // 8 CTAs of 256 per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

template <typename T, int D>
cudaError_t merge_typed(const void* o_parts, const float* lse_parts, int S, void* o, float* lse,
                        long long rows, cudaStream_t s) {
  constexpr int RPW = 32 / (D / V16<T>::n);
  merge_kernel<T, D><<<grid_for((rows + RPW - 1) / RPW, 8), 256, 0, s>>>(
      static_cast<const T*>(o_parts), lse_parts, S, static_cast<T*>(o), lse, rows);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const void* o_parts, const float* lse_parts, int S, void* o, float* lse,
                         long long rows, int d, fa_dtype dt, cudaStream_t s) {
  if (dt == FA_FP32)
    return d == 64 ? merge_typed<float, 64>(o_parts, lse_parts, S, o, lse, rows, s)
                   : merge_typed<float, 128>(o_parts, lse_parts, S, o, lse, rows, s);
  return d == 64 ? merge_typed<__nv_bfloat16, 64>(o_parts, lse_parts, S, o, lse, rows, s)
                 : merge_typed<__nv_bfloat16, 128>(o_parts, lse_parts, S, o, lse, rows, s);
}

cudaError_t launch_accumulate(float* acc, const void* x, long long n, fa_dtype dt,
                              cudaStream_t s) {
  const long long n4 = n / 4;
  if (dt == FA_FP32)
    accumulate_kernel<float><<<grid_for(n4, 256), 256, 0, s>>>(acc, static_cast<const float*>(x),
                                                                n4);
  else
    accumulate_kernel<__nv_bfloat16><<<grid_for(n4, 256), 256, 0, s>>>(
        acc, static_cast<const __nv_bfloat16*>(x), n4);
  return cudaGetLastError();
}

cudaError_t launch_finish(void* out, const float* acc, long long n, fa_dtype dt, cudaStream_t s) {
  const long long n4 = n / 4;
  if (dt == FA_FP32)
    finish_kernel<float><<<grid_for(n4, 256), 256, 0, s>>>(static_cast<float*>(out), acc, n4);
  else
    finish_kernel<__nv_bfloat16><<<grid_for(n4, 256), 256, 0, s>>>(
        static_cast<__nv_bfloat16*>(out), acc, n4);
  return cudaGetLastError();
}

}  // namespace fa

extern "C" {

fa_status fa_attn_merge(const void* o_parts, const float* lse_parts, int S, void* o, float* lse,
                        int B, int H, int N, int d, fa_dtype dtype, void* stream) {
  if (S < 1 || S > FA_MERGE_MAX_PARTS || B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
  if (!o_parts || !lse_parts || !o || !lse) return FA_ERR_INVALID_ARG;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!a16(o_parts) || !a16(o) || !a4(lse_parts) || !a4(lse)) return FA_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * N;
  const cudaError_t e = fa::launch_merge(o_parts, lse_parts, S, o, lse, rows, d, dtype,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_grad_accumulate(float* acc, const void* x, long long n, fa_dtype dtype,
                             void* stream) {
  if (!acc || !x || n < 1 || (n & 3) != 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(acc) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(x) & (dtype == FA_FP32 ? 15u : 7u)) != 0)
    return FA_ERR_INVALID_ARG;
  const cudaError_t e = fa::launch_accumulate(acc, x, n, dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_grad_finish(void* out, const float* acc, long long n, fa_dtype dtype, void* stream) {
  if (!acc || !out || n < 1 || (n & 3) != 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(acc) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(out) & (dtype == FA_FP32 ? 15u : 7u)) != 0)
    return FA_ERR_INVALID_ARG;
  const cudaError_t e = fa::launch_finish(out, acc, n, dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
