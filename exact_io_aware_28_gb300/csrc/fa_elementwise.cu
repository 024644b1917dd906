// HBM-bound elementwise kernels of the backward pass.
//
//  * preprocess: D_i = sum_c dO_ic * O_ic for every row (fp32), and, when asked,
//    zeroes the fp32 dQ accumulator row in the same pass.  D is the row term of
//    dS = P o (dP - D); since O = P V and rows of P sum to one it equals
//    sum_j P_ij dP_ij, so it can be formed from O and dO alone before the main
//    backward kernel runs (answer page "How FlashAttention works for training",
//    section 3.1: the backward needs only O, the saved statistics and dO).
//  * dq_convert: dQ = scale * dQacc rounded once to the output type.
//
// Both read and write every byte exactly once with 16-byte vector accesses and a
// grid-stride loop over a grid sized to the SM count.
#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
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
};
template <> struct Vec<float> {
  static constexpr int n = 4;
  __device__ static void load(const float* p, float* out) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(p));
    out[0] = f.x; out[1] = f.y; out[2] = f.z; out[3] = f.w;
  }
};

// TPR lanes per row; each lane loads one 16-byte vector of O and of dO.
template <typename T, int D>
__global__ void __launch_bounds__(256)
preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dO, float* __restrict__ Dsum,
                  float* __restrict__ dq_acc, long long rows) {
  constexpr int VEC = Vec<T>::n;
  constexpr int TPR = D / VEC;           // 8 or 16 (bf16), 16 or 32 (fp32)
  constexpr int RPW = 32 / TPR;          // rows per warp per iteration
  // O of the forward just launched, and the dQ accumulator the previous convert read.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int sub = lane / TPR, part = lane % TPR;
  for (long long r0 = warp * RPW; r0 < rows; r0 += nwarps * RPW) {
    const long long row = r0 + sub;
    float acc = 0.f;
    if (row < rows) {
      float a[VEC], g[VEC];
      Vec<T>::load(o + row * D + part * VEC, a);
      Vec<T>::load(dO + row * D + part * VEC, g);
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc = fmaf(a[i], g[i], acc);
      if (dq_acc) {
        // D fp32 elements per row; each lane clears D / TPR = VEC of them.
        float4* z = reinterpret_cast<float4*>(dq_acc + row * D + part * VEC);
#pragma unroll
        for (int i = 0; i < VEC / 4; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0) Dsum[row] = acc;
  }
}

// Eight elements per thread: two 16-byte fp32 loads, one 16-byte bf16 store.
__global__ void __launch_bounds__(256)
dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, float scale,
                  long long n8) {
  ptx::griddep_wait();   // the backward main kernel's reduce-adds
  ptx::griddep_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
    uint4 out;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&out);
    h[0] = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    h[1] = __floats2bfloat162_rn(a.z * scale, a.w * scale);
    h[2] = __floats2bfloat162_rn(b.x * scale, b.y * scale);
    h[3] = __floats2bfloat162_rn(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = out;
  }
}

template <typename T, int D>
cudaError_t preprocess_typed(const Problem& p, const void* o, const void* dO, float* Dsum,
                             float* dq_acc, cudaStream_t s) {
  const long long rows = (long long)p.B * p.H * p.N;
  constexpr int RPW = 32 / (D / Vec<T>::n);
  const long long warps_needed = (rows + RPW - 1) / RPW;
  long long blocks = (warps_needed + 7) / 8;
  const long long cap = (long long)sm_count() * 8;  // 8 CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  return launch_dependent(preprocess_kernel<T, D>, dim3((unsigned)blocks), dim3(256), 0, s,
                          (const T*)o, (const T*)dO, Dsum, dq_acc, rows);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const Problem& p, fa_dtype dt, const void* o, const void* dO,
                                  float* Dsum, float* dq_acc, cudaStream_t s) {
  if (dt == FA_FP32)
    return p.d == 64 ? preprocess_typed<float, 64>(p, o, dO, Dsum, dq_acc, s)
                     : preprocess_typed<float, 128>(p, o, dO, Dsum, dq_acc, s);
  return p.d == 64 ? preprocess_typed<__nv_bfloat16, 64>(p, o, dO, Dsum, dq_acc, s)
                   : preprocess_typed<__nv_bfloat16, 128>(p, o, dO, Dsum, dq_acc, s);
}

cudaError_t launch_dq_convert(const Problem& p, const float* dq_acc, void* dq, cudaStream_t s) {
  const long long n8 = (long long)p.B * p.H * p.N * p.d / 8;
  long long blocks = (n8 + 255) / 256;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  return launch_dependent(dq_convert_kernel, dim3((unsigned)blocks), dim3(256), 0, s, dq_acc,
                          (__nv_bfloat16*)dq, p.scale, n8);
}

}  // namespace fa
