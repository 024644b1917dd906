// fp32 CUDA-core attention kernels (forward, dK/dV, dQ) for the FA_FP32 path.
//
// Same mathematics as the tensor-core path, in fp32 arithmetic throughout:
//   forward  -- tiles of keys staged in shared memory, a running row maximum m and
//               row sum l with O rescaled by e^{m_old - m_new} whenever the maximum
//               grows (course week 13, step 2; FlashAttention reading guide, "Method",
//               steps 1-4, in the unnormalised form: O is divided by l once at the end);
//   backward -- P recomputed from the saved logsumexp (answer page, section 3.1):
//               P_ij = exp(scale q_i.k_j - lse_i), dP_ij = dO_i.v_j,
//               dS_ij = P_ij (dP_ij - D_i); a key-outer kernel accumulates
//               dV_j = sum_i P_ij dO_i and dK_j = scale sum_i dS_ij q_i, a query-outer
//               kernel accumulates dQ_i = scale sum_j dS_ij k_j.  No atomics: the result
//               does not depend on scheduling.
// Scores are kept in the log2 domain (q pre-multiplied by scale*log2(e)) so that every
// exponential is an exp2.
//
// Dropout (threshold > 0): the probability of element (i, j) enters P V, dV and dP as
// P_ij Z_ij / (1 - p), with Z regenerated from the generator of fa_philox.cuh in each
// kernel; the row sums of the forward keep every term.  One generator call per element
// (this path serves small problems).
//
// Thread layout: four threads per row, each owning every fourth element of the head
// dimension; dot products finish with two xor-shuffles inside the group of four.
#include <math.h>

#include "fa_internal.cuh"
#include "fa_philox.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kTPR = 4;        // threads per row
constexpr int kRows = 64;      // rows owned by one CTA (divides the 128-row mask block)
constexpr int kTile = 32;      // rows of the other operand staged per shared-memory tile
constexpr int kThreads = kRows * kTPR;

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ int key_limit(const Problem& p, int b) {
  if (!p.kv_len) return p.N;
  int L = p.kv_len[b];
  return L < 0 ? 0 : (L > p.N ? p.N : L);
}

// Z_ij / (1 - p) of element (bh, i, j): 0 when dropped, the keep scale otherwise (1 with
// no dropout).
__device__ __forceinline__ float drop_factor(const Problem& p, int bh, int i, int j) {
  if (p.drop_threshold <= 0) return 1.f;
  const philox::Words g = philox::call(p, bh, i, j);
  return philox::byte_of(g, i, j) >= static_cast<uint32_t>(p.drop_threshold) ? p.drop_scale
                                                                               : 0.f;
}

__device__ __forceinline__ float group_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                T* __restrict__ o, float* __restrict__ lse, Problem p) {
  constexpr int DS = D / kTPR;
  __shared__ float ks[kTile][D];
  __shared__ float vs[kTile][D];
  const int N = p.N;
  const int bh = blockIdx.y;
  const int b = bh / p.H;
  const size_t head = (size_t)bh * N * D;
  const int tid = threadIdx.x, r = tid / kTPR, part = tid % kTPR;
  const int row0 = blockIdx.x * kRows;
  const int row = row0 + r;
  const bool valid_row = row < N;
  const float c = p.scale * kLog2e;

  float qr[DS], acc[DS];
#pragma unroll
  for (int t = 0; t < DS; ++t) {
    qr[t] = valid_row ? to_f(q[head + (size_t)row * D + part + kTPR * t]) * c : 0.f;
    acc[t] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  int kend = key_limit(p, b);
  if (p.causal) kend = min(kend, min(N, row0 + kRows));
  const int nb = (N + kMaskBlock - 1) / kMaskBlock;

  for (int k0 = 0; k0 < kend; k0 += kTile) {
    if (p.blockmask && !p.blockmask[(row0 / kMaskBlock) * nb + k0 / kMaskBlock]) continue;
    __syncthreads();
    for (int e = tid; e < kTile * D; e += kThreads) {
      const int j = e / D, cc = e % D, key = k0 + j;
      ks[j][cc] = key < N ? to_f(k[head + (size_t)key * D + cc]) : 0.f;
      vs[j][cc] = key < N ? to_f(v[head + (size_t)key * D + cc]) : 0.f;
    }
    __syncthreads();
    const int jmax = min(kTile, kend - k0);
    for (int j = 0; j < jmax; ++j) {
      float s = 0.f;
#pragma unroll
      for (int t = 0; t < DS; ++t) s += qr[t] * ks[j][part + kTPR * t];
      s = group_sum(s);
      const int key = k0 + j;
      if (!valid_row || (p.causal && key > row)) continue;
      if (s > m) {
        const float alpha = exp2f(m - s);
        l *= alpha;
#pragma unroll
        for (int t = 0; t < DS; ++t) acc[t] *= alpha;
        m = s;
      }
      const float pj = exp2f(s - m);
      l += pj;
      const float pz = pj * drop_factor(p, bh, row, key);
#pragma unroll
      for (int t = 0; t < DS; ++t) acc[t] += pz * vs[j][part + kTPR * t];
    }
  }
  if (valid_row) {
    const float inv = l > 0.f ? 1.f / l : 0.f;   // dropout's 1 / (1 - p) is in drop_factor
#pragma unroll
    for (int t = 0; t < DS; ++t) o[head + (size_t)row * D + part + kTPR * t] = from_f<T>(acc[t] * inv);
    if (part == 0) lse[(size_t)bh * N + row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

// Key-outer: one CTA owns 64 keys and walks every query row that may see them.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
bwd_dkdv_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const float* __restrict__ lse, const T* __restrict__ dO,
                     const float* __restrict__ Dsum, T* __restrict__ dk, T* __restrict__ dv,
                     Problem p) {
  constexpr int DS = D / kTPR;
  __shared__ float qs[kTile][D];
  __shared__ float dos[kTile][D];
  __shared__ float lses[kTile];
  __shared__ float Ds[kTile];
  const int N = p.N;
  const int bh = blockIdx.y;
  const int b = bh / p.H;
  const size_t head = (size_t)bh * N * D;
  const int tid = threadIdx.x, r = tid / kTPR, part = tid % kTPR;
  const int key0 = blockIdx.x * kRows;
  const int key = key0 + r;
  const int L = key_limit(p, b);
  const bool live_key = key < L;
  const float c = p.scale * kLog2e;

  float kr[DS], vr[DS], dka[DS], dva[DS];
#pragma unroll
  for (int t = 0; t < DS; ++t) {
    const size_t off = head + (size_t)key * D + part + kTPR * t;
    kr[t] = key < N ? to_f(k[off]) * c : 0.f;
    vr[t] = key < N ? to_f(v[off]) : 0.f;
    dka[t] = 0.f;
    dva[t] = 0.f;
  }
  const int nb = (N + kMaskBlock - 1) / kMaskBlock;
  const int qstart = p.causal ? (key0 / kTile) * kTile : 0;
  if (key0 < L) {
    for (int i0 = qstart; i0 < N; i0 += kTile) {
      if (p.blockmask && !p.blockmask[(i0 / kMaskBlock) * nb + key0 / kMaskBlock]) continue;
      __syncthreads();
      for (int e = tid; e < kTile * D; e += kThreads) {
        const int ii = e / D, cc = e % D, qrow = i0 + ii;
        qs[ii][cc] = qrow < N ? to_f(q[head + (size_t)qrow * D + cc]) : 0.f;
        dos[ii][cc] = qrow < N ? to_f(dO[head + (size_t)qrow * D + cc]) : 0.f;
      }
      if (tid < kTile) {
        const int qrow = i0 + tid;
        lses[tid] = qrow < N ? lse[(size_t)bh * N + qrow] * kLog2e : -INFINITY;
        Ds[tid] = qrow < N ? Dsum[(size_t)bh * N + qrow] : 0.f;
      }
      __syncthreads();
      const int imax = min(kTile, N - i0);
      for (int ii = 0; ii < imax; ++ii) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int t = 0; t < DS; ++t) {
          s += kr[t] * qs[ii][part + kTPR * t];
          dp += vr[t] * dos[ii][part + kTPR * t];
        }
        s = group_sum(s);
        dp = group_sum(dp);
        const int qrow = i0 + ii;
        const float l2 = lses[ii];
        if (!live_key || (p.causal && key > qrow) || l2 == -INFINITY) continue;
        const float pij = exp2f(s - l2);
        const float z = drop_factor(p, bh, qrow, key);
        const float ds = pij * (dp * z - Ds[ii]);
        const float pz = pij * z;
#pragma unroll
        for (int t = 0; t < DS; ++t) {
          dva[t] += pz * dos[ii][part + kTPR * t];
          dka[t] += ds * qs[ii][part + kTPR * t];
        }
      }
    }
  }
  if (key < N) {
#pragma unroll
    for (int t = 0; t < DS; ++t) {
      const size_t off = head + (size_t)key * D + part + kTPR * t;
      dk[off] = from_f<T>(dka[t] * p.scale);
      dv[off] = from_f<T>(dva[t]);
    }
  }
}

// Query-outer: one CTA owns 64 query rows and walks every key they may see.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
bwd_dq_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const float* __restrict__ lse, const T* __restrict__ dO,
                   const float* __restrict__ Dsum, T* __restrict__ dq, Problem p) {
  constexpr int DS = D / kTPR;
  __shared__ float ks[kTile][D];
  __shared__ float vs[kTile][D];
  const int N = p.N;
  const int bh = blockIdx.y;
  const int b = bh / p.H;
  const size_t head = (size_t)bh * N * D;
  const int tid = threadIdx.x, r = tid / kTPR, part = tid % kTPR;
  const int row0 = blockIdx.x * kRows;
  const int row = row0 + r;
  const bool valid_row = row < N;
  const float c = p.scale * kLog2e;

  float qr[DS], dor[DS], acc[DS];
#pragma unroll
  for (int t = 0; t < DS; ++t) {
    const size_t off = head + (size_t)row * D + part + kTPR * t;
    qr[t] = valid_row ? to_f(q[off]) * c : 0.f;
    dor[t] = valid_row ? to_f(dO[off]) : 0.f;
    acc[t] = 0.f;
  }
  const float l2 = valid_row ? lse[(size_t)bh * N + row] * kLog2e : -INFINITY;
  const float Di = valid_row ? Dsum[(size_t)bh * N + row] : 0.f;
  int kend = key_limit(p, b);
  if (p.causal) kend = min(kend, min(N, row0 + kRows));
  const int nb = (N + kMaskBlock - 1) / kMaskBlock;

  for (int k0 = 0; k0 < kend; k0 += kTile) {
    if (p.blockmask && !p.blockmask[(row0 / kMaskBlock) * nb + k0 / kMaskBlock]) continue;
    __syncthreads();
    for (int e = tid; e < kTile * D; e += kThreads) {
      const int j = e / D, cc = e % D, key = k0 + j;
      ks[j][cc] = key < N ? to_f(k[head + (size_t)key * D + cc]) : 0.f;
      vs[j][cc] = key < N ? to_f(v[head + (size_t)key * D + cc]) : 0.f;
    }
    __syncthreads();
    const int jmax = min(kTile, kend - k0);
    for (int j = 0; j < jmax; ++j) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int t = 0; t < DS; ++t) {
        s += qr[t] * ks[j][part + kTPR * t];
        dp += dor[t] * vs[j][part + kTPR * t];
      }
      s = group_sum(s);
      dp = group_sum(dp);
      const int key = k0 + j;
      if (!valid_row || (p.causal && key > row) || l2 == -INFINITY) continue;
      const float ds = exp2f(s - l2) * (dp * drop_factor(p, bh, row, key) - Di);
#pragma unroll
      for (int t = 0; t < DS; ++t) acc[t] += ds * ks[j][part + kTPR * t];
    }
  }
  if (valid_row) {
#pragma unroll
    for (int t = 0; t < DS; ++t)
      dq[head + (size_t)row * D + part + kTPR * t] = from_f<T>(acc[t] * p.scale);
  }
}

template <typename T, int D>
cudaError_t fwd_typed(const Problem& p, const void* q, const void* k, const void* v, void* o,
                      float* lse, cudaStream_t s) {
  dim3 grid((p.N + kRows - 1) / kRows, p.B * p.H);
  fwd_simt_kernel<T, D><<<grid, kThreads, 0, s>>>((const T*)q, (const T*)k, (const T*)v,
                                                  (T*)o, lse, p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_typed(const Problem& p, const void* q, const void* k, const void* v,
                      const float* lse, const void* dO, const float* Dsum, void* dq, void* dk,
                      void* dv, cudaStream_t s) {
  dim3 grid((p.N + kRows - 1) / kRows, p.B * p.H);
  bwd_dkdv_simt_kernel<T, D><<<grid, kThreads, 0, s>>>((const T*)q, (const T*)k, (const T*)v,
                                                       lse, (const T*)dO, Dsum, (T*)dk,
                                                       (T*)dv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_dq_simt_kernel<T, D><<<grid, kThreads, 0, s>>>((const T*)q, (const T*)k, (const T*)v, lse,
                                                     (const T*)dO, Dsum, (T*)dq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const Problem& p, fa_dtype dt, const void* q, const void* k,
                            const void* v, void* o, float* lse, cudaStream_t s) {
  if (dt == FA_FP32)
    return p.d == 64 ? fwd_typed<float, 64>(p, q, k, v, o, lse, s)
                     : fwd_typed<float, 128>(p, q, k, v, o, lse, s);
  return p.d == 64 ? fwd_typed<__nv_bfloat16, 64>(p, q, k, v, o, lse, s)
                   : fwd_typed<__nv_bfloat16, 128>(p, q, k, v, o, lse, s);
}

cudaError_t launch_bwd_simt(const Problem& p, fa_dtype dt, const void* q, const void* k,
                            const void* v, const float* lse, const void* dO, const float* D,
                            void* dq, void* dk, void* dv, cudaStream_t s) {
  if (dt == FA_FP32)
    return p.d == 64 ? bwd_typed<float, 64>(p, q, k, v, lse, dO, D, dq, dk, dv, s)
                     : bwd_typed<float, 128>(p, q, k, v, lse, dO, D, dq, dk, dv, s);
  return p.d == 64 ? bwd_typed<__nv_bfloat16, 64>(p, q, k, v, lse, dO, D, dq, dk, dv, s)
                   : bwd_typed<__nv_bfloat16, 128>(p, q, k, v, lse, dO, D, dq, dk, dv, s);
}

}  // namespace fa
