// Dropout generator bytes as a tensor: u(bh, i, j) for every head, query row and key of a
// [BH, n_q, n_k] block, from the same generator and element map the attention kernels use
// (fa_philox.cuh).  For inspecting and testing the mask; the attention kernels never read
// it back.
#include "fa_internal.cuh"
#include "fa_philox.cuh"

namespace fa {
namespace {

// One thread per generator call: 2 query rows (i, i + 8) x 8 keys, scattered to `out`.
__global__ void dropout_bytes_kernel(uint8_t* __restrict__ out, int n_q, int n_k, Problem p) {
  const int bh = blockIdx.y;
  const int n_rho = 8 * ((n_q + 15) / 16), n_kappa = 4 * ((n_k + 31) / 32);
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(n_rho) * n_kappa) return;
  const int rho = static_cast<int>(idx / n_kappa), kappa = static_cast<int>(idx % n_kappa);
  const int i0 = 16 * (rho >> 3) + (rho & 7);            // rows i0 and i0 + 8
  const int j0 = 32 * (kappa >> 2) + 2 * (kappa & 3);    // keys j0 + {0, 1} + {0, 8, 16, 24}
  const philox::Words g = philox::call(p, bh, i0, j0);
  uint8_t* head = out + static_cast<size_t>(bh) * n_q * n_k;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = i0 + 8 * s;
    if (i >= n_q) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = j0 + 8 * c + e;
        if (j < n_k) head[static_cast<size_t>(i) * n_k + j] = static_cast<uint8_t>(philox::byte_of(g, i, j));
      }
    }
  }
}

}  // namespace

cudaError_t launch_dropout_bytes(const Problem& p, uint8_t* out, int BH, int n_q, int n_k,
                                 cudaStream_t s) {
  const long long calls = static_cast<long long>(8 * ((n_q + 15) / 16)) * (4 * ((n_k + 31) / 32));
  const int threads = 256;
  dim3 grid(static_cast<unsigned>((calls + threads - 1) / threads), static_cast<unsigned>(BH));
  dropout_bytes_kernel<<<grid, threads, 0, s>>>(out, n_q, n_k, p);
  return cudaGetLastError();
}

}  // namespace fa
