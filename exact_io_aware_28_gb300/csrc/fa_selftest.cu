// Self-test of the kernels' failure detection: a single warp waits on an mbarrier that
// nothing ever arrives on, with the same bounded wait the tensor-core kernels use.  The
// wait must give up after the limit, record FA_ERR_TIMEOUT in the device error word and
// return, leaving the context usable.  It uses no TMA and no tensor memory.
#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncwarp();
  // Phase 0 never completes: no thread arrives.
  ptx::mbar_wait_warp(&bar, 0, &abort_flag, err, limit_ns);
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_selftest_wait_timeout(unsigned int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 10000) return FA_ERR_INVALID_ARG;
  int* err = fa::error_word();
  if (!err) return FA_ERR_CUDA;
  fa::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      err, static_cast<unsigned long long>(limit_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
