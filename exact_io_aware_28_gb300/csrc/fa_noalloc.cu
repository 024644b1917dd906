// fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code running inside another
// framework's memory pool that does not expose an allocator, plug-ins and embedded
// runtimes whose device memory was planned up front, or hooks that run where a
// cudaMalloc would synchronise the device or is simply not permitted.  For them this
// entry point runs the same three backward stages as fa_bwd, with the workspace (the
// fp32 row sums D and the fp32 dQ accumulator) placed in a fixed array that lives in the
// library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds
// FA_NOALLOC_SCRATCH_BYTES of it until the process exits.  In host code its name only
// stands in for the symbol, it is not a device address, so the address is fetched with
// cudaGetSymbolAddress, once per device, with that device current, on the first call
// made on that device (make that first call before any stream capture).  That first call
// is safe from several host threads at once: the cached address is atomic and each thread
// that races stores the same value.  All calls share
// the one array and it keeps the previous call's contents: the preprocess stage rewrites
// D and zeroes the accumulator at the start of every call, and two calls whose work
// overlaps on the GPU (for example on two streams) race on it.
#include <stdint.h>

#include <atomic>

#include "fa_internal.cuh"

namespace fa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];  // device address of the array, per device

// Device address of the scratch array on the current device, or nullptr on failure.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* cached = g_scratch_ptr[dev].load();
  if (!cached) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev].store(ptr);
    cached = ptr;
  }
  return cached;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dO, void* dq, void* dk,
                                    void* dv, int B, int H, int N, int d, int causal,
                                    const uint8_t* blockmask, const int32_t* kv_len,
                                    float scale, fa_dtype dtype, void* stream) {
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0) {  // invalid sizes: let the ordinary validation name the problem
    return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, blockmask, kv_len, scale,
                  dtype, nullptr, 0, stream);
  }
  if (need > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES)) return FA_ERR_UNSUPPORTED;
  void* scratch = fa::scratch_address();
  if (!scratch) return FA_ERR_CUDA;
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, blockmask, kv_len, scale,
                dtype, scratch, static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES), stream);
}
