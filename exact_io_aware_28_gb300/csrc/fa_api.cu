// C-ABI boundary of libfa_gb300.so: argument validation, workspace carving and kernel
// dispatch.  Every entry point validates on the host before launching anything; no entry
// point allocates device memory or synchronises the stream (fa_device_error excepted).
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>

#include "fa_internal.cuh"

namespace fa {

namespace {
constexpr int kMaxDevices = 64;
// Per-device caches.  Host threads may fill them concurrently: each slot is atomic and a
// race only stores the same value twice.
std::atomic<int> g_sm_count[kMaxDevices];    // 0 = not yet queried
std::atomic<int*> g_err_ptr[kMaxDevices];    // device address of the error word
}  // namespace

// Device error word: a kernel whose bounded wait runs out stores FA_ERR_TIMEOUT here.
static __device__ int g_device_error;

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 148;
  int n = g_sm_count[dev].load();
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_sm_count[dev].store(n);
  }
  return n;
}

int* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* cached = g_err_ptr[dev].load();
  if (!cached) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess || !ptr) return nullptr;
    cached = static_cast<int*>(ptr);
    g_err_ptr[dev].store(cached);
  }
  return cached;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

fa_status check_shape(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H > 65535) return FA_ERR_UNSUPPORTED;
  if (N > (1 << 24)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

unsigned long long wait_limit_ns() {
  // Initialised once (a function-local static is thread-safe).
  static const unsigned long long ns = [] {
    unsigned long long v = 2000ull;
    if (const char* s = getenv("FA_WAIT_LIMIT_MS")) {
      const long long ms = atoll(s);
      if (ms > 0 && ms < 600000) v = static_cast<unsigned long long>(ms);
    }
    return v * 1000000ull;
  }();
  return ns;
}

}  // namespace fa

using namespace fa;

extern "C" {

size_t fa_decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || Hq % Hkv != 0) return 0;
  if (d != 64 && d != 128) return 0;
  const size_t splits = static_cast<size_t>(decode_splits(B, Hkv, Lmax, d));
  return static_cast<size_t>(B) * Hq * splits * (d + 4) * sizeof(float);
}

fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int Hq, int Hkv, int Lmax, int d, const int32_t* cache_len,
                    float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return FA_ERR_UNSUPPORTED;
  if ((long long)B * Hkv > 65535 || Lmax > (1 << 24)) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace))
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cache_len) & 3u) != 0) return FA_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (workspace_bytes < fa_decode_workspace_bytes(B, Hq, Hkv, Lmax, d)) return FA_ERR_INVALID_ARG;
  int* err = error_word();
  if (!err) return FA_ERR_CUDA;
  const int splits = decode_splits(B, Hkv, Lmax, d);
  cudaError_t e = launch_decode(q, k, v, o, lse, B, Hq, Hkv, Lmax, d, cache_len, scale,
                                static_cast<float*>(workspace), splits, err, wait_limit_ns(),
                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: shape not supported";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime error";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded device wait ran out";
  }
  return "FA_ERR_UNKNOWN";
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d) != FA_OK) return 0;
  const size_t rows = (size_t)B * H * N;
  return round_up(rows * sizeof(float), 256) + rows * (size_t)d * sizeof(float);
}

}  // extern "C"

namespace fa {
namespace {

// Dropout arguments as the kernels take them; threshold 0 is no dropout.
void set_dropout(Problem* p, int threshold, uint64_t seed, uint32_t offset) {
  p->drop_threshold = threshold;
  p->drop_seed_lo = static_cast<uint32_t>(seed);
  p->drop_seed_hi = static_cast<uint32_t>(seed >> 32);
  p->drop_offset = offset;
  p->drop_scale = 256.f / static_cast<float>(256 - threshold);
}

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, int causal,
                   const uint8_t* blockmask, const int32_t* kv_len,
                   float scale, fa_dtype dtype, void* stream,
                   int drop_threshold, uint64_t seed, uint32_t offset) {
  fa_status st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  int* err = error_word();
  if (!err) return FA_ERR_CUDA;
  Problem p{B, H, N, d, causal ? 1 : 0, blockmask, kv_len, scale, err, wait_limit_ns()};
  set_dropout(&p, drop_threshold, seed, offset);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = dtype == FA_BF16 ? launch_fwd_sm103(p, q, k, v, o, lse, s)
                                   : launch_fwd_simt(p, dtype, q, k, v, o, lse, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, int causal,
                 const uint8_t* blockmask, const int32_t* kv_len,
                 float scale, fa_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, causal, blockmask, kv_len, scale, dtype, stream,
                  0, 0, 0);
}

fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, int causal,
                         const uint8_t* blockmask, const int32_t* kv_len,
                         float scale, fa_dtype dtype, int drop_threshold,
                         unsigned long long seed, unsigned int offset, void* stream) {
  if (drop_threshold < 0 || drop_threshold > 255) return FA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, N, d, causal, blockmask, kv_len, scale, dtype, stream,
                  drop_threshold, seed, offset);
}

namespace {

struct Workspace {
  float* Dsum;
  float* dq_acc;
};

Workspace carve(void* workspace, int B, int H, int N) {
  const size_t rows = (size_t)B * H * N;
  Workspace w;
  w.Dsum = static_cast<float*>(workspace);
  w.dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                      fa::round_up(rows * sizeof(float), 256));
  return w;
}

fa_status check_common(int B, int H, int N, int d, fa_dtype dtype, void* workspace,
                       size_t workspace_bytes) {
  fa_status st = fa::check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
  if (workspace_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

bool bad_ptr(const void* p) { return !p || !fa::aligned16(p); }

fa_status check_masks_scale(const int32_t* kv_len, const float* lse, float scale) {
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0) return FA_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status to_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace

fa_status fa_bwd_preprocess(const void* o, const void* dO, int B, int H, int N, int d,
                            fa_dtype dtype, void* workspace, size_t workspace_bytes,
                            void* stream) {
  fa_status st = check_common(B, H, N, d, dtype, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  if (bad_ptr(o) || bad_ptr(dO)) return FA_ERR_INVALID_ARG;
  Problem p{B, H, N, d, 0, nullptr, nullptr, 1.f, nullptr, 0};
  Workspace w = carve(workspace, B, H, N);
  return to_status(launch_bwd_preprocess(p, dtype, o, dO, w.Dsum,
                                         dtype == FA_BF16 ? w.dq_acc : nullptr,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

fa_status bwd_main_impl(const void* q, const void* k, const void* v, const float* lse,
                        const void* dO, void* dq, void* dk, void* dv,
                        int B, int H, int N, int d, int causal,
                        const uint8_t* blockmask, const int32_t* kv_len,
                        float scale, fa_dtype dtype,
                        void* workspace, size_t workspace_bytes, void* stream,
                        int drop_threshold, uint64_t seed, uint32_t offset) {
  fa_status st = check_common(B, H, N, d, dtype, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  if (bad_ptr(q) || bad_ptr(k) || bad_ptr(v) || bad_ptr(dO) || bad_ptr(dk) || bad_ptr(dv))
    return FA_ERR_INVALID_ARG;
  if (dtype == FA_FP32 && bad_ptr(dq)) return FA_ERR_INVALID_ARG;
  st = check_masks_scale(kv_len, lse, scale);
  if (st != FA_OK) return st;
  int* err = fa::error_word();
  if (!err) return FA_ERR_CUDA;
  Problem p{B, H, N, d, causal ? 1 : 0, blockmask, kv_len, scale, err, wait_limit_ns()};
  fa::set_dropout(&p, drop_threshold, seed, offset);
  Workspace w = carve(workspace, B, H, N);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == FA_BF16)
    return to_status(launch_bwd_sm103(p, q, k, v, lse, dO, w.Dsum, w.dq_acc, dk, dv, s));
  return to_status(launch_bwd_simt(p, dtype, q, k, v, lse, dO, w.Dsum, dq, dk, dv, s));
}

fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv,
                   int B, int H, int N, int d, int causal,
                   const uint8_t* blockmask, const int32_t* kv_len,
                   float scale, fa_dtype dtype,
                   void* workspace, size_t workspace_bytes, void* stream,
                   int drop_threshold, uint64_t seed, uint32_t offset) {
  fa_status st = check_common(B, H, N, d, dtype, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  if (bad_ptr(q) || bad_ptr(k) || bad_ptr(v) || bad_ptr(o) || bad_ptr(dO) || bad_ptr(dq) ||
      bad_ptr(dk) || bad_ptr(dv))
    return FA_ERR_INVALID_ARG;
  st = check_masks_scale(kv_len, lse, scale);
  if (st != FA_OK) return st;
  st = fa_bwd_preprocess(o, dO, B, H, N, d, dtype, workspace, workspace_bytes, stream);
  if (st != FA_OK) return st;
  st = bwd_main_impl(q, k, v, lse, dO, dq, dk, dv, B, H, N, d, causal, blockmask, kv_len, scale,
                     dtype, workspace, workspace_bytes, stream, drop_threshold, seed, offset);
  if (st != FA_OK) return st;
  return fa_bwd_dq_convert(dq, B, H, N, d, scale, dtype, workspace, workspace_bytes, stream);
}

}  // namespace

extern "C" {

fa_status fa_bwd_main(const void* q, const void* k, const void* v, const float* lse,
                      const void* dO, void* dq, void* dk, void* dv,
                      int B, int H, int N, int d, int causal,
                      const uint8_t* blockmask, const int32_t* kv_len,
                      float scale, fa_dtype dtype,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_main_impl(q, k, v, lse, dO, dq, dk, dv, B, H, N, d, causal, blockmask, kv_len,
                       scale, dtype, workspace, workspace_bytes, stream, 0, 0, 0);
}

fa_status fa_bwd_main_dropout(const void* q, const void* k, const void* v, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal,
                              const uint8_t* blockmask, const int32_t* kv_len,
                              float scale, fa_dtype dtype, int drop_threshold,
                              unsigned long long seed, unsigned int offset,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (drop_threshold < 0 || drop_threshold > 255) return FA_ERR_INVALID_ARG;
  return bwd_main_impl(q, k, v, lse, dO, dq, dk, dv, B, H, N, d, causal, blockmask, kv_len,
                       scale, dtype, workspace, workspace_bytes, stream, drop_threshold, seed,
                       offset);
}

fa_status fa_bwd_dq_convert(void* dq, int B, int H, int N, int d, float scale, fa_dtype dtype,
                            void* workspace, size_t workspace_bytes, void* stream) {
  fa_status st = check_common(B, H, N, d, dtype, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  if (bad_ptr(dq)) return FA_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dtype == FA_FP32) return FA_OK;
  Problem p{B, H, N, d, 0, nullptr, nullptr, scale, nullptr, 0};
  Workspace w = carve(workspace, B, H, N);
  return to_status(launch_dq_convert(p, w.dq_acc, dq, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, int causal,
                 const uint8_t* blockmask, const int32_t* kv_len,
                 float scale, fa_dtype dtype,
                 void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, blockmask, kv_len, scale,
                  dtype, workspace, workspace_bytes, stream, 0, 0, 0);
}

fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, int causal,
                         const uint8_t* blockmask, const int32_t* kv_len,
                         float scale, fa_dtype dtype, int drop_threshold,
                         unsigned long long seed, unsigned int offset,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (drop_threshold < 0 || drop_threshold > 255) return FA_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, blockmask, kv_len, scale,
                  dtype, workspace, workspace_bytes, stream, drop_threshold, seed, offset);
}

fa_status fa_dropout_random_bytes(void* out, int BH, int n_q, int n_k, unsigned long long seed,
                                  unsigned int offset, void* stream) {
  if (!out || BH < 1 || n_q < 1 || n_k < 1 || BH > 65535) return FA_ERR_INVALID_ARG;
  if ((long long)n_q * n_k > (1ll << 31)) return FA_ERR_UNSUPPORTED;
  Problem p{1, BH, n_q, 64, 0, nullptr, nullptr, 1.f, nullptr, 0};
  set_dropout(&p, 0, seed, offset);
  return to_status(launch_dropout_bytes(p, static_cast<uint8_t*>(out), BH, n_q, n_k,
                                        static_cast<cudaStream_t>(stream)));
}

size_t fa_fp8_vt_bytes(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d) != FA_OK || d != 128) return 0;
  return static_cast<size_t>(B) * H * d * round_up(static_cast<size_t>(N), 128);
}

namespace {

fa_status check_fp8(int B, int H, int N, int d) {
  fa_status st = fa::check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  return d == 128 ? FA_OK : FA_ERR_UNSUPPORTED;
}

bool bad_scale(const float* s) { return !s || (reinterpret_cast<uintptr_t>(s) & 3u) != 0; }

}  // namespace

fa_status fa_fp8_quantize_qk(const void* x, void* x8, float* scale, int B, int H, int N, int d,
                             void* stream) {
  fa_status st = check_fp8(B, H, N, d);
  if (st != FA_OK) return st;
  if (bad_ptr(x) || bad_ptr(x8) || bad_scale(scale)) return FA_ERR_INVALID_ARG;
  return to_status(launch_fp8_quantize_rows(x, x8, scale, B * H, N,
                                            static_cast<cudaStream_t>(stream)));
}

fa_status fa_fp8_quantize_v(const void* v, void* vt8, float* scale, int B, int H, int N, int d,
                            void* stream) {
  fa_status st = check_fp8(B, H, N, d);
  if (st != FA_OK) return st;
  if (bad_ptr(v) || bad_ptr(vt8) || bad_scale(scale)) return FA_ERR_INVALID_ARG;
  return to_status(launch_fp8_quantize_v(v, vt8, scale, B * H, N,
                                         static_cast<cudaStream_t>(stream)));
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale,
                     const float* k_scale, const float* v_scale, void* o, float* lse,
                     int B, int H, int N, int d, int causal, const uint8_t* blockmask,
                     const int32_t* kv_len, float scale, void* stream) {
  fa_status st = check_fp8(B, H, N, d);
  if (st != FA_OK) return st;
  if (bad_ptr(q8) || bad_ptr(k8) || bad_ptr(vt8) || bad_ptr(o)) return FA_ERR_INVALID_ARG;
  if (bad_scale(q_scale) || bad_scale(k_scale) || bad_scale(v_scale)) return FA_ERR_INVALID_ARG;
  st = check_masks_scale(kv_len, lse, scale);
  if (st != FA_OK) return st;
  int* err = error_word();
  if (!err) return FA_ERR_CUDA;
  Problem p{B, H, N, d, causal ? 1 : 0, blockmask, kv_len, scale, err, wait_limit_ns()};
  return to_status(launch_fwd_fp8(p, q8, k8, vt8, q_scale, k_scale, v_scale, o, lse,
                                  static_cast<cudaStream_t>(stream)));
}

fa_status fa_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int* err = error_word();
  if (!err) return FA_ERR_CUDA;
  int host = 0;
  if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  return host == 0 ? FA_OK : static_cast<fa_status>(host);
}

}  // extern "C"
