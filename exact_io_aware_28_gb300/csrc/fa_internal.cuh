// Internal declarations shared by the translation units of libfa_gb300.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "fa.h"

namespace fa {

constexpr int kMaskBlock = FA_MASK_BLOCK;

// Problem description handed from the C-ABI layer to the launchers.  Pointers are
// device pointers; element pointers are typed by the launcher.
struct Problem {
  int B, H, N, d;
  int causal;
  const uint8_t* blockmask;  // [nb, nb] or nullptr
  const int32_t* kv_len;     // [B] or nullptr
  float scale;
  int* err;                  // device error word
  unsigned long long wait_ns;  // bound of every mbarrier wait in the tensor-core kernels
  // Dropout on the probabilities (threshold 0: none): element (bh, i, j) is dropped when its
  // generator byte is below drop_threshold, kept ones are scaled by drop_scale.
  int drop_threshold = 0;
  uint32_t drop_seed_lo = 0, drop_seed_hi = 0, drop_offset = 0;
  float drop_scale = 1.f;    // 256 / (256 - drop_threshold)
};

// Bound of device-side waits: FA_WAIT_LIMIT_MS from the environment (read once), else 2 s.
unsigned long long wait_limit_ns();

// Device error codes written into the error word (match fa_status).
constexpr int kErrTimeout = FA_ERR_TIMEOUT;

// Launch of a kernel of the training step (forward, preprocess, backward main, dQ convert)
// with programmatic stream serialization: it may be scheduled while the previous kernel in
// the stream drains, runs its set-up (barriers, tensor memory, descriptor prefetch), and waits
// in griddep_wait before it touches global memory.  Every such kernel calls griddep_wait in
// every CTA before it can exit, so completion stays ordered along the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers.  Each returns cudaSuccess or the launch error.
cudaError_t launch_fwd_simt(const Problem& p, fa_dtype dt, const void* q, const void* k,
                            const void* v, void* o, float* lse, cudaStream_t s);
cudaError_t launch_bwd_simt(const Problem& p, fa_dtype dt, const void* q, const void* k,
                            const void* v, const float* lse, const void* dO, const float* D,
                            void* dq, void* dk, void* dv, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const Problem& p, fa_dtype dt, const void* o, const void* dO,
                                  float* D, float* dq_acc, cudaStream_t s);
cudaError_t launch_dq_convert(const Problem& p, const float* dq_acc, void* dq, cudaStream_t s);
cudaError_t launch_fwd_sm103(const Problem& p, const void* q, const void* k, const void* v,
                             void* o, float* lse, cudaStream_t s);
cudaError_t launch_bwd_sm103(const Problem& p, const void* q, const void* k, const void* v,
                             const float* lse, const void* dO, const float* D, float* dq_acc,
                             void* dk, void* dv, cudaStream_t s);

// Generator bytes of dropout for [BH, n_q, n_k] elements (fa_dropout.cu).
cudaError_t launch_dropout_bytes(const Problem& p, uint8_t* out, int BH, int n_q, int n_k,
                                 cudaStream_t s);

// Tensor map of a [B*H, N, d] bf16 tensor (d innermost) with 64 x 128 boxes and 128-byte
// swizzle; rows beyond N read as zero.  Returns false if the driver rejects it.
bool make_head_map(CUtensorMap* map, const void* ptr, int BH, int N, int d);
// The same view with 64-column boxes of `box_rows` rows (1..256).
bool make_head_map_rows(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows);

// Tensor map of a [BH, rows, inner] byte tensor (inner contiguous, a multiple of 16) with
// 128 x 128 boxes and 128-byte swizzle; bytes outside the tensor read as zero.
bool make_u8_map(CUtensorMap* map, const void* ptr, int BH, int rows, int inner);

// FP8 (e4m3) path, d = 128 (fa_fp8.cu): encoders and the forward.
cudaError_t launch_fp8_quantize_rows(const void* x, void* x8, float* scale, int BH, int N,
                                     cudaStream_t s);
cudaError_t launch_fp8_quantize_v(const void* v, void* vt8, float* scale, int BH, int N,
                                  cudaStream_t s);
cudaError_t launch_fwd_fp8(const Problem& p, const void* q8, const void* k8, const void* vt8,
                           const float* q_scale, const float* k_scale, const float* v_scale,
                           void* o, float* lse, cudaStream_t s);

// Decode over a key/value cache (split kernel + combine kernel); see fa_decode.cu.
cudaError_t launch_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int Lmax, int d, const int32_t* cache_len,
                          float scale, float* partials, int splits, int* err,
                          unsigned long long wait_ns, cudaStream_t s);
// Number of key splits per (sequence, key/value head) the decode uses on this device.
int decode_splits(int B, int Hkv, int Lmax, int d);
// The tensor-core split kernel (fa_decode_tc.cu, d = 64 or 128) and its number of splits.
int decode_tc_splits(int B, int Hkv, int Lmax);
cudaError_t launch_decode_tc(const void* q, const void* k, const void* v, int B, int Hq,
                             int Hkv, int Lmax, int d, const int32_t* cache_len, float scale,
                             float* part, int splits, int* err, unsigned long long wait_ns,
                             cudaStream_t s);

// Sequence sharding (fa_shard.cu): merge of partial (O, lse) results, fp32 gradient sums.
cudaError_t launch_merge(const void* o_parts, const float* lse_parts, int S, void* o, float* lse,
                         long long rows, int d, fa_dtype dt, cudaStream_t s);
cudaError_t launch_accumulate(float* acc, const void* x, long long n, fa_dtype dt,
                              cudaStream_t s);
cudaError_t launch_finish(void* out, const float* acc, long long n, fa_dtype dt, cudaStream_t s);

// Tensor map of a [B*H, N, d] fp32 accumulator with 32 x 32 boxes (128-byte swizzle), for bulk
// reduce-add; rows beyond N are outside the map.
bool make_acc_map(CUtensorMap* map, const void* ptr, int BH, int N, int d);

// Device address of the library's error word on the current device (nullptr on failure).
int* error_word();

// Number of SMs of the current device (cached per device).
int sm_count();

}  // namespace fa
