/*
 * fa.h -- C ABI of the exact IO-aware attention library (libfa_gb300.so).
 *
 * What it computes (FlashAttention pages):
 *   forward  -- "How FlashAttention works for training" (aivaro.ru answer 474),
 *               sections 1 and 2.1: O = softmax(Q K^T * scale) V, computed tile by
 *               tile with a running row maximum and row sum (online softmax, FlashAttention
 *               reading guide arXiv 2205.14135, "Method", steps 1-4), never writing
 *               the N x N score or probability matrix to memory.  Besides O it writes the
 *               per-row logsumexp, the one statistic the backward needs (course week 13,
 *               step 2).
 *   backward -- answer page section 3.1 and course week 13, step 2: S and P are
 *               recomputed block by block from Q, K and the saved logsumexp; with
 *               D = rowsum(dO o O) the gradients are the chain-rule ones
 *               dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K,
 *               dK = scale dS^T Q.
 *   masks    -- causal (course week 13, step 2: key j visible to query i iff j <= i, tiles
 *               wholly above the diagonal are skipped) and block-sparse (reading guide,
 *               "Extension: block-sparse FlashAttention": a 0/1 mask over blocks; zero
 *               blocks are skipped).  Per-sequence key padding masks key j >= kv_len[b].
 *
 * Layout: Q, K, V, O, dO, dQ, dK, dV are dense row-major [B, H, N, d] (d innermost,
 * then N, then H, then B), element type given by `dtype`.  lse and the D row sums are
 * fp32 [B, H, N].  Only d = 64 and d = 128 are supported.
 *
 * Memory: every pointer (tensors, kv_len, blockmask, workspace) is a DEVICE pointer owned
 * by the caller; the library allocates no device memory per call.  Tensor pointers must be
 * 16-byte aligned.  Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 * NULL is the legacy default stream): outputs are valid once the stream has synchronised.
 * The kernels of fa_fwd, fa_fwd_dropout and the three backward stages are launched with
 * programmatic stream serialization: one may be scheduled while the previous kernel in the
 * stream is still running, but it reads and writes global memory only after that kernel
 * has completed, so stream order holds as for ordinary launches (also inside a captured
 * CUDA graph, which keeps the attribute).
 *
 * Errors: arguments are validated on the host before any launch; a failed check returns
 * FA_ERR_INVALID_ARG (bad pointer, size, alignment, dtype, workspace) or FA_ERR_UNSUPPORTED
 * (a shape the kernels do not cover) and launches nothing.  A launch failure reported by the
 * CUDA runtime returns FA_ERR_CUDA; so does a tensor-core kernel that was built with another
 * register count than its in-kernel register split assumes (the first call on a device
 * checks it and then launches nothing).  Device-side faults surface at the caller's next
 * synchronisation.  A bounded wait inside a kernel that runs out records FA_ERR_TIMEOUT in
 * the library's device error word, readable with fa_device_error().
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_CUDA = 3,
  FA_ERR_TIMEOUT = 4
} fa_status;

typedef enum {
  FA_BF16 = 0, /* bf16 tensors; tcgen05 tensor-core kernels, fp32 accumulation */
  FA_FP32 = 1  /* fp32 tensors; fp32 CUDA-core kernels                          */
} fa_dtype;

/* Block-mask granularity: one mask entry covers 128 query rows x 128 key columns. */
#define FA_MASK_BLOCK 128

/*
 * Forward pass.
 *   q, k, v   in : [B, H, N, d] of `dtype`.
 *   o         out: [B, H, N, d] of `dtype`, O = softmax(scale Q K^T + mask) V.
 *   lse       out: fp32 [B, H, N], natural-log logsumexp of each masked, scaled score row;
 *                  -inf for a row that sees no key (its O row is 0).
 *   causal       : nonzero = key j is visible to query i only when j <= i (top-left aligned).
 *   blockmask    : NULL, or device uint8 [nb, nb] with nb = ceil(N / 128), row-major, shared by
 *                  every (b, h); entry [I][J] = 0 hides keys 128J..128J+127 from queries
 *                  128I..128I+127 (the block is skipped).
 *   kv_len       : NULL, or device int32 [B]; keys j >= kv_len[b] are hidden from every query of
 *                  sequence b.  Values are clamped to [0, N] on the device.
 *   scale        : multiplier of Q K^T, normally 1/sqrt(d); must be finite and > 0.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, int causal,
                 const uint8_t* blockmask, const int32_t* kv_len,
                 float scale, fa_dtype dtype, void* stream);

/*
 * Bytes of device workspace fa_bwd needs: the fp32 row sums D [B, H, N] followed (at a
 * 256-byte aligned offset) by the fp32 dQ accumulator [B, H, N, d].  Returns 0 when the
 * sizes are invalid.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass for the loss gradient dO = dL/dO.
 *   q, k, v, o   in : as given to / returned by fa_fwd (same masks, same scale).
 *   lse          in : fp32 [B, H, N] as returned by fa_fwd.
 *   dO           in : [B, H, N, d] of `dtype`.
 *   dq, dk, dv   out: [B, H, N, d] of `dtype`.
 *   workspace       : device buffer of at least fa_bwd_workspace_bytes(B, H, N, d) bytes,
 *                     256-byte aligned; its contents on entry do not matter.
 * Rows that see no key (lse = -inf) contribute nothing to any gradient.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, int causal,
                 const uint8_t* blockmask, const int32_t* kv_len,
                 float scale, fa_dtype dtype,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three stages fa_bwd runs, in order, on `stream` (same arguments and workspace; the
 * workspace must not be reused by another call until the last stage has run):
 *   fa_bwd_preprocess  -- D = rowsum(dO o O) (fp32, into the workspace) and, for bf16,
 *                         zeroes the fp32 dQ accumulator;
 *   fa_bwd_main        -- recomputes S and P block by block and forms dK and dV (written
 *                         to dk, dv) and dQ (bf16: summed into the fp32 accumulator;
 *                         fp32: written to dq directly);
 *   fa_bwd_dq_convert  -- bf16: dq = bf16(scale * accumulator); fp32: nothing to do.
 * They exist so that each kernel can be timed on its own; fa_bwd is their composition.
 */
fa_status fa_bwd_preprocess(const void* o, const void* dO, int B, int H, int N, int d,
                            fa_dtype dtype, void* workspace, size_t workspace_bytes,
                            void* stream);
fa_status fa_bwd_main(const void* q, const void* k, const void* v, const float* lse,
                      const void* dO, void* dq, void* dk, void* dv,
                      int B, int H, int N, int d, int causal,
                      const uint8_t* blockmask, const int32_t* kv_len,
                      float scale, fa_dtype dtype,
                      void* workspace, size_t workspace_bytes, void* stream);
fa_status fa_bwd_dq_convert(void* dq, int B, int H, int N, int d, float scale, fa_dtype dtype,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Size of the library's built-in backward scratch array (64 MiB): the largest
 * fa_bwd_workspace_bytes(B, H, N, d) that fa_bwd_noalloc accepts.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * fa_bwd without a caller-supplied workspace.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory -- code running inside
 * another framework's memory pool without access to its allocator, plug-ins and embedded
 * runtimes whose device memory is planned up front, or hooks where a cudaMalloc would
 * synchronise the device or is not allowed.  It allocates nothing: the workspace is a
 * fixed FA_NOALLOC_SCRATCH_BYTES array in the library's own device memory, which every
 * GPU that loads the library holds until the process exits.
 *   Arguments, layouts and results are those of fa_bwd minus the workspace.
 *   Returns FA_ERR_UNSUPPORTED, launching nothing, when fa_bwd_workspace_bytes(B, H, N, d)
 *   exceeds FA_NOALLOC_SCRATCH_BYTES; other errors as fa_bwd.
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *   with that device current); make that first call before any stream capture.
 *   All calls share the array and it keeps the last call's contents; every call rewrites
 *   D and zeroes the dQ accumulator before using them.  Calls whose work overlaps on the
 *   GPU (for example on two streams) race on the array: serialise them.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, int causal,
                         const uint8_t* blockmask, const int32_t* kv_len,
                         float scale, fa_dtype dtype, void* stream);

/*
 * Decode attention over a key/value cache with grouped key/value heads: one new query token
 * per sequence (course page week 13, step 1, the bullet on attention in decode: every
 * sequence has its own cache, the step reads it once at about Hq / Hkv FLOP per byte).
 *   q         in : bf16 [B, Hq, d], the new tokens' queries.
 *   k, v      in : bf16 [B, Hkv, Lmax, d], the caches; query head h reads key/value head
 *                  h / (Hq / Hkv) (contiguous groups).
 *   cache_len in : NULL (every sequence has Lmax keys) or device int32 [B]; keys
 *                  j >= cache_len[b] are ignored and never read into the result, whatever
 *                  those rows hold.  Values are clamped to [0, Lmax] on the device.
 *   o         out: bf16 [B, Hq, d] = softmax(scale q K^T) V over the visible keys; 0 for a
 *                  sequence with no key.
 *   lse       out: fp32 [B, Hq], natural-log logsumexp of the scaled scores (-inf: no key).
 *   scale        : multiplier of q K^T, normally 1/sqrt(d); finite and > 0.
 *   workspace    : device buffer of at least fa_decode_workspace_bytes(B, Hq, Hkv, Lmax, d)
 *                  bytes, 16-byte aligned, for the per-split fp32 partial results; its
 *                  contents on entry do not matter.
 * Supported: d in {64, 128}; Hq / Hkv in {1, 2, 4, 8} (FA_ERR_UNSUPPORTED otherwise);
 * Hq must be a multiple of Hkv (FA_ERR_INVALID_ARG otherwise).  Two kernels run on
 * `stream`: the split kernel and the combine kernel.
 */
size_t fa_decode_workspace_bytes(int B, int Hq, int Hkv, int Lmax, int d);
fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int Hq, int Hkv, int Lmax, int d, const int32_t* cache_len,
                    float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 (e4m3) forward, d = 128 only (FA_ERR_UNSUPPORTED otherwise).  The pages name FP8
 * operands as a FlashAttention-3 feature (answer page "How FlashAttention works for
 * training", section 7; course week 13, step 2) without further detail.  Here both
 * products take e4m3 operands on the tensor cores (tcgen05 kind::f8f6f4, fp32 accumulation);
 * the probabilities P are rounded to e4m3 for the P V product, the row sums use them
 * unrounded.  Encoding: x = s * e4m3(x / s) with power-of-two scales s = 2^k, k the smallest
 * integer with max|x| <= 448 * 2^k over the scale's block (round to nearest even, saturating).
 * Inputs must be finite.
 *
 * fa_fp8_quantize_qk: x bf16 [B, H, N, 128] -> x8 e4m3 bytes [B, H, N, 128] (same layout)
 *   and scale fp32 [B, H, ceil(N / 128)], one per block of 128 rows.  For Q and K.
 * fa_fp8_quantize_v: v bf16 [B, H, N, 128] -> vt8, e4m3 bytes of V transposed, [B, H, 128,
 *   Np] with Np = ceil(N / 128) * 128 (fa_fp8_vt_bytes() bytes in all; columns past N are 0),
 *   and scale fp32 [B, H], one per head.  Within each block of 128 keys, column k holds key
 *   32(k>>5) + 16((k>>2)&1) + 8((k>>1)&1) + 2((k>>3)&3) + (k&1) of the block: the order in
 *   which the forward's softmax threads hold P.  Treat vt8 as opaque input to fa_fwd_fp8.
 *   Three kernels and one memset run on `stream`; `scale` is overwritten in between.
 * fa_fwd_fp8: O and lse as fa_fwd (bf16 O [B, H, N, 128], fp32 lse [B, H, N]) of
 *   softmax(scale Q K^T + mask) V with Q = q_scale * q8, K = k_scale * k8, V = v_scale * V8
 *   decoded per block / per head; masks, kv_len and scale as fa_fwd.
 * Every pointer is a device pointer; tensors 16-byte aligned, scale arrays 4-byte aligned.
 */
size_t fa_fp8_vt_bytes(int B, int H, int N, int d);
fa_status fa_fp8_quantize_qk(const void* x, void* x8, float* scale, int B, int H, int N, int d,
                             void* stream);
fa_status fa_fp8_quantize_v(const void* v, void* vt8, float* scale, int B, int H, int N, int d,
                            void* stream);
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale,
                     const float* k_scale, const float* v_scale, void* o, float* lse,
                     int B, int H, int N, int d, int causal, const uint8_t* blockmask,
                     const int32_t* kv_len, float scale, void* stream);

/*
 * Attention with dropout on the probabilities.  The reading guide (arXiv 2205.14135, "Key
 * ideas", kernel fusion) lists dropout among the steps fused into the one attention kernel;
 * the reading taken here is inverted dropout on P:
 *   O = (P o Z) V / (1 - p),   p = drop_threshold / 256,
 * with lse that of the undropped softmax.  The backward regenerates Z instead of reading a
 * stored mask and computes dV = (P o Z)^T dO / (1 - p), dS = P o (Z o dP / (1 - p) - D),
 * D = rowsum(dO o O) of the dropped O, dQ and dK as fa_bwd.
 *   drop_threshold : 0..255 (FA_ERR_INVALID_ARG otherwise); element (b, h, i, j) is dropped
 *                    when its generator byte u is below it; 0 keeps everything.
 *   seed, offset   : Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2,
 *                    3", SC 2011) with key (seed mod 2^32, seed >> 32) and counter
 *                    (kappa, rho, b H + h, offset), rho = 8 (i >> 4) + (i & 7),
 *                    kappa = 4 (j >> 5) + ((j >> 1) & 3); u is byte 2 ((i >> 3) & 1) + (j & 1)
 *                    of output word (j >> 3) & 3.  The forward and backward of one step must
 *                    get the same (drop_threshold, seed, offset).
 * Every other argument, layout, result and error as fa_fwd / fa_bwd / fa_bwd_main; the bf16
 * and fp32 paths both support dropout.  fa_bwd_main_dropout is the middle stage of
 * fa_bwd_dropout (fa_bwd_preprocess and fa_bwd_dq_convert are shared with fa_bwd).
 */
fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, int causal,
                         const uint8_t* blockmask, const int32_t* kv_len,
                         float scale, fa_dtype dtype, int drop_threshold,
                         unsigned long long seed, unsigned int offset, void* stream);
fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, int causal,
                         const uint8_t* blockmask, const int32_t* kv_len,
                         float scale, fa_dtype dtype, int drop_threshold,
                         unsigned long long seed, unsigned int offset,
                         void* workspace, size_t workspace_bytes, void* stream);
fa_status fa_bwd_main_dropout(const void* q, const void* k, const void* v, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal,
                              const uint8_t* blockmask, const int32_t* kv_len,
                              float scale, fa_dtype dtype, int drop_threshold,
                              unsigned long long seed, unsigned int offset,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * The dropout generator's byte u(bh, i, j) of every element of a [BH, n_q, n_k] block, for
 * inspecting a mask (dropped where u < drop_threshold).  out: device uint8 [BH, n_q, n_k],
 * row-major; BH <= 65535, n_q * n_k <= 2^31 (FA_ERR_UNSUPPORTED otherwise).  Asynchronous on
 * `stream`.
 */
fa_status fa_dropout_random_bytes(void* out, int BH, int n_q, int n_k, unsigned long long seed,
                                  unsigned int offset, void* stream);

/*
 * Attention split over key/value shards of one sequence (sequence sharding).
 *
 * The FlashAttention reading guide (arXiv 2205.14135) merges the softmax statistics of a
 * vector split into parts ("Method": m = max(m1, m2), l = e^{m1 - m} l1 + e^{m2 - m} l2)
 * and names attention over several GPUs as open work ("Limitations").  When the keys and
 * values of a sequence are split into S shards, fa_fwd on (the queries, one shard) gives a
 * partial (O_k, lse_k) normalised over that shard's keys; fa_attn_merge combines them:
 *   lse = ln sum_k e^{lse_k},   O = sum_k e^{lse_k - lse} O_k,
 * which is the attention over all the keys.  For the backward, fa_bwd_preprocess of the
 * merged (O, dO) gives D and zeroes the dQ accumulator; fa_bwd_main with the merged lse
 * then runs once per shard, adding each shard's dQ contribution to the same accumulator and
 * writing that shard's dK, dV contributions; fa_grad_accumulate sums contributions to a
 * shard's dK, dV that come from several query shards, fa_grad_finish rounds a sum to the
 * output type, and fa_bwd_dq_convert finishes dQ.
 */

/* Largest number of partial results fa_attn_merge accepts. */
#define FA_MERGE_MAX_PARTS 1024

/*
 * Merge S partial results of the same query rows over disjoint key sets.
 *   o_parts  in : [S, B, H, N, d] of `dtype` (part k at o_parts + k * B*H*N*d), each part
 *                 normalised over its own keys (a fa_fwd output); 16-byte aligned.
 *   lse_parts in: fp32 [S, B, H, N], the parts' logsumexps; -inf where a part has no
 *                 visible key (that part then weighs nothing).
 *   o        out: [B, H, N, d] of `dtype`; 0 in a row that no part sees.
 *   lse      out: fp32 [B, H, N]; -inf in a row that no part sees.
 *   S             1 .. FA_MERGE_MAX_PARTS.  d = 64 or 128.  o must not alias o_parts.
 * Returns FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED before launching on a bad argument.
 */
fa_status fa_attn_merge(const void* o_parts, const float* lse_parts, int S, void* o, float* lse,
                        int B, int H, int N, int d, fa_dtype dtype, void* stream);

/*
 * acc[i] += x[i] for i < n: fp32 running sum of gradient contributions (for example the dK of
 * one key shard from several query shards).  acc: device fp32, 16-byte aligned; x: device,
 * `dtype` elements, 8-byte (bf16) or 16-byte (fp32) aligned; n a positive multiple of 4.
 */
fa_status fa_grad_accumulate(float* acc, const void* x, long long n, fa_dtype dtype,
                             void* stream);

/*
 * out[i] = acc[i] rounded once (round-to-nearest-even) to `dtype`, for i < n.  Alignment and
 * n as for fa_grad_accumulate.
 */
fa_status fa_grad_finish(void* out, const float* acc, long long n, fa_dtype dtype, void* stream);

/* Static, human-readable name of a status code (never NULL). */
const char* fa_status_string(fa_status s);

/*
 * Synchronises `stream`, then reads and clears the device error word of the current
 * device: FA_OK if no kernel recorded an error, FA_ERR_TIMEOUT if a bounded wait ran out,
 * FA_ERR_CUDA if the synchronisation itself failed.
 */
fa_status fa_device_error(void* stream);

/*
 * Self-test of failure detection (no counterpart on the pages; for tests and diagnostics).
 * Launches one warp that waits, with the bounded mbarrier wait the attention kernels use,
 * on a barrier nothing ever arrives on.  After `limit_ms` milliseconds (1..10000) the wait
 * gives up and records FA_ERR_TIMEOUT in the device error word, which the next
 * fa_device_error(stream) returns (and clears).  Uses no TMA and no tensor memory; the
 * context stays usable.  Returns FA_ERR_INVALID_ARG for a limit out of range.
 */
fa_status fa_selftest_wait_timeout(unsigned int limit_ms, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
