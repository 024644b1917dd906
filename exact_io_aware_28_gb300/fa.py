"""ctypes binding of libfa_gb300.so (names as in include/fa.h).

Argument marshalling only: every step of the attention path runs in the library's
CUDA kernels.  torch supplies device memory and the current stream.  If the library
has not been built, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_BF16, FA_FP32 = 0, 1

# Every symbol include/fa.h declares.
EXPORTS = ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_preprocess", "fa_bwd_main",
           "fa_bwd_dq_convert", "fa_bwd_noalloc", "fa_status_string", "fa_device_error",
           "fa_selftest_wait_timeout", "fa_decode_workspace_bytes", "fa_decode",
           "fa_fp8_vt_bytes", "fa_fp8_quantize_qk", "fa_fp8_quantize_v", "fa_fwd_fp8",
           "fa_fwd_dropout", "fa_bwd_dropout", "fa_bwd_main_dropout", "fa_dropout_random_bytes",
           "fa_attn_merge", "fa_grad_accumulate", "fa_grad_finish")

# Largest number of partial results fa_attn_merge accepts.
FA_MERGE_MAX_PARTS = 1024

# Largest workspace (bytes) fa_bwd_noalloc can serve from its built-in scratch array.
FA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)}")


_lib: Optional[ctypes.CDLL] = None


def load() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m exact_io_aware_28_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, F, I, P]
    lib.fa_fwd.restype = I
    lib.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, F, I, P, S, P]
    lib.fa_bwd.restype = I
    lib.fa_bwd_preprocess.argtypes = [P, P, I, I, I, I, I, P, S, P]
    lib.fa_bwd_preprocess.restype = I
    lib.fa_bwd_main.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, F, I, P, S, P]
    lib.fa_bwd_main.restype = I
    lib.fa_bwd_dq_convert.argtypes = [P, I, I, I, I, F, I, P, S, P]
    lib.fa_bwd_dq_convert.restype = I
    lib.fa_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, F, I, P]
    lib.fa_bwd_noalloc.restype = I
    lib.fa_bwd_workspace_bytes.argtypes = [I, I, I, I]
    lib.fa_bwd_workspace_bytes.restype = S
    lib.fa_status_string.argtypes = [I]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_device_error.argtypes = [P]
    lib.fa_device_error.restype = I
    lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
    lib.fa_selftest_wait_timeout.restype = I
    lib.fa_decode_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.fa_decode_workspace_bytes.restype = S
    lib.fa_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, P, F, P, S, P]
    lib.fa_decode.restype = I
    lib.fa_fp8_vt_bytes.argtypes = [I, I, I, I]
    lib.fa_fp8_vt_bytes.restype = S
    lib.fa_fp8_quantize_qk.argtypes = [P, P, P, I, I, I, I, P]
    lib.fa_fp8_quantize_qk.restype = I
    lib.fa_fp8_quantize_v.argtypes = [P, P, P, I, I, I, I, P]
    lib.fa_fp8_quantize_v.restype = I
    lib.fa_fwd_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, F, P]
    lib.fa_fwd_fp8.restype = I
    U64, U32 = ctypes.c_ulonglong, ctypes.c_uint
    lib.fa_fwd_dropout.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, F, I, I, U64, U32, P]
    lib.fa_fwd_dropout.restype = I
    lib.fa_bwd_dropout.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, F, I, I, U64,
                                   U32, P, S, P]
    lib.fa_bwd_dropout.restype = I
    lib.fa_bwd_main_dropout.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, F, I, I,
                                        U64, U32, P, S, P]
    lib.fa_bwd_main_dropout.restype = I
    lib.fa_dropout_random_bytes.argtypes = [P, I, I, I, U64, U32, P]
    lib.fa_dropout_random_bytes.restype = I
    L = ctypes.c_longlong
    lib.fa_attn_merge.argtypes = [P, P, I, P, P, I, I, I, I, I, P]
    lib.fa_attn_merge.restype = I
    lib.fa_grad_accumulate.argtypes = [P, P, L, I, P]
    lib.fa_grad_accumulate.restype = I
    lib.fa_grad_finish.argtypes = [P, P, L, I, P]
    lib.fa_grad_finish.restype = I
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    """Device address of ``t`` for the library (every tensor argument is device memory)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("the library takes CUDA tensors (device memory); got a "
                         f"{t.device.type} tensor")
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _check_dense(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, H, N, d]")


def fa_status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N, d))


def fa_device_error(stream=None) -> int:
    return int(load().fa_device_error(_stream(stream)))


def fa_selftest_wait_timeout(limit_ms: int, stream=None) -> None:
    """Launch the bounded-wait self-test; fa_device_error() then reports FA_ERR_TIMEOUT."""
    st = load().fa_selftest_wait_timeout(int(limit_ms), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_selftest_wait_timeout")


def fa_fwd(q, k, v, o, lse, causal: bool = False, blockmask=None, kv_len=None,
           scale: Optional[float] = None, stream=None) -> None:
    """O and lse for [B, H, N, d] tensors q, k, v (outputs o, lse preallocated)."""
    _check_dense(q, k, v, o, lse, blockmask, kv_len)
    B, H, N, d = q.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    st = load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(causal),
                       _ptr(blockmask), _ptr(kv_len), scale, _dtype_code(q), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd")


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, workspace, causal: bool = False, blockmask=None,
           kv_len=None, scale: Optional[float] = None, stream=None) -> None:
    """dq, dk, dv (preallocated) for the upstream gradient ``do``."""
    _check_dense(q, k, v, o, lse, do, dq, dk, dv, blockmask, kv_len)
    B, H, N, d = q.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                       _ptr(dk), _ptr(dv), B, H, N, d, int(causal), _ptr(blockmask),
                       _ptr(kv_len), scale, _dtype_code(q), _ptr(workspace), ws_bytes,
                       _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd")


def fa_bwd_preprocess(o, do, workspace, stream=None) -> None:
    B, H, N, d = o.shape
    st = load().fa_bwd_preprocess(_ptr(o), _ptr(do), B, H, N, d, _dtype_code(o),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_preprocess")


def fa_bwd_main(q, k, v, lse, do, dq, dk, dv, workspace, causal=False, blockmask=None,
                kv_len=None, scale=None, stream=None) -> None:
    _check_dense(q, k, v, lse, do, dq, dk, dv, blockmask, kv_len)
    B, H, N, d = q.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    st = load().fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                            _ptr(dv), B, H, N, d, int(causal), _ptr(blockmask), _ptr(kv_len),
                            scale, _dtype_code(q), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_main")


def fa_bwd_dq_convert(dq, workspace, scale=None, stream=None) -> None:
    B, H, N, d = dq.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    st = load().fa_bwd_dq_convert(_ptr(dq), B, H, N, d, scale, _dtype_code(dq), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_dq_convert")


def fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, causal: bool = False, blockmask=None,
                   kv_len=None, scale: Optional[float] = None, stream=None) -> None:
    """fa_bwd with the library's built-in scratch array instead of a workspace.

    For callers that cannot allocate device memory.  Problems whose workspace would exceed
    FA_NOALLOC_SCRATCH_BYTES are rejected; calls that overlap on the GPU share the array
    and race, so serialise them.
    """
    _check_dense(q, k, v, o, lse, do, dq, dk, dv, blockmask, kv_len)
    B, H, N, d = q.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    st = load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, int(causal),
                               _ptr(blockmask), _ptr(kv_len), scale, _dtype_code(q),
                               _stream(stream))
    if st != FA_OK:
        need = fa_bwd_workspace_bytes(B, H, N, d)
        if st == FA_ERR_UNSUPPORTED and need > FA_NOALLOC_SCRATCH_BYTES:
            raise FaError(st, f"fa_bwd_noalloc: needs {need} bytes of scratch, the built-in "
                              f"array holds {FA_NOALLOC_SCRATCH_BYTES}")
        raise FaError(st, "fa_bwd_noalloc")


# ----------------------------------------------------------- allocating helpers

def alloc_workspace(B: int, H: int, N: int, d: int, device="cuda") -> torch.Tensor:
    n = fa_bwd_workspace_bytes(B, H, N, d)
    if n == 0:
        raise FaError(FA_ERR_INVALID_ARG, "fa_bwd_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward(q, k, v, causal=False, blockmask=None, kv_len=None, scale=None, stream=None):
    """Allocate O and lse with torch and run fa_fwd.  Returns (o, lse)."""
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, causal, blockmask, kv_len, scale, stream)
    return o, lse


def backward(q, k, v, o, lse, do, causal=False, blockmask=None, kv_len=None, scale=None,
             workspace=None, stream=None):
    """Allocate dQ, dK, dV (and the workspace unless given) and run fa_bwd."""
    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = alloc_workspace(B, H, N, d, q.device)
    fa_bwd(q, k, v, o, lse, do, dq, dk, dv, workspace, causal, blockmask, kv_len, scale, stream)
    return dq, dk, dv


# ----------------------------------------------------------- decode

def fa_decode_workspace_bytes(B: int, Hq: int, Hkv: int, Lmax: int, d: int) -> int:
    return int(load().fa_decode_workspace_bytes(B, Hq, Hkv, Lmax, d))


def fa_decode(q, k, v, o, lse, workspace, cache_len=None, scale=None, stream=None):
    """q [B, Hq, d], k/v [B, Hkv, Lmax, d] bf16; o [B, Hq, d] bf16, lse [B, Hq] fp32 out."""
    _check_dense(q, k, v, o, lse, cache_len, workspace)
    B, Hq, d = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("decode takes bf16 q, k, v")
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    st = load().fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Lmax, d,
                          _ptr(cache_len), float(scale), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_decode")


def decode(q, k, v, cache_len=None, scale=None, workspace=None, stream=None):
    """Allocate o, lse (and the workspace unless given) with torch and run fa_decode."""
    B, Hq, d = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = fa_decode_workspace_bytes(B, Hq, Hkv, Lmax, d)
        if n == 0:
            raise FaError(FA_ERR_INVALID_ARG, "fa_decode_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    fa_decode(q, k, v, o, lse, workspace, cache_len, scale, stream)
    return o, lse


def fa_fp8_vt_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_fp8_vt_bytes(B, H, N, d))


def _need_bf16(*ts):
    for t in ts:
        if t.dtype != torch.bfloat16:
            raise TypeError("the FP8 encoders take bf16 tensors")


def fa_fp8_quantize_qk(x, x8, scale, stream=None) -> None:
    """x bf16 [B, H, N, 128] -> x8 uint8 [B, H, N, 128], scale fp32 [B, H, ceil(N/128)]."""
    _check_dense(x, x8, scale)
    _need_bf16(x)
    B, H, N, d = x.shape
    st = load().fa_fp8_quantize_qk(_ptr(x), _ptr(x8), _ptr(scale), B, H, N, d, _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fp8_quantize_qk")


def fa_fp8_quantize_v(v, vt8, scale, stream=None) -> None:
    """v bf16 [B, H, N, 128] -> vt8 uint8 [B, H, 128, Np] (opaque key order), scale [B, H]."""
    _check_dense(v, vt8, scale)
    _need_bf16(v)
    B, H, N, d = v.shape
    st = load().fa_fp8_quantize_v(_ptr(v), _ptr(vt8), _ptr(scale), B, H, N, d, _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fp8_quantize_v")


def fa_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, causal=False, blockmask=None,
               kv_len=None, scale=None, stream=None) -> None:
    """O (bf16, preallocated) and lse of attention on e4m3-encoded inputs."""
    _check_dense(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, blockmask, kv_len)
    B, H, N, d = q8.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    st = load().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(q_scale), _ptr(k_scale),
                           _ptr(v_scale), _ptr(o), _ptr(lse), B, H, N, d, int(causal),
                           _ptr(blockmask), _ptr(kv_len), scale, _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8")


def fp8_quantize_qk(x, stream=None):
    """Allocate and encode: returns (x8 uint8 [B, H, N, 128], scale fp32 [B, H, nb])."""
    B, H, N, d = x.shape
    x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    scale = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=x.device)
    fa_fp8_quantize_qk(x, x8, scale, stream)
    return x8, scale


def fp8_quantize_v(v, stream=None):
    """Allocate and encode: returns (vt8 uint8 [B, H, 128, Np], scale fp32 [B, H])."""
    B, H, N, d = v.shape
    Np = (N + 127) // 128 * 128
    vt8 = torch.empty((B, H, d, Np), dtype=torch.uint8, device=v.device)
    scale = torch.empty((B, H), dtype=torch.float32, device=v.device)
    fa_fp8_quantize_v(v, vt8, scale, stream)
    return vt8, scale


def forward_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, causal=False, blockmask=None,
                kv_len=None, scale=None, stream=None):
    """Allocate o (bf16) and lse with torch and run fa_fwd_fp8."""
    B, H, N, d = q8.shape
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    fa_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, causal, blockmask, kv_len,
               scale, stream)
    return o, lse


def attention_fp8(q, k, v, causal=False, blockmask=None, kv_len=None, scale=None, stream=None):
    """bf16 q, k, v -> (o, lse) with e4m3 tensor-core products: encode, then the forward."""
    q8, sq = fp8_quantize_qk(q, stream)
    k8, sk = fp8_quantize_qk(k, stream)
    vt8, sv = fp8_quantize_v(v, stream)
    return forward_fp8(q8, k8, vt8, sq, sk, sv, causal, blockmask, kv_len, scale, stream)


# ----------------------------------------------------------- dropout

def _drop_args(drop_threshold: int, seed: int, offset: int):
    t = int(drop_threshold)
    if not 0 <= t <= 255:
        raise ValueError("drop_threshold must be in [0, 255] (drop probability t / 256)")
    return t, int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 32 - 1)


def fa_fwd_dropout(q, k, v, o, lse, drop_threshold: int, seed: int, offset: int = 0,
                   causal: bool = False, blockmask=None, kv_len=None,
                   scale: Optional[float] = None, stream=None) -> None:
    """fa_fwd with dropout on P: element (b, h, i, j) is dropped with probability t / 256
    (its Philox4x32-10 byte below t), kept ones are scaled by 256 / (256 - t)."""
    _check_dense(q, k, v, o, lse, blockmask, kv_len)
    B, H, N, d = q.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    t, sd, off = _drop_args(drop_threshold, seed, offset)
    st = load().fa_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                               int(causal), _ptr(blockmask), _ptr(kv_len), scale,
                               _dtype_code(q), t, sd, off, _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_dropout")


def fa_bwd_dropout(q, k, v, o, lse, do, dq, dk, dv, workspace, drop_threshold: int, seed: int,
                   offset: int = 0, causal: bool = False, blockmask=None, kv_len=None,
                   scale: Optional[float] = None, stream=None) -> None:
    """Gradients of the dropped forward; the same (threshold, seed, offset) regenerate the
    mask."""
    _check_dense(q, k, v, o, lse, do, dq, dk, dv, blockmask, kv_len)
    B, H, N, d = q.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    t, sd, off = _drop_args(drop_threshold, seed, offset)
    st = load().fa_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, int(causal),
                               _ptr(blockmask), _ptr(kv_len), scale, _dtype_code(q), t, sd, off,
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_dropout")


def fa_bwd_main_dropout(q, k, v, lse, do, dq, dk, dv, workspace, drop_threshold: int,
                        seed: int, offset: int = 0, causal=False, blockmask=None, kv_len=None,
                        scale=None, stream=None) -> None:
    _check_dense(q, k, v, lse, do, dq, dk, dv, blockmask, kv_len)
    B, H, N, d = q.shape
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    t, sd, off = _drop_args(drop_threshold, seed, offset)
    st = load().fa_bwd_main_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(do), _ptr(dq),
                                    _ptr(dk), _ptr(dv), B, H, N, d, int(causal),
                                    _ptr(blockmask), _ptr(kv_len), scale, _dtype_code(q), t, sd,
                                    off, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_main_dropout")


def fa_dropout_random_bytes(out, seed: int, offset: int = 0, stream=None) -> None:
    """The generator byte of every element of a [BH, n_q, n_k] uint8 tensor ``out``."""
    if out.dtype != torch.uint8 or out.dim() != 3 or not out.is_contiguous():
        raise ValueError("out must be a contiguous uint8 [BH, n_q, n_k] tensor")
    BH, n_q, n_k = out.shape
    _, sd, off = _drop_args(0, seed, offset)
    st = load().fa_dropout_random_bytes(_ptr(out), BH, n_q, n_k, sd, off, _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_dropout_random_bytes")


def forward_dropout(q, k, v, drop_threshold, seed, offset=0, causal=False, blockmask=None,
                    kv_len=None, scale=None, stream=None):
    """Allocate O and lse with torch and run fa_fwd_dropout.  Returns (o, lse)."""
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd_dropout(q, k, v, o, lse, drop_threshold, seed, offset, causal, blockmask, kv_len,
                   scale, stream)
    return o, lse


def backward_dropout(q, k, v, o, lse, do, drop_threshold, seed, offset=0, causal=False,
                     blockmask=None, kv_len=None, scale=None, workspace=None, stream=None):
    """Allocate dQ, dK, dV (and the workspace unless given) and run fa_bwd_dropout."""
    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = alloc_workspace(B, H, N, d, q.device)
    fa_bwd_dropout(q, k, v, o, lse, do, dq, dk, dv, workspace, drop_threshold, seed, offset,
                   causal, blockmask, kv_len, scale, stream)
    return dq, dk, dv


# ----------------------------------------------------------- sequence sharding

def fa_attn_merge(o_parts, lse_parts, o, lse, stream=None) -> None:
    """Merge S partial (O, lse) results of the same rows over disjoint key sets:
    o_parts [S, B, H, N, d], lse_parts fp32 [S, B, H, N] -> o [B, H, N, d], lse [B, H, N]."""
    _check_dense(o_parts, lse_parts, o, lse)
    S, B, H, N, d = o_parts.shape
    if tuple(lse_parts.shape) != (S, B, H, N) or lse_parts.dtype != torch.float32:
        raise ValueError("lse_parts must be fp32 [S, B, H, N]")
    if o.dtype != o_parts.dtype:
        raise TypeError("o and o_parts must have the same dtype")
    st = load().fa_attn_merge(_ptr(o_parts), _ptr(lse_parts), S, _ptr(o), _ptr(lse), B, H, N, d,
                              _dtype_code(o_parts), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_attn_merge")


def fa_grad_accumulate(acc, x, stream=None) -> None:
    """acc (fp32) += x (bf16 or fp32, same number of elements)."""
    _check_dense(acc, x)
    if acc.dtype != torch.float32 or acc.numel() != x.numel():
        raise ValueError("acc must be fp32 with as many elements as x")
    st = load().fa_grad_accumulate(_ptr(acc), _ptr(x), acc.numel(), _dtype_code(x),
                                   _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_grad_accumulate")


def fa_grad_finish(out, acc, stream=None) -> None:
    """out (bf16 or fp32) = acc (fp32) rounded once."""
    _check_dense(acc, out)
    if acc.dtype != torch.float32 or acc.numel() != out.numel():
        raise ValueError("acc must be fp32 with as many elements as out")
    st = load().fa_grad_finish(_ptr(out), _ptr(acc), acc.numel(), _dtype_code(out),
                               _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_grad_finish")
