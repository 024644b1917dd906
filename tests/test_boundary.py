"""The C-ABI library: it loads, exports what include/fa.h declares, and rejects bad
arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from exact_io_aware_28_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

pytestmark = pytest.mark.skipif(not os.path.exists(fa.LIB_PATH),
                                reason="libfa_gb300.so not built")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(fa.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    for code in range(5):
        assert fa.fa_status_string(code).startswith("FA_")
    assert "UNKNOWN" in fa.fa_status_string(99)


def test_workspace_bytes():
    B, H, N, d = 1, 32, 16384, 128
    rows = B * H * N
    assert fa.fa_bwd_workspace_bytes(B, H, N, d) == rows * 4 + rows * d * 4
    assert fa.fa_bwd_workspace_bytes(1, 1, 7, 64) == 256 + 7 * 64 * 4
    assert fa.fa_bwd_workspace_bytes(1, 1, 0, 64) == 0
    assert fa.fa_bwd_workspace_bytes(1, 1, 8, 96) == 0


A = 0x10000  # a fake, 16-byte aligned address: never dereferenced on the host


def fwd(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=64, causal=0, bm=None,
                kv=None, scale=0.125, dtype=fa.FA_BF16)
    args.update(kw)
    lib = fa.load()
    return lib.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                      args["H"], args["N"], args["d"], args["causal"], args["bm"], args["kv"],
                      args["scale"], args["dtype"], None)


def bwd(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, do=A, dq=A, dk=A, dv=A, B=1, H=1, N=128, d=64,
                causal=0, bm=None, kv=None, scale=0.125, dtype=fa.FA_BF16, ws=A,
                wsb=1 << 30)
    args.update(kw)
    lib = fa.load()
    return lib.fa_bwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["do"],
                      args["dq"], args["dk"], args["dv"], args["B"], args["H"], args["N"],
                      args["d"], args["causal"], args["bm"], args["kv"], args["scale"],
                      args["dtype"], args["ws"], args["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    ({"q": None}, fa.FA_ERR_INVALID_ARG),
    ({"lse": None}, fa.FA_ERR_INVALID_ARG),
    ({"N": 0}, fa.FA_ERR_INVALID_ARG),
    ({"B": 0}, fa.FA_ERR_INVALID_ARG),
    ({"d": 96}, fa.FA_ERR_UNSUPPORTED),
    ({"d": 256}, fa.FA_ERR_UNSUPPORTED),
    ({"k": A + 8}, fa.FA_ERR_INVALID_ARG),
    ({"o": A + 2}, fa.FA_ERR_INVALID_ARG),
    ({"lse": A + 1}, fa.FA_ERR_INVALID_ARG),
    ({"kv": A + 2}, fa.FA_ERR_INVALID_ARG),
    ({"dtype": 7}, fa.FA_ERR_INVALID_ARG),
    ({"scale": float("nan")}, fa.FA_ERR_INVALID_ARG),
    ({"scale": float("inf")}, fa.FA_ERR_INVALID_ARG),
    ({"scale": 0.0}, fa.FA_ERR_INVALID_ARG),
    ({"scale": -0.125}, fa.FA_ERR_INVALID_ARG),
    ({"B": 300, "H": 300}, fa.FA_ERR_UNSUPPORTED),
])
def test_fwd_rejects_bad_arguments(kw, code):
    assert fwd(**kw) == code


@pytest.mark.parametrize("kw,code", [
    ({"do": None}, fa.FA_ERR_INVALID_ARG),
    ({"ws": None}, fa.FA_ERR_INVALID_ARG),
    ({"dq": A + 4}, fa.FA_ERR_INVALID_ARG),
    ({"ws": A + 16}, fa.FA_ERR_INVALID_ARG),
    ({"wsb": 1000}, fa.FA_ERR_INVALID_ARG),
    ({"d": 32}, fa.FA_ERR_UNSUPPORTED),
    ({"N": -5}, fa.FA_ERR_INVALID_ARG),
    ({"dtype": -1}, fa.FA_ERR_INVALID_ARG),
])
def test_bwd_rejects_bad_arguments(kw, code):
    assert bwd(**kw) == code


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        fa.load()


def dec(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=2, Hq=8, Hkv=2, L=300, d=128, cl=None,
                scale=0.088, ws=A, wsb=1 << 30)
    args.update(kw)
    lib = fa.load()
    return lib.fa_decode(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                         args["Hq"], args["Hkv"], args["L"], args["d"], args["cl"],
                         args["scale"], args["ws"], args["wsb"], None)


def test_decode_workspace_bytes():
    n = fa.fa_decode_workspace_bytes(2, 8, 2, 300, 128)
    per_split = 2 * 8 * (128 + 4) * 4
    assert n > 0 and n % per_split == 0
    assert fa.fa_decode_workspace_bytes(2, 8, 3, 300, 128) == 0   # 8 % 3 != 0
    assert fa.fa_decode_workspace_bytes(2, 8, 2, 300, 96) == 0
    assert fa.fa_decode_workspace_bytes(0, 8, 2, 300, 128) == 0


@pytest.mark.parametrize("kw,code", [
    ({"q": None}, fa.FA_ERR_INVALID_ARG),
    ({"ws": None}, fa.FA_ERR_INVALID_ARG),
    ({"wsb": 16}, fa.FA_ERR_INVALID_ARG),
    ({"Hkv": 3}, fa.FA_ERR_INVALID_ARG),          # query heads not a multiple of K/V heads
    ({"Hq": 12, "Hkv": 4}, fa.FA_ERR_UNSUPPORTED),  # three query heads per K/V head
    ({"Hq": 32, "Hkv": 2}, fa.FA_ERR_UNSUPPORTED),  # sixteen
    ({"d": 96}, fa.FA_ERR_UNSUPPORTED),
    ({"L": 0}, fa.FA_ERR_INVALID_ARG),
    ({"k": A + 8}, fa.FA_ERR_INVALID_ARG),
    ({"lse": A + 2}, fa.FA_ERR_INVALID_ARG),
    ({"cl": A + 1}, fa.FA_ERR_INVALID_ARG),
    ({"scale": 0.0}, fa.FA_ERR_INVALID_ARG),
    ({"scale": float("nan")}, fa.FA_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments(kw, code):
    assert dec(**kw) == code


def test_fp8_vt_bytes():
    assert fa.fa_fp8_vt_bytes(1, 2, 300, 128) == 2 * 128 * 384
    assert fa.fa_fp8_vt_bytes(1, 32, 16384, 128) == 32 * 128 * 16384
    assert fa.fa_fp8_vt_bytes(1, 2, 300, 64) == 0      # d = 128 only
    assert fa.fa_fp8_vt_bytes(1, 2, 0, 128) == 0


def fwd8(**kw):
    args = dict(q8=A, k8=A, vt8=A, sq=A, sk=A, sv=A, o=A, lse=A, B=1, H=2, N=300, d=128,
                causal=1, bm=None, kv=None, scale=0.088)
    args.update(kw)
    return fa.load().fa_fwd_fp8(args["q8"], args["k8"], args["vt8"], args["sq"], args["sk"],
                                args["sv"], args["o"], args["lse"], args["B"], args["H"],
                                args["N"], args["d"], args["causal"], args["bm"], args["kv"],
                                args["scale"], None)


@pytest.mark.parametrize("kw,code", [
    ({"q8": None}, fa.FA_ERR_INVALID_ARG),
    ({"vt8": A + 8}, fa.FA_ERR_INVALID_ARG),
    ({"o": A + 2}, fa.FA_ERR_INVALID_ARG),
    ({"sq": None}, fa.FA_ERR_INVALID_ARG),
    ({"sk": A + 2}, fa.FA_ERR_INVALID_ARG),
    ({"sv": None}, fa.FA_ERR_INVALID_ARG),
    ({"lse": None}, fa.FA_ERR_INVALID_ARG),
    ({"kv": A + 1}, fa.FA_ERR_INVALID_ARG),
    ({"d": 64}, fa.FA_ERR_UNSUPPORTED),
    ({"N": 0}, fa.FA_ERR_INVALID_ARG),
    ({"scale": 0.0}, fa.FA_ERR_INVALID_ARG),
    ({"scale": float("inf")}, fa.FA_ERR_INVALID_ARG),
])
def test_fwd_fp8_rejects_bad_arguments(kw, code):
    assert fwd8(**kw) == code


@pytest.mark.parametrize("fn", ["fa_fp8_quantize_qk", "fa_fp8_quantize_v"])
@pytest.mark.parametrize("kw,code", [
    ({"x": None}, fa.FA_ERR_INVALID_ARG),
    ({"x8": A + 4}, fa.FA_ERR_INVALID_ARG),
    ({"s": None}, fa.FA_ERR_INVALID_ARG),
    ({"s": A + 2}, fa.FA_ERR_INVALID_ARG),
    ({"d": 64}, fa.FA_ERR_UNSUPPORTED),
    ({"H": 0}, fa.FA_ERR_INVALID_ARG),
])
def test_fp8_encoders_reject_bad_arguments(fn, kw, code):
    args = dict(x=A, x8=A, s=A, B=1, H=2, N=300, d=128)
    args.update(kw)
    f = getattr(fa.load(), fn)
    assert f(args["x"], args["x8"], args["s"], args["B"], args["H"], args["N"], args["d"],
             None) == code


def fwd_drop(t, **kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=64, causal=0, bm=None,
                kv=None, scale=0.125, dtype=fa.FA_BF16)
    args.update(kw)
    return fa.load().fa_fwd_dropout(args["q"], args["k"], args["v"], args["o"], args["lse"],
                                    args["B"], args["H"], args["N"], args["d"], args["causal"],
                                    args["bm"], args["kv"], args["scale"], args["dtype"], t,
                                    12345, 0, None)


def bwd_drop(t, main=False, **kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, do=A, dq=A, dk=A, dv=A, B=1, H=1, N=128, d=64,
                causal=0, bm=None, kv=None, scale=0.125, dtype=fa.FA_BF16, ws=A,
                wsb=1 << 30)
    args.update(kw)
    lib = fa.load()
    if main:
        return lib.fa_bwd_main_dropout(args["q"], args["k"], args["v"], args["lse"], args["do"],
                                       args["dq"], args["dk"], args["dv"], args["B"], args["H"],
                                       args["N"], args["d"], args["causal"], args["bm"],
                                       args["kv"], args["scale"], args["dtype"], t, 7, 1,
                                       args["ws"], args["wsb"], None)
    return lib.fa_bwd_dropout(args["q"], args["k"], args["v"], args["o"], args["lse"],
                              args["do"], args["dq"], args["dk"], args["dv"], args["B"],
                              args["H"], args["N"], args["d"], args["causal"], args["bm"],
                              args["kv"], args["scale"], args["dtype"], t, 7, 1, args["ws"],
                              args["wsb"], None)


@pytest.mark.parametrize("t", [-1, 256, 1000])
def test_dropout_rejects_thresholds_outside_a_byte(t):
    assert fwd_drop(t) == fa.FA_ERR_INVALID_ARG
    assert bwd_drop(t) == fa.FA_ERR_INVALID_ARG
    assert bwd_drop(t, main=True) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    ({"q": None}, fa.FA_ERR_INVALID_ARG),
    ({"d": 96}, fa.FA_ERR_UNSUPPORTED),
    ({"scale": float("nan")}, fa.FA_ERR_INVALID_ARG),
    ({"lse": A + 1}, fa.FA_ERR_INVALID_ARG),
])
def test_dropout_entry_points_validate_like_the_plain_ones(kw, code):
    assert fwd_drop(100, **kw) == code
    assert bwd_drop(100, **kw) == code


def test_dropout_python_binding_checks_the_threshold():
    with pytest.raises(ValueError):
        fa._drop_args(256, 0, 0)
    assert fa._drop_args(255, -1, 2 ** 32 + 5) == (255, 2 ** 64 - 1, 5)


@pytest.mark.parametrize("args,code", [
    ((None, 1, 4, 4), fa.FA_ERR_INVALID_ARG),
    ((A, 0, 4, 4), fa.FA_ERR_INVALID_ARG),
    ((A, 1, 0, 4), fa.FA_ERR_INVALID_ARG),
    ((A, 70000, 4, 4), fa.FA_ERR_INVALID_ARG),
    ((A, 1, 65536, 65536), fa.FA_ERR_UNSUPPORTED),
])
def test_dropout_random_bytes_rejects_bad_sizes(args, code):
    assert fa.load().fa_dropout_random_bytes(*args, 1, 0, None) == code


# ------------------------------------------------------------------ sequence sharding

def merge(**kw):
    args = dict(parts=A, lses=A, S=4, o=A, lse=A, B=1, H=2, N=128, d=128, dtype=fa.FA_BF16)
    args.update(kw)
    return fa.load().fa_attn_merge(args["parts"], args["lses"], args["S"], args["o"],
                                   args["lse"], args["B"], args["H"], args["N"], args["d"],
                                   args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    ({"S": 0}, fa.FA_ERR_INVALID_ARG),
    ({"S": fa.FA_MERGE_MAX_PARTS + 1}, fa.FA_ERR_INVALID_ARG),
    ({"B": 0}, fa.FA_ERR_INVALID_ARG),
    ({"N": -1}, fa.FA_ERR_INVALID_ARG),
    ({"d": 96}, fa.FA_ERR_UNSUPPORTED),
    ({"dtype": 5}, fa.FA_ERR_INVALID_ARG),
    ({"parts": None}, fa.FA_ERR_INVALID_ARG),
    ({"lse": None}, fa.FA_ERR_INVALID_ARG),
    ({"o": A + 8}, fa.FA_ERR_INVALID_ARG),
    ({"lses": A + 2}, fa.FA_ERR_INVALID_ARG),
])
def test_merge_rejects_bad_arguments(kw, code):
    assert merge(**kw) == code


@pytest.mark.parametrize("fn", ["fa_grad_accumulate", "fa_grad_finish"])
@pytest.mark.parametrize("args,code", [
    ((None, A, 64, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((A, None, 64, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((A, A, 0, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((A, A, 66, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),     # not a multiple of 4
    ((A, A, 64, 9), fa.FA_ERR_INVALID_ARG),
])
def test_gradient_sums_reject_bad_arguments(fn, args, code):
    assert getattr(fa.load(), fn)(*args, None) == code


def test_gradient_sums_check_alignment():
    lib = fa.load()
    # fp32 sums are 16-byte aligned; bf16 contributions need 8 bytes, fp32 ones 16
    assert lib.fa_grad_accumulate(A + 8, A, 64, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_grad_accumulate(A, A + 8, 64, fa.FA_FP32, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_grad_finish(A + 4, A, 64, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_grad_finish(A, A + 8, 64, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG


def test_merge_binding_checks_shapes():
    import torch
    parts = torch.empty((2, 1, 1, 4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_attn_merge(parts, torch.empty((2, 1, 1, 5)), torch.empty((1, 1, 4, 64),
                                                                       dtype=torch.bfloat16),
                         torch.empty((1, 1, 4)))
    with pytest.raises(TypeError):
        fa.fa_attn_merge(parts, torch.empty((2, 1, 1, 4)), torch.empty((1, 1, 4, 64)),
                         torch.empty((1, 1, 4)))


def test_binding_refuses_host_tensors():
    # A host pointer reaching a kernel would fault the GPU: the binding refuses it first.
    import torch
    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        fa.fa_fwd(q, q, q, q.clone(), torch.zeros((1, 1, 8)))
    with pytest.raises(ValueError, match="CUDA tensors"):
        fa.fa_grad_accumulate(torch.zeros(8), torch.zeros(8, dtype=torch.bfloat16))
