"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Callers such as code inside another framework's memory pool, plug-ins with device memory
planned up front, or hooks where a cudaMalloc is not allowed get the backward without
passing a workspace; the library uses its own fixed scratch array instead.  These tests
call that entry point through the C ABI, twice in a row (the array keeps the previous
call's contents), and compare it with fa_bwd given an ordinary workspace, within the
parity tolerances.  The file is named to be collected last.
"""
import ctypes

import pytest
import torch

from exact_io_aware_28_gb300 import fa
from exact_io_aware_28_gb300 import workloads as W

from _parity import TOL, compare, run_oracle

pytestmark = pytest.mark.gpu


def _case(B, H, N, d, dtype, seed, **kw):
    w = W.custom("noalloc", B, H, N, d, dtype, **kw)
    x = W.make_inputs(w, seed=seed, device="cuda")
    o, lse = fa.forward(x.q, x.k, x.v, x.causal, x.blockmask, x.kv_len, x.scale)
    ref = fa.backward(x.q, x.k, x.v, o, lse, x.do, x.causal, x.blockmask, x.kv_len, x.scale)
    return x, o, lse, ref


def _noalloc(x, o, lse):
    dq, dk, dv = torch.empty_like(x.q), torch.empty_like(x.k), torch.empty_like(x.v)
    fa.fa_bwd_noalloc(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, x.causal, x.blockmask,
                      x.kv_len, x.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    return dq, dk, dv


def _close(got, ref, dtype):
    tol = TOL[dtype]["grad"]
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g, r = g.double(), r.double()
        assert torch.isfinite(g).all(), name
        scale = max(float(r.abs().max()), 1e-30)
        assert float((g - r).abs().max()) / scale <= tol, name


def test_two_calls_in_a_row_match_fa_bwd():
    a = _case(2, 3, 640, 128, "bf16", seed=21, causal=True)
    b = _case(1, 4, 300, 64, "bf16", seed=22)
    for case in (a, b, a):  # a different problem in between: no stale scratch contents
        x, o, lse, ref = case
        first = _noalloc(x, o, lse)
        second = _noalloc(x, o, lse)
        _close(first, ref, "bf16")
        _close(second, ref, "bf16")


def test_fp32_and_masks_match_fa_bwd():
    x, o, lse, ref = _case(2, 2, 257, 64, "fp32", seed=23, padded=True)
    for _ in range(2):
        _close(_noalloc(x, o, lse), ref, "fp32")
    nb = 3
    bm = torch.ones((nb, nb), dtype=torch.uint8)
    bm[2, 0] = 0
    w = W.custom("noalloc_bm", 1, 2, 300, 128, "bf16")
    x = W.make_inputs(w, seed=24, device="cuda")
    x.blockmask = bm.cuda()
    o, lse = fa.forward(x.q, x.k, x.v, False, x.blockmask, None, x.scale)
    ref = fa.backward(x.q, x.k, x.v, o, lse, x.do, False, x.blockmask, None, x.scale)
    for _ in range(2):
        _close(_noalloc(x, o, lse), ref, "bf16")


def test_matches_the_oracle_directly():
    # The same check against the CPU fp64 oracle rather than against fa_bwd: causal, two
    # calls in a row, every gradient within the bf16 tolerances.
    w = W.custom("noalloc_oracle", 1, 2, 384, 128, "bf16", causal=True)
    x = W.make_inputs(w, seed=25, device="cuda")
    o, lse = fa.forward(x.q, x.k, x.v, x.causal, None, None, x.scale)
    ref = run_oracle(x)
    for _ in range(2):
        dq, dk, dv = _noalloc(x, o, lse)
        compare((o, lse, dq, dk, dv), ref, "bf16")


def test_rejects_problems_larger_than_the_scratch_array():
    # 1 x 32 x 16384 x 128 needs ~270 MB of workspace: refused before any launch.
    lib = fa.load()
    A = ctypes.c_void_p(0x10000)
    st = lib.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, 1, 32, 16384, 128, 1, None, None,
                            0.088, fa.FA_BF16, None)
    assert st == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_workspace_bytes(1, 32, 16384, 128) > fa.FA_NOALLOC_SCRATCH_BYTES
