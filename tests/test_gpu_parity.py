"""GPU parity: the library (through the C ABI) against the CPU fp64 oracle.

Small shapes cover several tiles, ragged tails, every mask mode and the degenerate
cases (N = 1, rows that see no key, kv_len = 0); the five named workloads run at
their full sizes, the two largest on sampled (batch, head) pairs, which are
independent units of the computation.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_28_gb300 import fa
from exact_io_aware_28_gb300 import workloads as W

from _parity import compare, run_library, run_oracle

pytestmark = pytest.mark.gpu


def _mask_variants(N, seed=0):
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(seed + 100)
    bm = (torch.rand((nb, nb), generator=g) < 0.5).to(torch.uint8)
    bm.fill_diagonal_(1)
    return {
        "dense": {},
        "causal": {"causal": True},
        "padded": {"kv_len": True},
        "block": {"blockmask": bm},
        "block_causal": {"blockmask": bm, "causal": True},
    }


def _inputs(B, H, N, d, dtype, variant, seed=0):
    w = W.custom("edge", B, H, N, d, dtype, causal=variant.get("causal", False))
    x = W.make_inputs(w, seed=seed, device="cuda")
    if variant.get("kv_len"):
        g = torch.Generator().manual_seed(seed + 7)
        x.kv_len = torch.randint(1, N + 1, (B,), generator=g, dtype=torch.int32).cuda()
    if "blockmask" in variant:
        x.blockmask = variant["blockmask"].cuda()
    return x


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 128, 130, 257, 640])
@pytest.mark.parametrize("mode", ["dense", "causal", "padded", "block", "block_causal"])
def test_small_shapes(dtype, d, N, mode):
    variant = _mask_variants(N)[mode]
    x = _inputs(2, 2, N, d, dtype, variant, seed=N + d)
    compare(run_library(x), run_oracle(x), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_rows_without_visible_keys(dtype):
    N, d = 300, 64
    nb = 3
    bm = torch.ones((nb, nb), dtype=torch.uint8)
    bm[1, :] = 0  # query rows 128..255 see nothing
    x = _inputs(2, 2, N, d, dtype, {"blockmask": bm}, seed=3)
    x.kv_len = torch.tensor([0, 200], dtype=torch.int32, device="cuda")  # sequence 0: no keys
    out = run_library(x)
    compare(out, run_oracle(x), dtype)
    o, lse = out[0].float(), out[1]
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.all(o[1, :, 128:256] == 0)


def test_backward_dk_dv_deterministic():
    x = _inputs(1, 4, 700, 128, "bf16", {"causal": True}, seed=11)
    a = run_library(x)
    b = run_library(x)
    for i in (0, 1, 3, 4):  # o, lse, dk, dv: bitwise equal run to run
        assert torch.equal(a[i], b[i])
    assert torch.allclose(a[2].float(), b[2].float(), atol=0, rtol=1e-2)


@pytest.mark.parametrize("name", ["tiny_fp32", "gpt2_causal", "bert_padded"])
def test_named_workload_full(name):
    w = W.WORKLOADS[name]
    x = W.make_inputs(w, seed=0, device="cuda")
    errs = compare(run_library(x), run_oracle(x), w.dtype)
    print(name, errs)


@pytest.mark.slow
@pytest.mark.parametrize("name,heads", [
    ("block_sparse", [(0, 0), (1, 7)]),
    ("long_causal", [(0, 0), (0, 31)]),
])
def test_named_workload_sampled_heads(name, heads):
    w = W.WORKLOADS[name]
    x = W.make_inputs(w, seed=0, device="cuda")
    out = run_library(x)
    errs = compare(out, run_oracle(x, heads=heads), w.dtype, heads=heads)
    print(name, errs)
    # every head of the full launch is finite
    for t in out:
        assert torch.isfinite(t.float()).all() or t is out[1]


@pytest.mark.slow
def test_grouped_grid_order_with_a_ragged_last_group():
    # Both tensor-core kernels order their grids by groups of heads sized to L2 (at N = 16384,
    # d = 128: eight heads per forward group, four per backward group).  Nine heads leave a
    # last group of one head in both; that head and one from a full group against the oracle.
    x = _inputs(1, 9, 16384, 128, "bf16", {"causal": True}, seed=23)
    out = run_library(x)
    heads = [(0, 3), (0, 8)]
    errs = compare(out, run_oracle(x, heads=heads), "bf16", heads=heads)
    print(errs)
    for t in out:
        assert torch.isfinite(t.float()).all() or t is out[1]


@pytest.mark.slow
def test_long_sequence_sampled_rows_and_gradient_sums():
    # N = 2^16 + 77 (a ragged tail at a size far past the bench's), causal, d = 128: sampled
    # rows of O and lse against the oracle, one row at a time; the gradients through the
    # identities that hold at any size (rows of P sum to 1, rows of dS sum to 0):
    #   sum_j dK_j = 0   and   sum_j dV_j = sum_i dO_i.
    # On the GPU they are loose checks: P and dS are rounded to bf16 as MMA operands.
    N = (1 << 16) + 77
    x = _inputs(1, 2, N, 128, "bf16", {"causal": True}, seed=17)
    o, lse, dq, dk, dv = run_library(x)
    rows = np.array([0, 1, 127, 128, 4095, 32768, N - 78, N - 1])
    q, k, v = (t.detach().to("cpu", torch.float64).numpy() for t in (x.q, x.k, x.v))
    og, lg = o.double().cpu().numpy(), lse.double().cpu().numpy()
    for h in range(2):
        keep = np.arange(N)[None, :] <= rows[:, None]
        ro, rl, _ = oracle.forward_head(q[0, h, rows], k[0, h], v[0, h], x.scale, keep)
        assert np.abs(og[0, h, rows] - ro).max() <= 2e-2
        assert np.abs(lg[0, h, rows] - rl).max() <= 1e-3
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    dk64, dv64, do64 = (t.double() for t in (dk, dv, x.do))
    sk = dk64.sum(dim=2).abs()                       # [B, H, d]
    assert (sk <= 2e-2 * dk64.abs().sum(dim=2)).all()
    sv, sdo = dv64.sum(dim=2), do64.sum(dim=2)
    assert ((sv - sdo).abs() <= 2e-2 * do64.abs().sum(dim=2)).all()
