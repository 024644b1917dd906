"""GPU parity of the sequence-sharded path: the merge, accumulate and finish kernels, and
the whole ring schedule with every rank in one process (chunks of one sequence on one GPU),
against the CPU fp64 oracle over the whole sequence."""
import numpy as np
import pytest
import torch

import oracle
from oracle import seqshard as oss
from exact_io_aware_28_gb300 import fa
from exact_io_aware_28_gb300 import seqshard
from exact_io_aware_28_gb300 import workloads as W

from _parity import TOL, compare, np64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 5])
def test_merge_kernel_against_the_oracle(dtype, d, S):
    B, H, N = 2, 3, 77
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(S * d)
    o_parts = torch.randn((S, B, H, N, d), generator=g).to(tdt)
    lse_parts = 4 * torch.randn((S, B, H, N), generator=g)
    lse_parts[0, 0, 0, :5] = -float("inf")          # a part without visible keys
    lse_parts[:, 1, 2, 7] = -float("inf")           # a row that no part sees
    lse_parts[-1, 1, 1, 3] = 1e4                     # a dominant, large logsumexp
    o = torch.empty((B, H, N, d), dtype=tdt, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa.fa_attn_merge(o_parts.cuda(), lse_parts.cuda(), o, lse)
    torch.cuda.synchronize()
    ro, rlse = oss.merge_partials(np64(o_parts).reshape(S, -1, d), np64(lse_parts).reshape(S, -1))
    ro, rlse = ro.reshape(B, H, N, d), rlse.reshape(B, H, N)
    got_o, got_lse = np64(o), np64(lse)
    dead = np.isneginf(rlse)
    assert np.array_equal(np.isneginf(got_lse), dead) and dead[1, 2, 7]
    assert np.all(got_o[dead] == 0)
    tol = TOL[dtype]
    assert np.abs(got_o - ro).max() <= tol["o"]
    # the logsumexp is a plain fp32 computation: within a few ulps of its magnitude
    assert np.abs(got_lse[~dead] - rlse[~dead]).max() <= 1e-6 * max(1.0, np.abs(rlse[~dead]).max())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_accumulate_and_finish_kernels_are_exact(dtype):
    n = 4 * 12345
    g = torch.Generator().manual_seed(7)
    acc0 = torch.randn(n, generator=g)
    x = torch.randn(n, generator=g).to(dtype)
    acc = acc0.cuda()
    fa.fa_grad_accumulate(acc, x.cuda())
    out = torch.empty(n, dtype=dtype, device="cuda")
    fa.fa_grad_finish(out, acc)
    torch.cuda.synchronize()
    want = acc0 + x.float()                              # one fp32 addition per element
    assert torch.equal(acc.cpu(), want)
    assert torch.equal(out.cpu(), want.to(dtype))        # one round-to-nearest-even


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_chunked_schedule_against_the_oracle(dtype, world, causal, d):
    n = 200                                             # ragged against the 128-row tiles
    w = W.custom("chunks", 1, 2, world * n, d, dtype, causal=causal)
    x = W.make_inputs(w, seed=world + d, device="cuda")
    chunk = lambda t: [t[:, :, r * n:(r + 1) * n].contiguous() for r in range(world)]
    qs, ks, vs, dos = chunk(x.q), chunk(x.k), chunk(x.v), chunk(x.do)
    fwd = seqshard.chunked_forward(qs, ks, vs, causal, x.scale)
    os_, lses = [f[0] for f in fwd], [f[1] for f in fwd]
    bwd = seqshard.chunked_backward(qs, ks, vs, os_, lses, dos, causal, x.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    cat = lambda ts: torch.cat(list(ts), dim=2)
    got = (cat(os_), cat(lses), cat(b[0] for b in bwd), cat(b[1] for b in bwd),
           cat(b[2] for b in bwd))
    q, k, v, do = (np64(t) for t in (x.q, x.k, x.v, x.do))
    ro, rlse = oracle.forward(q, k, v, x.scale, causal)
    rdq, rdk, rdv, _ = oracle.backward(q, k, v, do, x.scale, causal)
    compare(got, (ro, rlse, rdq, rdk, rdv), dtype)


def test_chunked_schedule_at_the_long_context_shape():
    # The long-context shape (H = 32, N = 16384, d = 128, causal) split into four chunks of
    # 4096 rows; two sampled heads compared with the oracle.
    world, n = 4, 4096
    w = W.custom("chunks_long", 1, 32, world * n, 128, "bf16", causal=True)
    x = W.make_inputs(w, seed=0, device="cuda")
    chunk = lambda t: [t[:, :, r * n:(r + 1) * n].contiguous() for r in range(world)]
    qs, ks, vs, dos = chunk(x.q), chunk(x.k), chunk(x.v), chunk(x.do)
    fwd = seqshard.chunked_forward(qs, ks, vs, True, x.scale)
    os_, lses = [f[0] for f in fwd], [f[1] for f in fwd]
    bwd = seqshard.chunked_backward(qs, ks, vs, os_, lses, dos, True, x.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    heads = [(0, 5), (0, 30)]
    cat = lambda ts: torch.cat(list(ts), dim=2)
    got = (cat(os_), cat(lses), cat(b[0] for b in bwd), cat(b[1] for b in bwd),
           cat(b[2] for b in bwd))
    q, k, v, do = (np64(t) for t in (x.q, x.k, x.v, x.do))
    ro, rlse = oracle.forward(q, k, v, x.scale, True, heads=heads)
    rdq, rdk, rdv, _ = oracle.backward(q, k, v, do, x.scale, True, heads=heads)
    compare(got, (ro, rlse, rdq, rdk, rdv), "bf16", heads=heads)
