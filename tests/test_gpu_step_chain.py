"""Training steps issued back to back on one stream with no synchronisation between them.

The four kernels of a step (forward, preprocess, backward main, dQ convert) are launched with
programmatic dependent launch: each may start while the previous one drains and waits in the
kernel before it touches global memory.  Consecutive steps share one workspace, so the next
step's preprocess clears the dQ accumulator that the previous step's convert reads; if any
kernel ran ahead of its predecessor, a step's dQ (or O, lse, dK, dV) would come out wrong.
Every step here has its own inputs and outputs, and all of them are checked against the oracle.
"""
import pytest
import torch

from exact_io_aware_28_gb300 import fa
from exact_io_aware_28_gb300 import workloads as W

from _parity import compare, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,causal", [(64, True), (128, True), (128, False)])
def test_back_to_back_steps_share_a_workspace(d, causal):
    B, H, N, steps = 1, 3, 384, 4
    w = W.custom("chain", B, H, N, d, "bf16", causal=causal)
    xs = [W.make_inputs(w, seed=11 + s, device="cuda") for s in range(steps)]
    ws = fa.alloc_workspace(B, H, N, d, "cuda")
    outs = []
    torch.cuda.synchronize()
    for x in xs:
        o = torch.empty_like(x.q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        dq, dk, dv = (torch.empty_like(x.q) for _ in range(3))
        fa.fa_fwd(x.q, x.k, x.v, o, lse, x.causal, x.blockmask, x.kv_len, x.scale)
        fa.fa_bwd_preprocess(o, x.do, ws)
        fa.fa_bwd_main(x.q, x.k, x.v, lse, x.do, dq, dk, dv, ws, x.causal, x.blockmask,
                       x.kv_len, x.scale)
        fa.fa_bwd_dq_convert(dq, ws, x.scale)
        outs.append((o, lse, dq, dk, dv))
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    for x, out in zip(xs, outs):
        compare(out, run_oracle(x), "bf16")


def test_dropout_and_plain_steps_interleaved():
    # The dropout instances of the forward and backward kernels are chained the same way.
    B, H, N, d = 1, 2, 256, 128
    w = W.custom("chain", B, H, N, d, "bf16", causal=True)
    xs = [W.make_inputs(w, seed=31 + s, device="cuda") for s in range(3)]
    ws = fa.alloc_workspace(B, H, N, d, "cuda")
    plain = []
    torch.cuda.synchronize()
    for s, x in enumerate(xs):
        if s == 1:
            o, lse = fa.forward_dropout(x.q, x.k, x.v, 26, 99, 0, True)
            fa.backward_dropout(x.q, x.k, x.v, o, lse, x.do, 26, 99, 0, True, workspace=ws)
            continue
        o = torch.empty_like(x.q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        dq, dk, dv = (torch.empty_like(x.q) for _ in range(3))
        fa.fa_fwd(x.q, x.k, x.v, o, lse, True)
        fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, ws, True)
        plain.append((x, (o, lse, dq, dk, dv)))
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    for x, out in plain:
        compare(out, run_oracle(x), "bf16")


def test_foreign_kernels_before_and_after():
    # Inputs written by torch kernels launched just before the forward, outputs read by torch
    # kernels just after the backward, all on the current stream without synchronisation: the
    # library's kernels must wait for the writers and finish before the readers.
    B, H, N, d = 1, 2, 320, 128
    w = W.custom("chain", B, H, N, d, "bf16", causal=True)
    x = W.make_inputs(w, seed=51, device="cuda")
    ref = run_oracle(x)
    torch.cuda.synchronize()
    q2, k2, v2, do2 = (torch.zeros_like(t) for t in (x.q, x.k, x.v, x.do))
    for dst, src in zip((q2, k2, v2, do2), (x.q, x.k, x.v, x.do)):
        dst.add_(src)                      # a torch kernel writes each input
    o = torch.empty_like(q2)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(q2) for _ in range(3))
    ws = fa.alloc_workspace(B, H, N, d, "cuda")
    fa.fa_fwd(q2, k2, v2, o, lse, True)
    fa.fa_bwd(q2, k2, v2, o, lse, do2, dq, dk, dv, ws, True)
    copies = [t.clone() for t in (o, lse, dq, dk, dv)]   # torch kernels read each output
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    compare(tuple(copies), ref, "bf16")


def test_training_step_captured_in_a_cuda_graph():
    # The chained launches captured by stream capture and replayed: each replay on new inputs
    # copied into the captured buffers matches the oracle.
    B, H, N, d = 1, 2, 384, 128
    w = W.custom("chain", B, H, N, d, "bf16", causal=True)
    xs = [W.make_inputs(w, seed=61 + s, device="cuda") for s in range(3)]
    q, k, v, do = (t.clone() for t in (xs[0].q, xs[0].k, xs[0].v, xs[0].do))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = fa.alloc_workspace(B, H, N, d, "cuda")

    def step():
        fa.fa_fwd(q, k, v, o, lse, True)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                 # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for x in xs[1:]:
        for dst, src in zip((q, k, v, do), (x.q, x.k, x.v, x.do)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert fa.fa_device_error() == fa.FA_OK
        compare((o, lse, dq, dk, dv), run_oracle(x), "bf16")
