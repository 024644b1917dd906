"""The sequence-sharded schedule (``seqshard.py``) across ranks, on the CPU.

Two and three gloo ranks each hold one chunk of the sequence and run the ring schedule of
the library (the key/value chunks and the dK, dV sums travel by torch.distributed
point-to-point operations).  The per-step computations are supplied by the CPU fp64 oracle
through the same interface the CUDA kernels implement, so this checks the schedule and the
exchanges: every rank's rows of O, lse, dQ, dK, dV must equal the oracle's attention over the
whole sequence.  The same schedule with every rank in one process is checked too.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class OracleShardOps:
    """The per-step computations of a rank on the CPU fp64 oracle (float64 torch tensors)."""

    def partial_buffers(self, q, parts):
        B, H, n, d = q.shape
        return (torch.zeros((parts, B, H, n, d), dtype=torch.float64),
                torch.zeros((parts, B, H, n), dtype=torch.float64))

    def partial_forward(self, q, k, v, o, lse, causal, scale):
        import oracle
        ro, rlse = oracle.forward(q.numpy(), k.numpy(), v.numpy(), scale, causal)
        o.copy_(torch.from_numpy(ro))
        lse.copy_(torch.from_numpy(rlse))

    def merge(self, o_parts, lse_parts, used):
        from oracle import seqshard
        S, B, H, n, d = o_parts.shape
        o, lse = seqshard.merge_partials(o_parts[:used].reshape(used, -1, d).numpy(),
                                         lse_parts[:used].reshape(used, -1).numpy())
        return torch.from_numpy(o).reshape(B, H, n, d), torch.from_numpy(lse).reshape(B, H, n)

    def zeros_f32(self, like):
        return torch.zeros(like.shape, dtype=torch.float64)

    def backward_begin(self, q, o, do):
        return {"D": (o * do).sum(-1), "dq": torch.zeros_like(q)}

    def partial_backward(self, state, q, k, v, lse, do, causal, scale):
        import oracle
        from oracle import seqshard
        B, H, n, d = q.shape
        dk, dv = torch.zeros_like(k), torch.zeros_like(v)
        keep = oracle.keep_mask(n, causal)
        for b in range(B):
            for h in range(H):
                gq, gk, gv = seqshard.backward_head_with_stats(
                    q[b, h].numpy(), k[b, h].numpy(), v[b, h].numpy(), do[b, h].numpy(),
                    lse[b, h].numpy(), state["D"][b, h].numpy(), scale, keep)
                state["dq"][b, h] += torch.from_numpy(gq)
                dk[b, h], dv[b, h] = torch.from_numpy(gk), torch.from_numpy(gv)
        return dk, dv

    def accumulate(self, acc, x):
        acc += x

    def finish(self, acc, dtype):
        return acc.clone()

    def backward_end(self, state, q, scale):
        return state["dq"]


def _inputs(W, B=1, H=2, n=6, d=4, seed=0):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((B, H, W * n, d), generator=g, dtype=torch.float64) for _ in range(4)]


def _reference(q, k, v, do, causal, scale):
    import oracle
    o, lse = oracle.forward(q.numpy(), k.numpy(), v.numpy(), scale, causal)
    dq, dk, dv, _ = oracle.backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(), scale, causal)
    return o, lse, dq, dk, dv


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, causal, out):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from exact_io_aware_28_gb300 import seqshard
    from test_seqshard_ranks import OracleShardOps, _inputs
    q, k, v, do = _inputs(world)
    n = q.shape[2] // world
    sl = slice(rank * n, (rank + 1) * n)
    qr, kr, vr, dor = (t[:, :, sl].contiguous() for t in (q, k, v, do))
    ops = OracleShardOps()
    o, lse = seqshard.sharded_forward(qr, kr, vr, causal, 0.5, ops=ops)
    dq, dk, dv = seqshard.sharded_backward(qr, kr, vr, o, lse, dor, causal, 0.5, ops=ops)
    out[rank] = tuple(t.numpy() for t in (o, lse, dq, dk, dv))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.skipif(not dist.is_available(), reason="torch.distributed unavailable")
@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_ranks_reproduce_the_whole_sequence(world, causal):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), causal, out), nprocs=world,
                       start_method="spawn", join=True)
    q, k, v, do = _inputs(world)
    ref = _reference(q, k, v, do, causal, 0.5)
    n = q.shape[2] // world
    for r in range(world):
        sl = slice(r * n, (r + 1) * n)
        for got, want in zip(out[r], ref):
            np.testing.assert_allclose(got, want[:, :, sl], atol=1e-12)


@pytest.mark.parametrize("world", [1, 2, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_one_process_schedule_matches_the_oracle(world, causal):
    from exact_io_aware_28_gb300 import seqshard
    q, k, v, do = _inputs(world, seed=3)
    n = q.shape[2] // world
    chunk = lambda t: [t[:, :, r * n:(r + 1) * n].contiguous() for r in range(world)]
    qs, ks, vs, dos = chunk(q), chunk(k), chunk(v), chunk(do)
    ops = OracleShardOps()
    fwd = seqshard.chunked_forward(qs, ks, vs, causal, 0.5, ops=ops)
    os_, lses = [f[0] for f in fwd], [f[1] for f in fwd]
    bwd = seqshard.chunked_backward(qs, ks, vs, os_, lses, dos, causal, 0.5, ops=ops)
    ref = _reference(q, k, v, do, causal, 0.5)
    for r in range(world):
        sl = slice(r * n, (r + 1) * n)
        got = (os_[r], lses[r]) + tuple(bwd[r])
        for g, want in zip(got, ref):
            np.testing.assert_allclose(g.numpy(), want[:, :, sl], atol=1e-12)


def test_skipped_chunks_under_the_causal_mask():
    # Under the causal mask, rank r computes partials only for chunks s <= r.
    from exact_io_aware_28_gb300 import seqshard
    calls = []

    class Counting(OracleShardOps):
        def partial_forward(self, q, k, v, o, lse, causal, scale):
            calls.append(causal)
            super().partial_forward(q, k, v, o, lse, causal, scale)

    W = 4
    q, k, v, _ = _inputs(W, seed=5)
    n = q.shape[2] // W
    chunk = lambda t: [t[:, :, r * n:(r + 1) * n].contiguous() for r in range(W)]
    seqshard.chunked_forward(chunk(q), chunk(k), chunk(v), True, 0.5, ops=Counting())
    assert len(calls) == W * (W + 1) // 2 and sum(calls) == W
