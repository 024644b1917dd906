"""Attention over a sequence split into equal contiguous chunks, one chunk per rank.

The FlashAttention reading guide (arXiv 2205.14135) lists attention over several GPUs as
open work ("Limitations"); its "Method" already holds the tool: the softmax statistics of
a vector split into parts merge exactly (m = max(m1, m2), l = e^{m1 - m} l1 +
e^{m2 - m} l2).  Here rank r holds the query, key, value (and upstream-gradient) rows of
chunk r.  The key/value chunks travel around a ring of ranks:

* forward: at step t rank r holds the keys and values of chunk s = (r - t) mod W and
  computes the partial (O_s, lse_s) of its queries over them with ``fa_fwd`` (chunk s < r:
  every key visible; s = r: the causal diagonal chunk; s > r under the causal mask: no key
  visible, skipped).  After W steps ``fa_attn_merge`` combines the partials into this
  rank's rows of O and lse.
* backward: ``fa_bwd_preprocess`` of the merged (O, dO) gives D and clears the dQ
  accumulator; at each step ``fa_bwd_main`` with the merged lse adds chunk s's
  contribution to dQ and writes its contributions to dK_s, dV_s, which
  ``fa_grad_accumulate`` adds to fp32 sums that travel with the chunk; one last hop brings
  every chunk's sums home, where ``fa_grad_finish`` and ``fa_bwd_dq_convert`` round them.

Every arithmetic step runs in the library's kernels; this module schedules them and moves
tensors.  The move is a ring shift (send to rank r + 1, receive from rank r - 1) through
``torch.distributed`` point-to-point operations (NCCL between GPUs), posted before the
step's computation when the tensors are not changed by it (the key/value chunk) so that
the transfer overlaps the kernels.  The same per-rank schedule also runs with every rank
in one process (``chunked_forward`` / ``chunked_backward``), the ring shift then being a
rotation of Python lists; that form splits a long sequence into chunks on one GPU, each
emulated rank's kernels on a CUDA stream of its own (events order the hand-offs), so that
the launches of one rank fill the tails of another's.

Supported: bf16 or fp32 [B, H, n, d] chunks of equal length n, d in {64, 128}, dense or
causal attention (top-left aligned over the whole sequence).  Key padding and block masks
are not supported across chunks.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import fa


class CudaShardOps:
    """The per-step computations of a rank, on the library's CUDA kernels."""

    def partial_buffers(self, q, parts: int):
        B, H, n, d = q.shape
        return (torch.empty((parts, B, H, n, d), dtype=q.dtype, device=q.device),
                torch.empty((parts, B, H, n), dtype=torch.float32, device=q.device))

    def partial_forward(self, q, k, v, o, lse, causal: bool, scale: float):
        fa.fa_fwd(q, k, v, o, lse, causal, None, None, scale)

    def merge(self, o_parts, lse_parts, used: int):
        o = torch.empty(o_parts.shape[1:], dtype=o_parts.dtype, device=o_parts.device)
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
        fa.fa_attn_merge(o_parts[:used], lse_parts[:used], o, lse)
        return o, lse

    def zeros_f32(self, like):
        return torch.zeros(like.shape, dtype=torch.float32, device=like.device)

    def backward_begin(self, q, o, do):
        B, H, n, d = q.shape
        ws = fa.alloc_workspace(B, H, n, d, q.device)
        fa.fa_bwd_preprocess(o, do, ws)
        state = {"ws": ws}
        if q.dtype == torch.float32:        # the fp32 path writes dQ itself: sum it here
            state["dq_acc"] = self.zeros_f32(q)
        return state

    def partial_backward(self, state, q, k, v, lse, do, causal: bool, scale: float):
        dq = torch.empty_like(q)
        dk, dv = torch.empty_like(k), torch.empty_like(v)
        fa.fa_bwd_main(q, k, v, lse, do, dq, dk, dv, state["ws"], causal, None, None, scale)
        if "dq_acc" in state:
            self.accumulate(state["dq_acc"], dq)
        return dk, dv

    def accumulate(self, acc, x):
        fa.fa_grad_accumulate(acc, x)

    def finish(self, acc, dtype):
        out = torch.empty(acc.shape, dtype=dtype, device=acc.device)
        fa.fa_grad_finish(out, acc)
        return out

    def backward_end(self, state, q, scale: float):
        if "dq_acc" in state:
            return self.finish(state["dq_acc"], q.dtype)
        dq = torch.empty_like(q)
        fa.fa_bwd_dq_convert(dq, state["ws"], scale)
        return dq


def _visible(causal: bool, s: int, rank: int):
    """Key chunk s against query chunk ``rank``: None (no key visible) or the causal flag
    of the call (True only on the diagonal chunk)."""
    if not causal:
        return False
    if s < rank:
        return False
    if s == rank:
        return True
    return None


# A rank's schedule is a generator: it yields ("post", tag, tensors) to send tensors to the
# next rank, and ("wait", tag) to receive (as the value of the yield) what the previous
# rank posted under the same tag.  Every rank posts and waits on the same tags in the same
# order.

def _forward_schedule(ops, rank: int, world: int, q, k, v, causal: bool, scale: float):
    o_parts, lse_parts = ops.partial_buffers(q, world)
    used = 0
    kv = (k, v)
    for t in range(world):
        s = (rank - t) % world
        if t < world - 1:
            yield ("post", "kv", kv)
        c = _visible(causal, s, rank)
        if c is not None:
            ops.partial_forward(q, kv[0], kv[1], o_parts[used], lse_parts[used], c, scale)
            used += 1
        if t < world - 1:
            kv = yield ("wait", "kv")
    return ops.merge(o_parts, lse_parts, used)


def _backward_schedule(ops, rank: int, world: int, q, k, v, o, lse, do, causal: bool,
                       scale: float):
    state = ops.backward_begin(q, o, do)
    acc = (ops.zeros_f32(k), ops.zeros_f32(v))   # dK, dV sums of the chunk held
    kv = (k, v)
    for t in range(world):
        s = (rank - t) % world
        if t < world - 1:
            yield ("post", "kv", kv)
        c = _visible(causal, s, rank)
        if c is not None:
            dk_s, dv_s = ops.partial_backward(state, q, kv[0], kv[1], lse, do, c, scale)
            ops.accumulate(acc[0], dk_s)
            ops.accumulate(acc[1], dv_s)
        # The sums follow their chunk; after the last step this hop brings them home.
        yield ("post", "acc", acc)
        if t < world - 1:
            kv = yield ("wait", "kv")
        acc = yield ("wait", "acc")
    dq = ops.backward_end(state, q, scale)
    return dq, ops.finish(acc[0], k.dtype), ops.finish(acc[1], v.dtype)


def _run_distributed(gen, group):
    """Drive one rank's schedule with torch.distributed point-to-point operations."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    nxt = dist.get_global_rank(group, (rank + 1) % world) if group is not None else \
        (rank + 1) % world
    prv = dist.get_global_rank(group, (rank - 1) % world) if group is not None else \
        (rank - 1) % world
    pending = {}
    value = None
    while True:
        try:
            msg = gen.send(value)
        except StopIteration as stop:
            return stop.value
        value = None
        if msg[0] == "post":
            _, tag, tensors = msg
            recv = tuple(torch.empty_like(t) for t in tensors)
            ops = [dist.P2POp(dist.isend, t.contiguous(), nxt, group) for t in tensors]
            ops += [dist.P2POp(dist.irecv, r, prv, group) for r in recv]
            pending[tag] = (dist.batch_isend_irecv(ops), recv, tensors)
        else:
            reqs, recv, _sent = pending.pop(msg[1])
            for r in reqs:
                r.wait()
            value = recv


def _run_emulated(gens: List, streams=None):
    """Drive every rank's schedule in one process; a ring shift is a list rotation.

    With ``streams`` (one CUDA stream per rank) each rank's kernels go to its own stream, so
    that one rank's launches fill the tails of another's: a posted tensor carries an event
    recorded on the poster's stream, which the receiving rank's stream waits for, and it is
    marked as used on the receiving stream for the caching allocator.  The caller's stream
    waits for every rank's stream before the results are returned."""
    world = len(gens)
    results = [None] * world
    values = [None] * world
    posted = [dict() for _ in range(world)]
    live = list(range(world))
    caller = torch.cuda.current_stream() if streams is not None else None
    if streams is not None:
        for st in streams:
            st.wait_stream(caller)          # the inputs were written on the caller's stream

    def on(r):
        return torch.cuda.stream(streams[r]) if streams is not None else _nullctx()

    while live:
        waiting = {}
        for r in live:
            with on(r):
                while True:
                    try:
                        msg = gens[r].send(values[r])
                    except StopIteration as stop:
                        results[r] = stop.value
                        break
                    values[r] = None
                    if msg[0] == "post":
                        ev = None
                        if streams is not None:
                            ev = torch.cuda.Event()
                            ev.record(streams[r])
                        posted[r][msg[1]] = (msg[2], ev)
                    else:
                        waiting[r] = msg[1]
                        break
        done = [r for r in live if results[r] is not None]
        live = [r for r in live if results[r] is None]
        if live and done:
            raise RuntimeError("ranks finished out of step")
        for r in live:
            tensors, ev = posted[(r - 1) % world][waiting[r]]
            if streams is not None:
                streams[r].wait_event(ev)
                for t in tensors:
                    t.record_stream(streams[r])
            values[r] = tensors
        for r in live:
            posted[(r - 1) % world].pop(waiting[r], None)
    if streams is not None:
        for r, st in enumerate(streams):
            caller.wait_stream(st)
            for t in _tensors_of(results[r]):
                t.record_stream(caller)
    return results


class _nullctx:
    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


def _tensors_of(x):
    if isinstance(x, torch.Tensor):
        return [x]
    if isinstance(x, (tuple, list)):
        return [t for y in x for t in _tensors_of(y)]
    return []


def _rank_streams(t: torch.Tensor, world: int):
    """One stream per emulated rank for CUDA tensors, none on the CPU."""
    if t.device.type != "cuda":
        return None
    return [torch.cuda.Stream(device=t.device) for _ in range(world)]


def _check(chunks: Sequence[torch.Tensor]):
    n = chunks[0].shape[2]
    for t in chunks:
        if t.dim() != 4 or t.shape[2] != n or not t.is_contiguous():
            raise ValueError("chunks must be contiguous [B, H, n, d] tensors of one length n")


def sharded_forward(q, k, v, causal: bool = False, scale: Optional[float] = None, group=None,
                    ops=None):
    """This rank's rows of (O, lse) for the whole sequence; q, k, v are this rank's chunk
    (chunk ``rank`` of ``world`` equal chunks, in order)."""
    import torch.distributed as dist
    _check([q, k, v])
    scale = 1.0 / q.shape[-1] ** 0.5 if scale is None else float(scale)
    ops = ops or CudaShardOps()
    gen = _forward_schedule(ops, dist.get_rank(group), dist.get_world_size(group), q, k, v,
                            causal, scale)
    return _run_distributed(gen, group)


def sharded_backward(q, k, v, o, lse, do, causal: bool = False, scale: Optional[float] = None,
                     group=None, ops=None):
    """This rank's dQ, dK, dV; o, lse are this rank's rows of the merged forward."""
    import torch.distributed as dist
    _check([q, k, v, o, do])
    scale = 1.0 / q.shape[-1] ** 0.5 if scale is None else float(scale)
    ops = ops or CudaShardOps()
    gen = _backward_schedule(ops, dist.get_rank(group), dist.get_world_size(group), q, k, v, o,
                             lse, do, causal, scale)
    return _run_distributed(gen, group)


def chunked_forward(qs, ks, vs, causal: bool = False, scale: Optional[float] = None, ops=None):
    """Every chunk's (O, lse) in one process: the ring schedule with W = len(qs) ranks."""
    _check(list(qs) + list(ks) + list(vs))
    scale = 1.0 / qs[0].shape[-1] ** 0.5 if scale is None else float(scale)
    ops = ops or CudaShardOps()
    W = len(qs)
    return _run_emulated([_forward_schedule(ops, r, W, qs[r], ks[r], vs[r], causal, scale)
                          for r in range(W)], _rank_streams(qs[0], W))


def chunked_backward(qs, ks, vs, os_, lses, dos, causal: bool = False,
                     scale: Optional[float] = None, ops=None):
    """Every chunk's (dQ, dK, dV) in one process."""
    _check(list(qs) + list(ks) + list(vs) + list(os_) + list(dos))
    scale = 1.0 / qs[0].shape[-1] ** 0.5 if scale is None else float(scale)
    ops = ops or CudaShardOps()
    W = len(qs)
    return _run_emulated([_backward_schedule(ops, r, W, qs[r], ks[r], vs[r], os_[r], lses[r],
                                             dos[r], causal, scale) for r in range(W)],
                         _rank_streams(qs[0], W))
