#!/usr/bin/env python
"""Benchmark: exact attention forward + backward on GB300 through the C ABI.

One step = fa_fwd + the three backward stages (preprocess, main, dQ convert) over one
batch of seeded synthetic input already resident in HBM (with dropout: fa_fwd_dropout and
fa_bwd_main_dropout in place of fa_fwd and fa_bwd_main).  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long_causal]
    python bench.py --impl reference ...   # the CPU fp64 oracle on a bounded sample

Under torchrun (N > 1) every rank runs the same workload on its own GPU (replicas: the
(batch, head) units are independent, so there is no collective on the data path); the
timed region is bracketed by barriers and the slowest rank's time is reported.  ``--gpus``
must equal the number of ranks torchrun started (WORLD_SIZE); the script refuses otherwise.

The default run (long_causal) also times the other configurations and the dropout, FP8 and
decode workloads, each with the same CUDA events and clock sampler, and reports them in the
line's ``per_config`` block (``--no-per-config`` skips it).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from exact_io_aware_28_gb300 import accounting as acc  # noqa: E402
from exact_io_aware_28_gb300 import workloads as W  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s on 1 GB300 and % of dense bf16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
# Kernels launched per step by the library (fwd, preprocess, main, dQ convert).
KERNELS_PER_STEP = {"bf16": 4, "fp32": 4}
# Training-step workloads: the five plain ones and the one with attention dropout.
TRAIN_WORKLOADS = {**W.WORKLOADS, **W.DROPOUT_WORKLOADS}


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ------------------------------------------------------------------ clock sampling

class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().splitlines() if r.strip()]
        os.unlink(self.file.name)
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if self.uuid:
            mine = [r for r in rows if self.uuid in r[0]]
            rows = mine or rows
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        under_load = [s for s in sm if mx and s > 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(under_load) if under_load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def check_world(gpus: int) -> None:
    """``--gpus N`` must match the ranks torchrun started: one process per GPU.  A mismatch
    (for example ``--gpus 8`` without torchrun, which would time one GPU) is refused."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if gpus != world:
        raise SystemExit(f"bench.py: --gpus {gpus} but WORLD_SIZE={world}; launch one process "
                         f"per GPU with `python -m torch.distributed.run --nproc-per-node {gpus} "
                         f"bench.py --gpus {gpus} ...`")


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle timing

def oracle_head_seconds(x, head, w=None) -> float:
    """Run the oracle's forward and backward on one (b, h) head; return wall seconds.
    With a dropout workload the mask generation is part of the timed work."""
    import oracle
    b, h = head
    q, k, v, do = (t[b, h].to(torch.float64).numpy() for t in (x.q, x.k, x.v, x.do))
    bm = None if x.blockmask is None else x.blockmask.numpy()
    kl = None if x.kv_len is None else int(x.kv_len[b])
    keep = oracle.keep_mask(q.shape[0], x.causal, bm, kl)
    t0 = time.perf_counter()
    if w is not None and w.drop_threshold:
        dr = oracle.dropout
        z = dr.keep_drop_mask(w.drop_seed, 0, b * x.q.shape[1] + h, q.shape[0], w.drop_threshold)
        dr.forward_head(q, k, v, x.scale, keep, z, w.drop_threshold)
        dr.backward_head(q, k, v, do, x.scale, keep, z, w.drop_threshold)
    else:
        oracle.forward_head(q, k, v, x.scale, keep)
        oracle.backward_head(q, k, v, do, x.scale, keep)
    return time.perf_counter() - t0


def head_flops(w: W.Workload, x) -> float:
    bm = None if x.blockmask is None else x.blockmask.numpy()
    return acc.flops(1, 1, w.N, w.d, w.causal, bm)["fwd_bwd"]


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def sample_heads(time_head, H: int, min_s: float = 10.0, max_heads: int = 4):
    """Time heads (0, 0), (0, 1), ... with ``time_head`` until about ``min_s`` seconds of CPU
    work have run (at most ``max_heads`` heads); returns (heads timed, total seconds)."""
    n, total = 0, 0.0
    while n < min(H, max_heads) and (n == 0 or total < min_s):
        total += time_head((0, n))
        n += 1
    return n, total


def cpu_baseline(w: W.Workload, x_cpu) -> dict:
    n, secs = sample_heads(lambda hd: oracle_head_seconds(x_cpu, hd, w), w.H)
    return {"value": n * head_flops(w, x_cpu) / secs / 1e12, "unit": UNIT, "cores": cpu_cores(),
            "kind": "oracle",
            "sample": f"{n} (batch, head) pair(s) of {w.describe()}: fp64 NumPy forward + "
                      f"backward, {secs:.1f} s; FLOPs by the same convention as the GPU figure"}


def run_reference(args, world, rank):
    """The CPU fp64 oracle as it stands: one (batch, head) of the workload per step."""
    if rank != 0:
        return
    w = TRAIN_WORKLOADS[args.workload]
    x = W.make_inputs(w, seed=0)
    small = W.make_inputs(W.custom("warm", 1, 1, 256, w.d, w.dtype, causal=w.causal), seed=1)
    for _ in range(args.warmup):
        oracle_head_seconds(small, (0, 0), w)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    # A long-sequence head takes seconds in fp64: time at most 20 of the requested steps so
    # that the whole run stays within a few minutes, and say so in the line.
    timed = max(1, min(args.steps, 20))
    times = [oracle_head_seconds(x, heads[i % len(heads)], w) for i in range(timed)]
    mean = sum(times) / len(times)
    value = head_flops(w, x) / mean / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.describe(),
                   "sample": f"one (batch, head) per step; {timed} of {args.steps} steps timed"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"one (batch, head) of {w.describe()} per step, "
                                   f"{timed} steps timed"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per full-size launch of ``kernel`` recorded from an ncu capture, or None."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        with open(path) as f:
            return json.load(f).get(workload, {}).get(kernel)
    except (OSError, ValueError):
        return None


def summarize(ms):
    """Median, p95 and the 95% Student-t interval of the mean of per-step event times (ms)."""
    ms = np.asarray(ms, dtype=np.float64)
    n = len(ms)
    out = {"median": float(np.median(ms)), "p95": float(np.percentile(ms, 95)),
           "mean": float(ms.mean()), "n": n}
    if n > 1:
        try:
            from scipy.stats import t as student_t
            q = float(student_t.ppf(0.975, n - 1))
        except Exception:  # scipy missing: normal quantile, slightly narrow for small n
            q = 1.96
        half = q * float(ms.std(ddof=1)) / np.sqrt(n)
        out["ci95"] = [float(out["mean"] - half), float(out["mean"] + half)]
    return out


def pipelined_e2e(steps, host_in, dev_in, dev_out, host_out, compute, comp_stream, rates=None):
    """End-to-end time per step with the copies inside the timed region.

    Every step copies its inputs from pinned host memory (``host_in``) to the device and its
    results back to pinned host memory (``host_out``).  Two device buffer sets
    (``dev_in[0|1]``, ``dev_out[0|1]``) let step i+1's inputs travel on one copy stream and
    step i-1's results on another while step i computes, as a pipelined caller would run it.
    ``compute(inputs, outputs)`` launches one step on ``comp_stream``.  Returns ms per step;
    if ``rates`` is a dict, it also gets the median time of one step's input copies
    (``h2d_ms``) and of its result copies (``d2h_ms``), each timed on its copy stream.
    """
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    timed = rates is not None
    in_ready = [torch.cuda.Event(enable_timing=timed) for _ in range(steps)]
    done = [torch.cuda.Event() for _ in range(steps)]
    copied = [torch.cuda.Event(enable_timing=timed) for _ in range(steps)]
    h_beg = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if timed else None
    d_beg = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if timed else None
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(h2d_s)
    for i in range(steps):
        k = i & 1
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(done[i - 2])  # buffer set k is free again
            if timed:
                h_beg[i].record(h2d_s)
            for hsrc, ddst in zip(host_in, dev_in[k]):
                ddst.copy_(hsrc, non_blocking=True)
            in_ready[i].record(h2d_s)
        comp_stream.wait_event(in_ready[i])
        if i >= 2:
            comp_stream.wait_event(copied[i - 2])  # its results have left output set k
        compute(dev_in[k], dev_out[k])
        done[i].record(comp_stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(done[i])
            if timed:
                d_beg[i].record(d2h_s)
            for hdst, dsrc in zip(host_out, dev_out[k]):
                hdst.copy_(dsrc, non_blocking=True)
            copied[i].record(d2h_s)
    d2h_s.wait_event(copied[steps - 1])
    t1.record(d2h_s)
    torch.cuda.synchronize()
    if timed:
        rates["h2d_ms"] = float(np.median([h_beg[i].elapsed_time(in_ready[i])
                                           for i in range(steps)]))
        rates["d2h_ms"] = float(np.median([d_beg[i].elapsed_time(copied[i])
                                           for i in range(steps)]))
    return t0.elapsed_time(t1) / steps


def device_uuid(dev):
    try:
        return str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


def measure_train(fa, w, x, steps, warmup, world, dev, tag=""):
    """Time ``steps`` training steps (forward + the three backward stages) of workload ``w``
    on inputs ``x`` already resident on ``dev``: CUDA events around every kernel on the
    launching stream, nvidia-smi clocks sampled during the timed region.  Inputs smaller
    than twice the L2 are flushed from it (a 256 MiB write) before every step."""
    B, H, N, d = w.B, w.H, w.N, w.d
    o = torch.empty_like(x.q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(x.q), torch.empty_like(x.q), torch.empty_like(x.q)
    ws = fa.alloc_workspace(B, H, N, d, dev)
    bm_np = None if x.blockmask is None else x.blockmask.cpu().numpy()
    fl = acc.flops(B, H, N, d, w.causal, bm_np)
    elem = 2 if w.dtype == "bf16" else 4
    in_bytes = 4 * B * H * N * d * elem
    flush = in_bytes < 2 * L2_BYTES
    scratch = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush else None
    stream = torch.cuda.current_stream()
    drop = (w.drop_threshold, w.drop_seed, 0)

    def fwd_call(q_, k_, v_, o_, lse_):
        if w.drop_threshold:
            fa.fa_fwd_dropout(q_, k_, v_, o_, lse_, *drop, x.causal, x.blockmask, x.kv_len,
                              x.scale, stream)
        else:
            fa.fa_fwd(q_, k_, v_, o_, lse_, x.causal, x.blockmask, x.kv_len, x.scale, stream)

    def main_call(q_, k_, v_, lse_, do_, dq_, dk_, dv_):
        if w.drop_threshold:
            fa.fa_bwd_main_dropout(q_, k_, v_, lse_, do_, dq_, dk_, dv_, ws, *drop, x.causal,
                                   x.blockmask, x.kv_len, x.scale, stream)
        else:
            fa.fa_bwd_main(q_, k_, v_, lse_, do_, dq_, dk_, dv_, ws, x.causal, x.blockmask,
                           x.kv_len, x.scale, stream)

    def compute(inp, out):
        q_, k_, v_, do_ = inp
        o_, lse_, dq_, dk_, dv_ = out
        fwd_call(q_, k_, v_, o_, lse_)
        fa.fa_bwd_preprocess(o_, do_, ws, stream)
        main_call(q_, k_, v_, lse_, do_, dq_, dk_, dv_)
        fa.fa_bwd_dq_convert(dq_, ws, x.scale, stream)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        fwd_call(x.q, x.k, x.v, o, lse)
        if ev:
            ev[1].record(stream)
        fa.fa_bwd_preprocess(o, x.do, ws, stream)
        if ev:
            ev[2].record(stream)
        main_call(x.q, x.k, x.v, lse, x.do, dq, dk, dv)
        if ev:
            ev[3].record(stream)
        fa.fa_bwd_dq_convert(dq, ws, x.scale, stream)
        if ev:
            ev[4].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_error() != fa.FA_OK:
        raise RuntimeError(f"device error word set during warm-up {tag}")

    sampler = ClockSampler(device_uuid(dev))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    # Pass 1: an event between every two kernels, for the per-kernel times.
    for i in range(steps):
        if flush:
            scratch.fill_(i & 0xFF)
        step(evs[i])
    # Pass 2: the step as it runs, events only at its ends (the four kernels back to back, each
    # launched to overlap its set-up with the previous one's tail).
    ends = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        if flush:
            scratch.fill_(i & 0xFF)
        ends[i][0].record(stream)
        step()
        ends[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    if fa.fa_device_error() != fa.FA_OK:
        raise RuntimeError(f"device error word set during the timed region {tag}")

    phase = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(4)]
                      for i in range(steps)])  # ms: fwd, preprocess, main, convert
    step_ms = np.array([ends[i][0].elapsed_time(ends[i][1]) for i in range(steps)])
    timing = {name: summarize(col) for name, col in
              (("step_ms", step_ms), ("phase_sum_ms", phase.sum(axis=1)),
               ("fwd_ms", phase[:, 0]), ("preprocess_ms", phase[:, 1]),
               ("bwd_main_ms", phase[:, 2]), ("dq_convert_ms", phase[:, 3]))}
    # Inputs larger than L2: the whole loop of pass 2 (no flush in it); else the mean of the
    # per-step times, which leave the flush out.
    ms_per_step = float(step_ms.mean()) if flush else t_start.elapsed_time(t_end) / steps
    ms_per_step = max_over_ranks(ms_per_step, world)
    mean_phase = phase.mean(axis=0)
    bwd_ms = mean_phase[1:].sum()
    pk = peaks()
    value = world * fl["fwd_bwd"] / (ms_per_step * 1e-3) / 1e12
    return {
        "value": value, "ms_per_step": ms_per_step, "flops": fl, "flush": flush,
        "in_bytes": in_bytes, "timing": timing, "clocks": clocks, "mean_phase": mean_phase,
        "fwd_tflops": fl["fwd"] / (mean_phase[0] * 1e-3) / 1e12,
        "bwd_tflops": fl["bwd"] / (bwd_ms * 1e-3) / 1e12,
        "bwd_main_tflops": fl["bwd"] / (mean_phase[2] * 1e-3) / 1e12,
        "preprocess_gbs": acc.preprocess_bytes(B, H, N, d, elem) / (mean_phase[1] * 1e-3) / 1e9,
        "dq_convert_gbs": (acc.dq_convert_bytes(B, H, N, d, elem) / (mean_phase[3] * 1e-3) / 1e9
                           if w.dtype == "bf16" else None),
        "pct_of_peak_burst": value / world / pk["bf16_tflops"],
        "launches": 2 * KERNELS_PER_STEP[w.dtype] * steps,   # both timed passes
        "compute": compute, "buffers": (o, lse, dq, dk, dv), "stream": stream,
    }


def device_inputs(w, dev, x_cpu=None):
    """The workload's seeded inputs (drawn on the CPU) moved to ``dev``."""
    x_cpu = x_cpu if x_cpu is not None else W.make_inputs(w, seed=0)
    q, k, v, do = (t.to(dev) for t in (x_cpu.q, x_cpu.k, x_cpu.v, x_cpu.do))
    return W.Inputs(q, k, v, do,
                    None if x_cpu.kv_len is None else x_cpu.kv_len.to(dev),
                    None if x_cpu.blockmask is None else x_cpu.blockmask.to(dev),
                    x_cpu.causal, x_cpu.scale)


# The other configurations timed in the default run's ``per_config`` block (the headline
# workload itself is the line's value), and the sequence-sharded schedule on one GPU.
PER_CONFIG = ["tiny_fp32", "gpt2_causal", "bert_padded", "block_sparse", "long_causal_dropout",
              "long_causal_fp8", "decode_llama8b", "long_causal_chunks4"]
CHUNKED = {"long_causal_chunks4": ("long_causal", 4)}


def measure_chunked(fa, base: str, chunks: int, steps, warmup, world, dev):
    """The sequence-sharded schedule with every rank in one process on one GPU: workload
    ``base`` split into ``chunks`` equal contiguous chunks, the ring's forward (partial
    forwards + merge) and backward per step, timed with CUDA events; and the merge kernel
    alone on partials of the same size (HBM-bound)."""
    from exact_io_aware_28_gb300 import seqshard
    w = TRAIN_WORKLOADS[base]
    x = device_inputs(w, dev)
    n = w.N // chunks
    cut = lambda t: [t[:, :, r * n:(r + 1) * n].contiguous() for r in range(chunks)]
    qs, ks, vs, dos = cut(x.q), cut(x.k), cut(x.v), cut(x.do)
    del x
    stream = torch.cuda.current_stream()

    def step():
        fwd = seqshard.chunked_forward(qs, ks, vs, w.causal, w.scale)
        seqshard.chunked_backward(qs, ks, vs, [f[0] for f in fwd], [f[1] for f in fwd], dos,
                                  w.causal, w.scale)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_error() != fa.FA_OK:
        raise RuntimeError("device error word set during warm-up (chunked)")
    sampler = ClockSampler(device_uuid(dev))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for e0, e1 in evs:
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = np.array([e0.elapsed_time(e1) for e0, e1 in evs])
    fl = acc.flops(w.B, w.H, w.N, w.d, w.causal)["fwd_bwd"]
    # the merge of `chunks` partials of one chunk's rows (what each rank merges)
    parts = torch.randn((chunks, w.B, w.H, n, w.d), device=dev).to(torch.bfloat16)
    lses = torch.randn((chunks, w.B, w.H, n), device=dev)
    o = torch.empty((w.B, w.H, n, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, n), dtype=torch.float32, device=dev)
    for _ in range(3):
        fa.fa_attn_merge(parts, lses, o, lse)
    mevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(steps)]
    for e0, e1 in mevs:
        e0.record(stream)
        fa.fa_attn_merge(parts, lses, o, lse)
        e1.record(stream)
    torch.cuda.synchronize()
    mms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in mevs]))
    rows = w.B * w.H * n
    merge_bytes = chunks * rows * (w.d * 2 + 4) + rows * (w.d * 2 + 4)
    pk = peaks()
    return {"describe": f"{w.describe()} in {chunks} chunks of {n} rows, ring schedule in one "
                        f"process", "value": fl / (ms.mean() * 1e-3) / 1e12,
            "ms_per_step": float(ms.mean()), "timing": {"step_ms": summarize(ms)},
            "clocks": clocks, "merge_gbs": merge_bytes / (mms * 1e-3) / 1e9,
            "merge_frac_of_hbm": merge_bytes / (mms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "merge_ms": mms, "merge_bytes": merge_bytes,
            # per rank r: v visible chunks (r + 1 under the causal mask, else all), v partial
            # forwards + 1 merge; backward: preprocess, v mains with 2 accumulates each,
            # 2 finishes, dQ convert
            "launches": steps * sum(4 * v + 5 for v in
                                    ((r + 1) if w.causal else chunks for r in range(chunks)))}


def per_config(fa, args, world, dev, headline):
    """Time every other configuration and workload with the same events and clock sampler
    (at most 20 timed steps each after at least 3 warm-up steps)."""
    steps, warmup = max(2, min(args.steps, 20)), max(3, args.warmup)
    out = {}
    pk = peaks()
    for name in PER_CONFIG:
        if name == headline:
            continue
        t0 = time.perf_counter()
        if name in TRAIN_WORKLOADS:
            w = TRAIN_WORKLOADS[name]
            r = measure_train(fa, w, device_inputs(w, dev), steps, warmup, world, dev, name)
            entry = {"workload": w.describe(), "metric": "fwd+bwd TFLOP/s", "value": r["value"],
                     "fwd_tflops": r["fwd_tflops"], "bwd_tflops": r["bwd_tflops"],
                     "bwd_main_tflops": r["bwd_main_tflops"], "ms_per_step": r["ms_per_step"],
                     "pct_of_peak_burst": r["pct_of_peak_burst"],
                     "timing": {"step_ms": r["timing"]["step_ms"]}, "clocks": r["clocks"],
                     "launches": r["launches"], "steps": steps,
                     "l2": "flushed between steps (256 MiB write)" if r["flush"] else
                           "inputs larger than L2"}
            if w.dtype == "fp32":
                entry["note"] = "fp32 CUDA-core path: no tensor-core peak applies"
                entry.pop("pct_of_peak_burst")
        elif name in CHUNKED:
            base, nch = CHUNKED[name]
            r = measure_chunked(fa, base, nch, steps, warmup, world, dev)
            entry = {"workload": r["describe"], "metric": "fwd+bwd TFLOP/s", "value": r["value"],
                     "pct_of_peak_burst": r["value"] / world / pk["bf16_tflops"],
                     "ms_per_step": r["ms_per_step"], "merge_gbs": r["merge_gbs"],
                     "merge_frac_of_hbm": r["merge_frac_of_hbm"], "merge_ms": r["merge_ms"],
                     "timing": r["timing"], "clocks": r["clocks"], "launches": r["launches"],
                     "steps": steps, "l2": "inputs larger than L2"}
        elif name in W.FP8_WORKLOADS:
            r = measure_fp8(fa, W.FP8_WORKLOADS[name], steps, warmup, world, dev)
            entry = {"workload": r["describe"], "metric": "fwd TFLOP/s (encode + e4m3 forward)",
                     "value": r["value"], "fwd_kernel_tflops": r["fwd_tflops"],
                     "ms_per_step": r["ms_per_step"],
                     "frac_of_fp8_burst": r["fwd_tflops"] / (2.0 * pk["bf16_tflops"]),
                     "timing": {"step_ms": r["timing"]["step_ms"]}, "clocks": r["clocks"],
                     "launches": r["launches"], "steps": steps}
        else:
            r = measure_decode(fa, W.DECODE_WORKLOADS[name], steps, warmup, world, dev)
            entry = {"workload": r["describe"], "metric": "KV-cache GB/s", "value": r["gbs"],
                     "frac_of_hbm": r["gbs"] / world / pk["hbm_gbs"],
                     "ms_per_step": r["ms_per_step"],
                     "timing": {"step_ms": r["timing"]["step_ms"]}, "clocks": r["clocks"],
                     "launches": r["launches"], "steps": steps}
        entry["wall_s"] = time.perf_counter() - t0
        out[name] = entry
        torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    from exact_io_aware_28_gb300 import fa

    dev = torch.device("cuda", torch.cuda.current_device())
    w = TRAIN_WORKLOADS[args.workload]
    if args.heads:
        w = dataclasses.replace(w, H=args.heads)
    x_cpu = W.make_inputs(w, seed=0)
    x = device_inputs(w, dev, x_cpu)
    B, H, N, d = w.B, w.H, w.N, w.d
    r = measure_train(fa, w, x, args.steps, args.warmup, world, dev)
    fl, mean_phase, value, ms_per_step = r["flops"], r["mean_phase"], r["value"], r["ms_per_step"]
    pk = peaks()
    main_tf = r["bwd_main_tflops"]
    # The dominant kernel is timed by CUDA events over a sub-second region, as a kernel run
    # in a burst: its roofline is the measured burst bf16 peak (the sustained figure, from a
    # seconds-long loop under the power cap, is kept beside it).
    peak_t = pk["bf16_tflops"]
    traffic = None if args.heads else recorded_traffic(args.workload, "bwd_main")
    roofline = {"kernel": "bwd main (dK, dV, dQ partials)", "bound": "tensor",
                "achieved": main_tf, "peak": peak_t, "unit": "TFLOP/s",
                "frac": main_tf / peak_t, "traffic": traffic,
                "peak_kind": f"{pk['source']} bf16 dense, burst",
                "peak_sustained": pk["bf16_tflops_sustained"],
                "frac_of_sustained": main_tf / pk["bf16_tflops_sustained"]}

    # e2e: the same step through the public API with every step's inputs copied from pinned
    # host memory and its results copied back, inside the timed region (pipelined).
    o, lse, dq, dk, dv = r["buffers"]
    pin = [t.pin_memory() for t in (x_cpu.q, x_cpu.k, x_cpu.v, x_cpu.do)]
    outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, dq, dk, dv)]
    e2e_steps = max(2, min(args.steps, 20))
    dev_in = [(x.q, x.k, x.v, x.do), tuple(torch.empty_like(t) for t in (x.q, x.k, x.v, x.do))]
    dev_out = [(o, lse, dq, dk, dv), tuple(torch.empty_like(t) for t in (o, lse, dq, dk, dv))]
    rates = {}
    e2e_ms = max_over_ranks(pipelined_e2e(e2e_steps, pin, dev_in, dev_out, outs, r["compute"],
                                          r["stream"], rates), world)
    del dev_in, dev_out
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    # The host link's rates as these copies saw them (both directions at once, beside the
    # compute): when one step's copies take longer than its compute, the e2e figure is the
    # link's, not the kernels'.
    e2e = {"value": world * fl["fwd_bwd"] / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "steps": e2e_steps, "copies": "pipelined: step i+1 in and step i-1 out during step i",
           "h2d_ms": rates["h2d_ms"], "d2h_ms": rates["d2h_ms"],
           "h2d_gbs": h2d / (rates["h2d_ms"] * 1e-3) / 1e9,
           "d2h_gbs": d2h / (rates["d2h_ms"] * 1e-3) / 1e9}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, x_cpu)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.describe(), "B": B, "H": H, "N": N, "d": d,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between steps (256 MiB write)" if r["flush"]
                   else f"inputs larger than L2 ({r['in_bytes'] / 1e6:.0f} MB of Q, K, V, dO)",
                   "flops_per_step": fl["fwd_bwd"]},
        "pct_of_peak": value / world / peak_t,
        "pct_of_peak_sustained": value / world / pk["bf16_tflops_sustained"],
        "peak_kind": f"{pk['source']} bf16 dense, burst (CUDA events over a sub-second region)",
        "timing": r["timing"],
        "phases": {"fwd_tflops": r["fwd_tflops"], "bwd_tflops": r["bwd_tflops"],
                   "bwd_main_tflops": main_tf,
                   "fwd_ms": mean_phase[0], "preprocess_ms": mean_phase[1],
                   "bwd_main_ms": mean_phase[2], "dq_convert_ms": mean_phase[3],
                   "preprocess_gbs": r["preprocess_gbs"], "dq_convert_gbs": r["dq_convert_gbs"],
                   "hbm_peak_gbs": pk["hbm_gbs"]},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if world == 1 and not args.no_per_config and not args.heads:
        del x, r, o, lse, dq, dk, dv, pin, outs
        torch.cuda.empty_cache()
        line["per_config"] = per_config(fa, args, world, dev, args.workload)
    if rank == 0:
        print(json.dumps(line, default=float), flush=True)


# ------------------------------------------------------------------ decode (second workload)

DECODE_METRIC = "decode attention: KV-cache GB/s on 1 GB300 and % of measured HBM bandwidth"


def decode_oracle_seconds(w, x, pairs=None):
    import oracle  # test infrastructure: the CPU baseline leg only
    t0 = time.perf_counter()
    oracle.decode(x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy(), w.scale,
                  x.cache_len.numpy(), pairs)
    return time.perf_counter() - t0


def decode_cpu_baseline(w, x_cpu) -> dict:
    # A bounded sample: the query heads of the first 8 sequences (the fp64 conversion of the
    # whole cache alone would take most of the budget), scaled to the metric's bytes.
    nb = min(8, w.B)
    sub = W.DecodeInputs(x_cpu.q[:nb], x_cpu.k[:nb], x_cpu.v[:nb], x_cpu.cache_len[:nb], w.scale)
    secs = decode_oracle_seconds(w, sub)
    gb = acc.decode_bytes(w.Hq, w.Hkv, w.d, sub.cache_len.numpy()) / 1e9
    return {"value": gb / secs, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{nb} of {w.B} sequences of {w.describe()}: fp64 NumPy, {secs:.2f} s"}


def run_decode_reference(args, world, rank):
    """The CPU fp64 oracle on the decode workload, a bounded sample per step."""
    if rank != 0:
        return
    w = W.DECODE_WORKLOADS[args.workload]
    x = W.make_decode_inputs(w, seed=0)
    nb = min(4, w.B)
    sub = W.DecodeInputs(x.q[:nb], x.k[:nb], x.v[:nb], x.cache_len[:nb], w.scale)
    timed = max(1, min(args.steps, 20))
    times = [decode_oracle_seconds(w, sub) for _ in range(timed)]
    mean = sum(times) / len(times)
    value = acc.decode_bytes(w.Hq, w.Hkv, w.d, sub.cache_len.numpy()) / 1e9 / mean
    sample = f"{nb} of {w.B} sequences per step, {timed} of {args.steps} steps timed"
    print(json.dumps({
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.describe(), "sample": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def measure_decode(fa, w, steps, warmup, world, dev, x_cpu=None):
    """Time ``steps`` decode steps (split kernel + combine) of workload ``w`` with CUDA events
    on the launching stream and the clock sampler around the timed region."""
    x_cpu = x_cpu if x_cpu is not None else W.make_decode_inputs(w, seed=0)
    x = W.DecodeInputs(*(t.to(dev) for t in (x_cpu.q, x_cpu.k, x_cpu.v, x_cpu.cache_len)),
                       w.scale)
    stream = torch.cuda.current_stream(dev)
    o = torch.empty_like(x.q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.L, w.d), dtype=torch.uint8,
                     device=dev)

    def compute(inp, out):
        fa.fa_decode(inp[0], inp[1], inp[2], out[0], out[1], ws, inp[3], x.scale, stream)

    for _ in range(warmup):
        compute((x.q, x.k, x.v, x.cache_len), (o, lse))
    torch.cuda.synchronize()
    if fa.fa_device_error() != fa.FA_OK:
        raise RuntimeError("device error word set during warm-up (decode)")
    sampler = ClockSampler(device_uuid(dev))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for e0, e1 in evs:
        e0.record(stream)
        compute((x.q, x.k, x.v, x.cache_len), (o, lse))
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    if fa.fa_device_error() != fa.FA_OK:
        raise RuntimeError("device error word set during the timed region (decode)")
    ms = np.array([e0.elapsed_time(e1) for e0, e1 in evs])
    ms_per_step = max_over_ranks(float(ms.mean()), world)
    cl = x_cpu.cache_len.numpy()
    nbytes = acc.decode_bytes(w.Hq, w.Hkv, w.d, cl)
    return {"describe": w.describe(), "x": x, "x_cpu": x_cpu, "o": o, "lse": lse, "ws": ws,
            "compute": compute, "stream": stream, "ms": ms, "ms_per_step": ms_per_step,
            "timing": {"step_ms": summarize(ms)}, "clocks": clocks, "nbytes": nbytes,
            "gbs": world * nbytes / (ms_per_step * 1e-3) / 1e9,
            "tflops": world * acc.decode_flops(w.Hq, w.d, cl) / (ms_per_step * 1e-3) / 1e12,
            "launches": 2 * steps}


def run_decode(args, world, rank, local):
    """Decode over a KV cache: fa_decode per step, KV bytes read / event time."""
    from exact_io_aware_28_gb300 import fa
    w = W.DECODE_WORKLOADS[args.workload]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: the product path has no CPU fallback")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load()
    r = measure_decode(fa, w, args.steps, args.warmup, world, dev)
    x, x_cpu, o, lse = r["x"], r["x_cpu"], r["o"], r["lse"]
    gbs, nbytes, ms_per_step = r["gbs"], r["nbytes"], r["ms_per_step"]
    pk = peaks()

    # e2e: the cache, the queries and the lengths come from pinned host memory every step and
    # o, lse go back (pipelined as for the attention step).
    pin = [t.pin_memory() for t in (x_cpu.q, x_cpu.k, x_cpu.v, x_cpu.cache_len)]
    outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
    e2e_steps = max(2, min(args.steps, 4))
    dev_in = [(x.q, x.k, x.v, x.cache_len),
              tuple(torch.empty_like(t) for t in (x.q, x.k, x.v, x.cache_len))]
    dev_out = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]
    e2e_ms = max_over_ranks(pipelined_e2e(e2e_steps, pin, dev_in, dev_out, outs, r["compute"],
                                          r["stream"]), world)
    del dev_in, dev_out
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = decode_cpu_baseline(w, x_cpu)
    if rank == 0:
        splits = None
        try:
            splits = fa.fa_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.L, w.d) // (
                w.B * w.Hq * (w.d + 4) * 4)
        except Exception:
            pass
        print(json.dumps({
            "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.describe(), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "L": w.L,
                       "d": w.d, "splits": splits,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB of KV cache)",
                       "bytes_per_step": nbytes},
            "tflops": r["tflops"],
            "timing": r["timing"],
            "roofline": {"kernel": "decode split kernel + combine", "bound": "hbm",
                         "achieved": gbs / world, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / world / pk["hbm_gbs"],
                         "traffic": None if args.batch else recorded_traffic(args.workload,
                                                                             "decode_split"),
                         "peak_kind": f"{pk['source']} HBM copy bandwidth"},
            "cpu_baseline": cpu,
            "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "steps": e2e_steps,
                    "copies": "pipelined: step i+1 in and step i-1 out during step i"},
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
        }, default=float), flush=True)


# ------------------------------------------------------------------ FP8 forward

FP8_METRIC = ("FP8 (e4m3) attention forward TFLOP/s on 1 GB300, bf16 inputs encoded on the "
              "device inside the step, and % of dense fp8 tensor peak")


def fp8_oracle_head_seconds(x, head) -> float:
    """The oracle's encoding of one (b, h) head and its forward on the decoded inputs."""
    from oracle import fp8 as ofp8  # test infrastructure: the CPU legs only
    import oracle
    b, h = head
    sl = (slice(b, b + 1), slice(h, h + 1))
    q, k, v = (t[sl].to(torch.float64).numpy() for t in (x.q, x.k, x.v))
    t0 = time.perf_counter()
    q8, sq = ofp8.quantize_blocks(q)
    k8, sk = ofp8.quantize_blocks(k)
    v8, sv = ofp8.quantize_heads(v)
    Q, K = ofp8.dequantize_blocks(q8, sq)[0, 0], ofp8.dequantize_blocks(k8, sk)[0, 0]
    V = (v8 * sv[:, :, None, None])[0, 0]
    keep = oracle.keep_mask(Q.shape[0], x.causal)
    oracle.forward_head(Q, K, V, x.scale, keep)
    return time.perf_counter() - t0


def run_fp8_reference(args, world, rank):
    """The CPU oracle (encoding + fp64 forward) on one (b, h) head of the workload per step."""
    if rank != 0:
        return
    w = W.FP8_WORKLOADS[args.workload]
    x = W.make_inputs(w, seed=0)
    small = W.make_inputs(W.custom("warm", 1, 1, 256, w.d, causal=w.causal), seed=1)
    for _ in range(args.warmup):
        fp8_oracle_head_seconds(small, (0, 0))
    timed = max(1, min(args.steps, 20))
    times = [fp8_oracle_head_seconds(x, (0, i % w.H)) for i in range(timed)]
    mean = sum(times) / len(times)
    value = acc.flops(1, 1, w.N, w.d, w.causal)["fwd"] / mean / 1e12
    sample = f"one (batch, head) of {w.describe()} per step; {timed} of {args.steps} steps timed"
    print(json.dumps({
        "impl": "reference", "metric": FP8_METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.describe(), "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def measure_fp8(fa, w, steps, warmup, world, dev, x_cpu=None):
    """Time ``steps`` FP8 steps (encode Q, K, V on the device + the e4m3 forward) of workload
    ``w`` with CUDA events on the launching stream and the clock sampler."""
    x_cpu = x_cpu if x_cpu is not None else W.make_inputs(w, seed=0)
    q, k, v = (t.to(dev) for t in (x_cpu.q, x_cpu.k, x_cpu.v))
    B, H, N, d = w.B, w.H, w.N, w.d
    nb = (N + 127) // 128
    Np = nb * 128
    stream = torch.cuda.current_stream(dev)
    enc = (torch.empty((B, H, N, d), dtype=torch.uint8, device=dev),
           torch.empty((B, H, nb), dtype=torch.float32, device=dev),
           torch.empty((B, H, N, d), dtype=torch.uint8, device=dev),
           torch.empty((B, H, nb), dtype=torch.float32, device=dev),
           torch.empty((B, H, d, Np), dtype=torch.uint8, device=dev),
           torch.empty((B, H), dtype=torch.float32, device=dev))
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)

    def run(inp, out, ev=None):
        q8, sq, k8, sk, vt8, sv = enc
        if ev:
            ev[0].record(stream)
        fa.fa_fp8_quantize_qk(inp[0], q8, sq, stream)
        fa.fa_fp8_quantize_qk(inp[1], k8, sk, stream)
        fa.fa_fp8_quantize_v(inp[2], vt8, sv, stream)
        if ev:
            ev[1].record(stream)
        fa.fa_fwd_fp8(q8, k8, vt8, sq, sk, sv, out[0], out[1], w.causal, None, None, w.scale,
                      stream)
        if ev:
            ev[2].record(stream)

    for _ in range(warmup):
        run((q, k, v), (o, lse))
    torch.cuda.synchronize()
    if fa.fa_device_error() != fa.FA_OK:
        raise RuntimeError("device error word set during warm-up (fp8)")
    sampler = ClockSampler(device_uuid(dev))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for i in range(steps):
        run((q, k, v), (o, lse), evs[i])
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    if fa.fa_device_error() != fa.FA_OK:
        raise RuntimeError("device error word set during the timed region (fp8)")
    phase = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(2)]
                      for i in range(steps)])  # ms: encode, forward
    step_ms = phase.sum(axis=1)
    ms_per_step = max_over_ranks(float(step_ms.mean()), world)
    fl = acc.flops(B, H, N, d, w.causal)["fwd"]
    mean_phase = phase.mean(axis=0)
    return {"describe": w.describe(), "x_cpu": x_cpu, "qkv": (q, k, v), "o": o, "lse": lse,
            "run": run, "stream": stream, "flops": fl, "ms_per_step": ms_per_step,
            "value": world * fl / (ms_per_step * 1e-3) / 1e12,
            "fwd_tflops": fl / (mean_phase[1] * 1e-3) / 1e12,
            "encode_gbs": acc.fp8_encode_bytes(B, H, N, d) / (mean_phase[0] * 1e-3) / 1e9,
            "timing": {"step_ms": summarize(step_ms), "encode_ms": summarize(phase[:, 0]),
                       "fwd_ms": summarize(phase[:, 1])},
            "clocks": clocks, "launches": 6 * steps}


def run_fp8(args, world, rank, local):
    """One step = encode Q, K, V to e4m3 (3 + 1 kernels) + the e4m3 forward (1 kernel)."""
    from exact_io_aware_28_gb300 import fa
    w = W.FP8_WORKLOADS[args.workload]
    if args.heads:
        w = dataclasses.replace(w, H=args.heads)
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: the product path has no CPU fallback")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load()
    r = measure_fp8(fa, w, args.steps, args.warmup, world, dev)
    B, H, N, d = w.B, w.H, w.N, w.d
    x_cpu, (q, k, v), o, lse = r["x_cpu"], r["qkv"], r["o"], r["lse"]
    fl, value, ms_per_step, fwd_tf = r["flops"], r["value"], r["ms_per_step"], r["fwd_tflops"]
    pk = peaks()
    # Dense fp8 peak: the measured burst bf16 figure times the nominal fp8 / bf16 ratio
    # (4.5 / 2.25); the forward kernel is timed by CUDA events over a sub-second region.
    peak8 = 2.0 * pk["bf16_tflops"]
    peak8_sustained = 2.0 * pk["bf16_tflops_sustained"]

    pin = [t.pin_memory() for t in (x_cpu.q, x_cpu.k, x_cpu.v)]
    outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
    e2e_steps = max(2, min(args.steps, 20))
    dev_in = [(q, k, v), tuple(torch.empty_like(t) for t in (q, k, v))]
    dev_out = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]

    def compute(inp, out):
        # the codes live on the compute stream only: one set serves every step
        r["run"](inp, out)

    e2e_ms = max_over_ranks(pipelined_e2e(e2e_steps, pin, dev_in, dev_out, outs, compute,
                                          r["stream"]), world)
    del dev_in, dev_out
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nh, secs = sample_heads(lambda hd: fp8_oracle_head_seconds(x_cpu, hd), H)
        cpu = {"value": nh * acc.flops(1, 1, N, d, w.causal)["fwd"] / secs / 1e12, "unit": UNIT,
               "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{nh} (batch, head) pair(s) of {w.describe()}: NumPy e4m3 encoding + "
                         f"fp64 forward, {secs:.1f} s; FLOPs by the same convention"}
    if rank == 0:
        print(json.dumps({
            "metric": FP8_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic",
            "config": {"workload": w.describe(), "B": B, "H": H, "N": N, "d": d,
                       "operands": "e4m3; power-of-two scales per 128 rows (Q, K), per head (V)",
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "inputs larger than L2 (402 MB of bf16 Q, K, V at the full size)",
                       "flops_per_step": fl},
            "pct_of_peak": value / world / peak8,
            "timing": r["timing"],
            "phases": {"encode_gbs": r["encode_gbs"], "fwd_kernel_tflops": fwd_tf,
                       "hbm_peak_gbs": pk["hbm_gbs"]},
            "roofline": {"kernel": "e4m3 forward", "bound": "tensor", "achieved": fwd_tf,
                         "peak": peak8, "unit": "TFLOP/s", "frac": fwd_tf / peak8,
                         "frac_of_sustained": fwd_tf / peak8_sustained,
                         "traffic": None if args.heads else recorded_traffic(args.workload,
                                                                             "fwd_fp8"),
                         "peak_kind": f"{pk['source']} bf16 dense burst x 2 (nominal "
                                      f"fp8/bf16 ratio)"},
            "cpu_baseline": cpu,
            "e2e": {"value": world * fl / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "steps": e2e_steps,
                    "copies": "pipelined: step i+1 in and step i-1 out during step i"},
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
        }, default=float), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload",
                    choices=W.ORDER + list(W.DROPOUT_WORKLOADS) + list(W.DECODE_WORKLOADS) +
                    list(W.FP8_WORKLOADS),
                    default="long_causal")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config block of the default run")
    ap.add_argument("--heads", type=int, default=0,
                    help="override the workload's head count (smaller cases for profiling)")
    ap.add_argument("--batch", type=int, default=0,
                    help="decode workloads: override the number of sequences (profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    check_world(args.gpus)
    world, rank, local = dist_setup()
    decode = args.workload in W.DECODE_WORKLOADS
    fp8 = args.workload in W.FP8_WORKLOADS
    if args.impl == "reference":
        ref = run_decode_reference if decode else run_fp8_reference if fp8 else run_reference
        ref(args, world, rank)
    else:
        (run_decode if decode else run_fp8 if fp8 else run_ours)(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
