"""Host-side pieces of the benchmark (no GPU): the timing statistics, the JSON line of the
reference arm, and the decode byte/FLOP accounting."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_io_aware_28_gb300 import accounting as acc  # noqa: E402


def test_summarize_statistics():
    x = np.array([6.70, 6.72, 6.69, 6.75, 6.71, 6.70, 6.68, 6.73, 6.71, 6.70])
    s = bench.summarize(x)
    assert s["median"] == pytest.approx(np.median(x))
    assert s["p95"] == pytest.approx(np.percentile(x, 95))
    assert s["mean"] == pytest.approx(x.mean())
    lo, hi = s["ci95"]
    assert lo < x.mean() < hi
    stats = pytest.importorskip("scipy.stats")
    half = stats.t.ppf(0.975, len(x) - 1) * x.std(ddof=1) / np.sqrt(len(x))
    assert hi - lo == pytest.approx(2 * half)
    assert "ci95" not in bench.summarize([1.0])


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    for k in ("metric", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "config",
              "cpu_baseline", "e2e", "dtype"):
        assert k in d, k
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


def test_decode_accounting():
    cache_len = np.array([8192, 4096])
    # per visible key and K/V head: K and V rows of d bf16 values
    assert acc.decode_bytes(32, 8, 128, cache_len) == (
        2 * (8192 + 4096) * 8 * 128 * 2 + 2 * 32 * (128 * 2 + 128 * 2 + 4))
    assert acc.decode_flops(32, 128, cache_len) == 4 * 128 * 32 * (8192 + 4096)
    # the course page's intensity: about Hq / Hkv FLOP per byte of cache
    fl, by = acc.decode_flops(32, 128, [8192]), acc.decode_bytes(32, 8, 128, [8192])
    assert fl / by == pytest.approx(32 / 8, rel=0.01)


def test_dropout_workload_and_its_oracle_leg():
    from exact_io_aware_28_gb300 import workloads as W
    w = bench.TRAIN_WORKLOADS["long_causal_dropout"]
    assert w.drop_threshold == 26 and "dropout 26/256" in w.describe()
    assert (w.B, w.H, w.N, w.d, w.causal) == (1, 32, 16384, 128, True)
    small = W.custom("drop_small", 1, 2, 256, 64, "bf16", causal=True, drop_threshold=26,
                     drop_seed=5)
    x = W.make_inputs(small, seed=0)
    assert bench.oracle_head_seconds(x, (0, 1), small) > 0
    assert bench.oracle_head_seconds(x, (0, 1)) > 0


def test_cpu_sample_stops_after_the_time_budget():
    calls = []

    def fake(head):
        calls.append(head)
        return 4.0
    assert bench.sample_heads(fake, H=32) == (3, 12.0)       # 4 s heads: three reach 10 s
    assert calls == [(0, 0), (0, 1), (0, 2)]
    assert bench.sample_heads(lambda hd: 30.0, H=32) == (1, 30.0)
    assert bench.sample_heads(lambda hd: 0.1, H=32) == (4, 0.4)   # never more than four
    assert bench.sample_heads(lambda hd: 0.1, H=2) == (2, 0.2)


def test_gpus_must_match_the_ranks_started(monkeypatch):
    # --gpus 8 without torchrun would time one GPU and call it eight: refused up front.
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.check_world(1)
    with pytest.raises(SystemExit, match="WORLD_SIZE=1"):
        bench.check_world(8)
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.check_world(2)
    with pytest.raises(SystemExit):
        bench.check_world(1)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "4",
                          "--impl", "reference", "--workload", "tiny_fp32"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env={k: v for k, v in os.environ.items() if k != "WORLD_SIZE"})
    assert out.returncode != 0 and "WORLD_SIZE=1" in out.stderr
    assert not [l for l in out.stdout.splitlines() if l.startswith("{")]


def test_per_config_covers_every_other_workload():
    from exact_io_aware_28_gb300 import workloads as W
    names = set(bench.PER_CONFIG)
    # the four other scope configurations, the dropout and FP8 steps and decode
    assert set(W.ORDER) - {"long_causal"} <= names
    assert {"long_causal_dropout", "long_causal_fp8", "decode_llama8b"} <= names
    assert "long_causal_chunks4" in names        # the sequence-sharded schedule (one GPU)
    for n in names:
        assert (n in bench.TRAIN_WORKLOADS or n in W.FP8_WORKLOADS or n in W.DECODE_WORKLOADS
                or n in bench.CHUNKED)
