"""Decode with grouped key/value heads: the CUDA path (fa_decode through the C ABI) against
the fp64 oracle on the same bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_28_gb300 import fa
from exact_io_aware_28_gb300 import workloads as W

from _parity import TOL

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _run(x, cache_len=True):
    cl = x.cache_len if cache_len else None
    o, lse = fa.decode(x.q, x.k, x.v, cl, x.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    return o, lse


def _check(o, lse, x, pairs=None, cache_len=True):
    cl = x.cache_len.cpu().numpy() if cache_len else None
    o_ref, lse_ref = oracle.decode(_np(x.q), _np(x.k), _np(x.v), x.scale, cl, pairs)
    o_g, lse_g = _np(o), _np(lse)
    if pairs is not None:
        idx = tuple(np.array(pairs).T)
        o_ref, lse_ref, o_g, lse_g = o_ref[idx], lse_ref[idx], o_g[idx], lse_g[idx]
    empty = ~np.isfinite(lse_ref)
    assert np.array_equal(~np.isfinite(lse_g), empty)
    assert np.all(o_g[empty] == 0)
    assert np.abs(o_g - o_ref).max() <= TOL["bf16"]["o"]
    live = ~empty
    if live.any():
        assert np.abs(lse_g[live] - lse_ref[live]).max() <= TOL["bf16"]["lse"]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hkv", [8, 4, 2, 1])
@pytest.mark.parametrize("L", [1, 63, 64, 300, 1000])
def test_small_shapes_ragged(d, Hkv, L):
    w = W.DecodeWorkload("t", 3, 8, Hkv, L, d, ragged=True)
    x = W.make_decode_inputs(w, seed=L + d + Hkv, device="cuda")
    _check(*_run(x), x)


@pytest.mark.parametrize("d", [64, 128])
def test_full_caches_without_lengths(d):
    w = W.DecodeWorkload("t", 2, 16, 4, 777, d)
    x = W.make_decode_inputs(w, seed=3, device="cuda")
    _check(*_run(x, cache_len=False), x, cache_len=False)


def test_rows_past_the_cache_length_are_never_read():
    w = W.DecodeWorkload("t", 4, 8, 2, 500, 128)
    x = W.make_decode_inputs(w, seed=5, device="cuda")
    x.cache_len = torch.tensor([1, 130, 257, 500], dtype=torch.int32, device="cuda")
    for b, n in enumerate(x.cache_len.tolist()):
        x.k[b, :, n:] = float("nan")
        x.v[b, :, n:] = float("nan")
    o, lse = _run(x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    _check(o, lse, x)


@pytest.mark.parametrize("d", [64, 128])
def test_empty_cache_gives_zero_and_minus_inf(d):
    w = W.DecodeWorkload("t", 3, 4, 2, 200, d)
    x = W.make_decode_inputs(w, seed=6, device="cuda")
    x.cache_len = torch.tensor([0, 200, 7], dtype=torch.int32, device="cuda")
    o, lse = _run(x)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    _check(o, lse, x)


def test_many_splits_one_long_sequence():
    # One (sequence, K/V head) pair: the cache is split into many key ranges.
    w = W.DecodeWorkload("t", 1, 8, 1, 20000, 128, ragged=True)
    x = W.make_decode_inputs(w, seed=9, device="cuda")
    _check(*_run(x), x)


def test_deterministic():
    w = W.DecodeWorkload("t", 4, 32, 8, 3000, 128, ragged=True)
    x = W.make_decode_inputs(w, seed=11, device="cuda")
    o1, l1 = _run(x)
    o2, l2 = _run(x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.slow
def test_llama8b_decode_workload_sampled():
    # The benchmark shape (64 sequences, 32 query heads over 8 K/V heads, 8192 keys, d=128),
    # checked on sampled (sequence, head) pairs against the oracle.
    w = W.DECODE_WORKLOADS["decode_llama8b"]
    x = W.make_decode_inputs(w, seed=0, device="cuda")
    o, lse = _run(x)
    rng = np.random.default_rng(0)
    pairs = sorted({(int(rng.integers(w.B)), int(rng.integers(w.Hq))) for _ in range(24)})
    pairs += [(0, 0), (w.B - 1, w.Hq - 1)]
    _check(o, lse, x, pairs)


@pytest.mark.slow
def test_million_key_cache():
    # A cache of 2^20 + 5 keys for one sequence (8 query heads over one K/V head, d = 128):
    # the longest ranges and the most splits of one (sequence, head) pair, with a ragged end.
    w = W.DecodeWorkload("t", 1, 8, 1, (1 << 20) + 5, 128)
    x = W.make_decode_inputs(w, seed=13, device="cuda")
    o, lse = _run(x, cache_len=False)
    _check(o, lse, x, cache_len=False)
