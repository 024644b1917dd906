"""Host-side logic: the seeded workload generator and the FLOP/byte accounting."""
import json
import os

import numpy as np
import pytest
import torch

from exact_io_aware_28_gb300 import accounting as acc
from exact_io_aware_28_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_generator_is_deterministic_and_shaped():
    w = W.custom("t", 2, 3, 130, 64, "bf16", padded=True)
    a = W.make_inputs(w, seed=7)
    b = W.make_inputs(w, seed=7)
    for x, y in zip((a.q, a.k, a.v, a.do), (b.q, b.k, b.v, b.do)):
        assert x.shape == (2, 3, 130, 64) and x.dtype == torch.bfloat16
        assert torch.equal(x, y)
    assert torch.equal(a.kv_len, b.kv_len)
    assert a.kv_len.dtype == torch.int32
    assert int(a.kv_len.min()) >= 128 and int(a.kv_len.max()) <= 130
    c = W.make_inputs(w, seed=8)
    assert not torch.equal(a.q, c.q)


def test_named_workloads():
    assert W.ORDER == list(W.WORKLOADS)
    w = W.WORKLOADS["tiny_fp32"]
    x = W.make_inputs(w)
    assert x.q.dtype == torch.float32 and x.q.shape == (1, 1, 128, 64)
    assert x.scale == pytest.approx(1 / 8)
    w = W.WORKLOADS["gpt2_causal"]
    assert (w.B, w.H, w.N, w.d, w.causal) == (4, 12, 1024, 64, True)
    # head 0 of Q is the fp32 draw times 4, an exact power-of-two scaling in bf16
    g = torch.Generator().manual_seed(0)
    q32 = torch.randn((4, 12, 1024, 64), generator=g)
    x = W.make_inputs(w)
    assert torch.equal(x.q[:, 0].float(), (q32[:, 0] * 4).to(torch.bfloat16).float())
    assert torch.equal(x.q[:, 1].float(), q32[:, 1].to(torch.bfloat16).float())
    w = W.WORKLOADS["block_sparse"]
    assert (w.B, w.H, w.N, w.d) == (2, 8, 8192, 64)


def test_block_mask_recipe():
    w = W.custom("bs", 1, 1, 8192, 64, "bf16", block_sparse=True)
    x = W.make_inputs(w)
    bm = x.blockmask.numpy()
    assert bm.shape == (64, 64) and bm.dtype == np.uint8
    assert np.all(np.diag(bm) == 1)
    off = bm[~np.eye(64, dtype=bool)]
    assert 0.2 < off.mean() < 0.3


def test_page_byte_figures():
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))
    for key in ("score_matrix_100k_fp16", "score_matrix_4096_32heads_fp16"):
        c = g[key]
        assert acc.score_matrix_bytes(c["n"], c["heads"], c["bytes_per_element"]) == c["bytes"]
    for n, d, ratio in g["memory_saving_ratio"]["cases"]:
        assert acc.memory_saving_ratio(n, d) == ratio
    for p, w_, ridge, tol in g["ridge_points"]["cases"]:
        assert abs(acc.ridge_point(p, w_) - ridge) < tol
    c = g["bf16_vector_add_intensity"]
    assert acc.intensity(c["flops"], c["bytes"]) == pytest.approx(1 / 6)


def test_flop_convention():
    f = acc.flops(1, 32, 16384, 128, causal=True)
    assert f["fwd"] == pytest.approx(2.199023e12, rel=1e-6)
    assert f["fwd_bwd"] == pytest.approx(7.696581e12, rel=1e-6)
    assert acc.flops(1, 1, 128, 64)["fwd_bwd"] == 14 * 128 * 128 * 64
    bm = np.eye(4, dtype=np.uint8)
    bm[3, 0] = 1
    f = acc.flops(1, 1, 4 * 128 - 5, 64, blockmask=bm)
    # three full diagonal blocks, one ragged diagonal block (123 x 123), one 123 x 128 block
    pairs = 3 * 128 * 128 + 123 * 123 + 123 * 128
    assert f["fwd"] == 4 * 64 * pairs


def test_hbm_byte_counts():
    assert acc.preprocess_bytes(1, 32, 16384, 128) == 2 * 134217728 + 2097152 + 268435456
    assert acc.dq_convert_bytes(1, 32, 16384, 128) == 268435456 + 134217728
