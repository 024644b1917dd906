"""GPU parity of attention with dropout: the library (through the C ABI) against the CPU
fp64 dropout oracle, which regenerates the same mask from its own Philox4x32-10.

The generator bytes are compared bit for bit (fa_dropout_random_bytes); the forward and
backward are compared with the tolerances of the plain path (tests/_parity.py), the O bound
multiplied by the keep scale 256 / (256 - t) that multiplies every rounding of O, on small
shapes over several tiles with ragged tails, every mask mode, d = 64 and 128, bf16 and
fp32, thresholds from 1 to 255, and on one full head of the bench's launch (1 x 32 x 16384
x 128, causal, threshold 26).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_28_gb300 import fa
from exact_io_aware_28_gb300 import workloads as W

from _parity import compare as _compare, np64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("BH,n_q,n_k,seed,offset", [
    (1, 16, 32, 0, 0), (3, 37, 129, 0x1234567890ABCDEF, 5), (2, 300, 257, 2 ** 64 - 1, 2 ** 32 - 1),
    (1, 1, 1, 7, 0), (4, 1024, 640, 99, 3),
])
def test_generator_bytes_match_the_oracle(BH, n_q, n_k, seed, offset):
    out = torch.full((BH, n_q, n_k), 0xAB, dtype=torch.uint8, device="cuda")
    fa.fa_dropout_random_bytes(out, seed, offset)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for bh in range(BH):
        ref = oracle.dropout.random_bytes(seed, offset, bh, n_q, n_k)
        assert np.array_equal(got[bh], ref), bh


def _inputs(B, H, N, d, dtype, causal=False, kv=False, bm=None, seed=0):
    w = W.custom("drop", B, H, N, d, dtype, causal=causal)
    x = W.make_inputs(w, seed=seed, device="cuda")
    if kv:
        g = torch.Generator().manual_seed(seed + 7)
        x.kv_len = torch.randint(1, N + 1, (B,), generator=g, dtype=torch.int32).cuda()
    if bm is not None:
        x.blockmask = bm.cuda()
    return x


def _run(x, t, seed, offset=0):
    o, lse = fa.forward_dropout(x.q, x.k, x.v, t, seed, offset, x.causal, x.blockmask,
                                x.kv_len, x.scale)
    dq, dk, dv = fa.backward_dropout(x.q, x.k, x.v, o, lse, x.do, t, seed, offset, x.causal,
                                     x.blockmask, x.kv_len, x.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    return o, lse, dq, dk, dv


def _oracle(x, t, seed, offset=0, heads=None):
    q, k, v, do = (np64(a) for a in (x.q, x.k, x.v, x.do))
    bm = None if x.blockmask is None else x.blockmask.cpu().numpy()
    kl = None if x.kv_len is None else x.kv_len.cpu().numpy()
    dr = oracle.dropout
    o, lse = dr.forward(q, k, v, x.scale, t, seed, offset, x.causal, bm, kl, heads=heads)
    dq, dk, dv, _ = dr.backward(q, k, v, do, x.scale, t, seed, offset, x.causal, bm, kl,
                                heads=heads)
    return o, lse, dq, dk, dv


def compare(lib_out, ref_out, dtype, t, heads=None):
    """The plain tolerances, the O bound times the keep scale 256 / (256 - t)."""
    return _compare(lib_out, ref_out, dtype, heads=heads, o_scale=256.0 / (256 - t))


def _blockmask(N, seed):
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand((nb, nb), generator=g) < 0.5).to(torch.uint8)
    bm.fill_diagonal_(1)
    return bm


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,mode", [(7, "dense"), (130, "causal"), (257, "padded"),
                                    (640, "block"), (300, "block_causal"), (384, "causal")])
def test_small_shapes(dtype, d, N, mode):
    kw = {"causal": "causal" in mode, "kv": mode == "padded",
          "bm": _blockmask(N, N) if "block" in mode else None}
    x = _inputs(2, 2, N, d, dtype, seed=N + d, **kw)
    seed = 1000 + N
    compare(_run(x, 64, seed), _oracle(x, 64, seed), dtype, 64)


@pytest.mark.parametrize("t", [1, 26, 128, 200, 255])
def test_thresholds(t):
    x = _inputs(1, 3, 520, 128, "bf16", causal=True, seed=t)
    compare(_run(x, t, 42, offset=t), _oracle(x, t, 42, offset=t), "bf16", t)


def test_rows_without_visible_keys():
    N = 300
    bm = torch.ones((3, 3), dtype=torch.uint8)
    bm[1, :] = 0
    x = _inputs(2, 2, N, 64, "bf16", bm=bm, seed=3)
    x.kv_len = torch.tensor([0, 200], dtype=torch.int32, device="cuda")
    out = _run(x, 100, 5)
    compare(out, _oracle(x, 100, 5), "bf16", 100)
    assert torch.all(out[0][0] == 0) and torch.all(torch.isneginf(out[1][0]))


def test_zero_threshold_is_the_plain_path():
    x = _inputs(1, 2, 300, 128, "bf16", causal=True, seed=9)
    o0, lse0 = fa.forward(x.q, x.k, x.v, x.causal, None, None, x.scale)
    o, lse = fa.forward_dropout(x.q, x.k, x.v, 0, 123, 0, x.causal, None, None, x.scale)
    assert torch.equal(o, o0) and torch.equal(lse, lse0)
    g0 = fa.backward(x.q, x.k, x.v, o0, lse0, x.do, x.causal, None, None, x.scale)
    g = fa.backward_dropout(x.q, x.k, x.v, o, lse, x.do, 0, 123, 0, x.causal, None, None,
                            x.scale)
    for a, b in zip(g, g0):
        torch.testing.assert_close(a.float(), b.float(), rtol=1e-2, atol=1e-3)


def test_seed_and_offset_select_the_mask_and_repeat_exactly():
    x = _inputs(1, 2, 400, 64, "bf16", seed=10)
    a = _run(x, 50, 7)
    b = _run(x, 50, 7)
    c = _run(x, 50, 8)
    e = _run(x, 50, 7, offset=1)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])   # dK, dV: no atomics
    assert not torch.equal(a[0], c[0]) and not torch.equal(a[0], e[0])
    assert torch.equal(a[1], c[1])   # lse does not depend on the mask


@pytest.mark.slow
def test_long_causal_dropout_full_size_one_head():
    w = W.DROPOUT_WORKLOADS["long_causal_dropout"]
    x = W.make_inputs(w, seed=0, device="cuda")
    out = _run(x, w.drop_threshold, w.drop_seed)
    heads = [(0, 21)]
    errs = compare(out, _oracle(x, w.drop_threshold, w.drop_seed, heads=heads), "bf16",
                   w.drop_threshold, heads=heads)
    print(errs)
    for t in (out[0], out[2], out[3], out[4]):
        assert torch.isfinite(t.float()).all()
