"""GPU parity of the FP8 (e4m3) path, through the C ABI, against the CPU oracle.

The encoders are integer work decided by floating point in the same precision on both
sides (bf16 inputs, exact power-of-two scaling, round to nearest even), so their codes
and scales must match the oracle's exactly.  The forward is compared with the oracle's
exact attention on the oracle's own decoding of the same bf16 inputs; its one extra
rounding (P to e4m3) is held to the bound of _fp8_bound: elementwise, and in root mean
square against the predicted spread.  The logsumexp comes from unrounded probabilities
and keeps the bf16 path's tolerance, 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from exact_io_aware_28_gb300 import fa
from exact_io_aware_28_gb300 import workloads as W

import _fp8_bound

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _vt_key():
    k = np.arange(128)
    return 32 * (k >> 5) + 16 * ((k >> 2) & 1) + 8 * ((k >> 1) & 1) + 2 * ((k >> 3) & 3) + (k & 1)


def _unpermute(vt8, N):
    """[B, H, 128, Np] e4m3 codes in the documented key order -> ([B, H, N, 128], padding)."""
    B, H, D, Np = vt8.shape
    keys = (np.arange(Np // 128)[:, None] * 128 + _vt_key()[None, :]).reshape(-1)
    v8 = np.zeros((B, H, Np, D), np.uint8)
    v8[:, :, keys, :] = vt8.transpose(0, 1, 3, 2)
    return v8[:, :, :N], v8[:, :, N:]


def _bf16(B, H, N, seed, mult=1.0):
    x = W.make_inputs(W.custom("fp8", B, H, N, 128), seed=seed)
    return (x.q.float() * mult).to(torch.bfloat16), x.k, x.v


def test_key_order_is_a_permutation_of_each_block():
    assert sorted(_vt_key().tolist()) == list(range(128))


@pytest.mark.parametrize("N", [1, 127, 300, 1024])
@pytest.mark.parametrize("mult", [1.0, 1000.0, 1e-3])
def test_quantize_qk_matches_the_oracle_exactly(N, mult):
    q, _, _ = _bf16(2, 3, N, seed=N, mult=mult)
    q[1, 2, :min(N, 128)] = 0  # an all-zero block: scale 1, codes 0
    x8, s = fa.fp8_quantize_qk(q.cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    ref8, refs = ofp8.quantize_blocks(_np(q))
    assert np.array_equal(_np(s), refs)
    assert np.array_equal(ofp8.e4m3_decode(x8.cpu().numpy()), ref8)


@pytest.mark.parametrize("N", [1, 200, 384, 1000])
@pytest.mark.parametrize("mult", [1.0, 300.0])
def test_quantize_v_matches_the_oracle_exactly(N, mult):
    _, _, v = _bf16(2, 3, N, seed=N + 1)
    v = (v.float() * mult).to(torch.bfloat16)
    v[0, 1] = 0  # an all-zero head
    vt8, s = fa.fp8_quantize_v(v.cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    ref8, refs = ofp8.quantize_heads(_np(v))
    assert np.array_equal(_np(s), refs)
    codes, pad = _unpermute(vt8.cpu().numpy(), N)
    assert np.array_equal(ofp8.e4m3_decode(codes), ref8)
    assert not pad.any()


def _decoded(x_q, x_k, x_v):
    q8, sq = ofp8.quantize_blocks(_np(x_q))
    k8, sk = ofp8.quantize_blocks(_np(x_k))
    v8, sv = ofp8.quantize_heads(_np(x_v))
    return (ofp8.dequantize_blocks(q8, sq), ofp8.dequantize_blocks(k8, sk),
            v8 * sv[:, :, None, None])


def _check(x, heads=None, rows=None):
    o, lse = fa.attention_fp8(x.q, x.k, x.v, x.causal, x.blockmask, x.kv_len, x.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    o, lse = _np(o), _np(lse)
    B, H, N, _ = x.q.shape
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    bm = None if x.blockmask is None else x.blockmask.cpu().numpy()
    kl = None if x.kv_len is None else x.kv_len.cpu().numpy()
    sel = slice(None) if rows is None else np.asarray(rows)
    worst = []
    for b, h in heads:
        Q, K, V = (a[0, 0] for a in _decoded(x.q[b:b + 1, h:h + 1], x.k[b:b + 1, h:h + 1],
                                              x.v[b:b + 1, h:h + 1]))
        keep = _fp8_bound.keep_for(N, x.causal, bm, kl, b)[sel]
        ro, rlse, _ = oracle.forward_head(Q[sel], K, V, x.scale, keep)
        worst.append(_fp8_bound.check(o[b, h][sel], ro, Q[sel], K, V, x.scale, keep))
        dead = np.isneginf(rlse)
        got = lse[b, h][sel]
        assert np.array_equal(np.isneginf(got), dead)
        assert np.all(o[b, h][sel][dead] == 0)
        if (~dead).any():
            assert np.abs(got[~dead] - rlse[~dead]).max() <= LSE_TOL
    return worst


def _inputs(B, H, N, causal=False, seed=0, **kw):
    w = W.custom("fp8", B, H, N, 128, causal=causal, **kw)
    return W.make_inputs(w, seed=seed, device="cuda")


def _blockmask(N, seed, density=0.5):
    nb = (N + 127) // 128
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand((nb, nb), generator=g) < density).to(torch.uint8)
    bm.fill_diagonal_(1)
    return bm


@pytest.mark.parametrize("B,H,N,causal", [
    (1, 2, 384, True), (2, 2, 300, False), (1, 3, 1000, True), (1, 2, 1, False),
    (1, 2, 129, True), (2, 1, 2048, False),
])
def test_forward_dense_and_causal(B, H, N, causal):
    print(_check(_inputs(B, H, N, causal, seed=N)))


def test_forward_key_padding():
    x = _inputs(3, 2, 640, seed=3)
    x.kv_len = torch.tensor([1, 500, 640], dtype=torch.int32, device="cuda")
    print(_check(x))


@pytest.mark.parametrize("causal", [False, True])
def test_forward_block_mask(causal):
    x = _inputs(1, 2, 768, causal, seed=5)
    x.blockmask = _blockmask(768, 5).cuda()
    print(_check(x))


def test_forward_rows_without_visible_keys():
    x = _inputs(2, 2, 384, seed=9)
    bm = _blockmask(384, 9, density=1.0)
    bm[1, :] = 0                       # query rows 128..255 see nothing
    x.blockmask = bm.cuda()
    x.kv_len = torch.tensor([0, 384], dtype=torch.int32, device="cuda")  # sequence 0: no keys
    print(_check(x))


def test_forward_large_logits():
    # Q head 0 x 4 (exact in bf16): sharper rows, most probabilities far below 2^-6.
    print(_check(_inputs(1, 2, 1024, True, seed=4, q_head0_mult=4.0)))


def test_forward_is_deterministic():
    x = _inputs(1, 4, 1024, True, seed=2)
    a = fa.attention_fp8(x.q, x.k, x.v, True)
    b = fa.attention_fp8(x.q, x.k, x.v, True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.slow
def test_long_causal_full_size_sampled_rows():
    # The benchmark launch (1 x 32 x 16384 x 128, causal), sampled: two heads, the first and
    # last rows, a tile boundary and a block of rows deep in the sequence.
    x = W.make_inputs(W.WORKLOADS["long_causal"], seed=0, device="cuda")
    rows = np.r_[0:4, 126:131, 8000:8064, 16380:16384]
    print(_check(x, heads=[(0, 0), (0, 31)], rows=rows))
