"""Pins of the dropout oracle (oracle/dropout.py) against things other than itself: the
published known-answer vectors of Philox4x32-10, numpy's Philox bit generator for the
shared round structure, brute-force recomputation of single bytes, the statistics a
uniform byte stream must have, the plain oracle at zero drop probability, the expectation
over masks, finite differences and the gradient identities of the chain rule."""
import json
import os

import numpy as np
import pytest

from oracle import attention as A
from oracle import dropout as DR

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")


def _masks(n, seed=0):
    g = np.random.default_rng(seed)
    nb = (n + 1) // 2
    bm = (g.random((nb, nb)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    hole = bm.copy()
    hole[0, :] = 0
    return {
        "dense": A.keep_mask(n),
        "causal": A.keep_mask(n, causal=True),
        "padded": A.keep_mask(n, kv_len=max(1, n - 2)),
        "block": A.keep_mask(n, blockmask=bm, block=2),
        "fully_masked_rows": A.keep_mask(n, blockmask=hole, block=2),
    }


# ---------------------------------------------------------------- the generator

def test_philox4x32_10_known_answer_vectors():
    kat = json.load(open(GOLDEN))
    for v in kat["vectors"]:
        ctr = [np.uint64(int(x, 16)) for x in v["counter"]]
        key = [int(x, 16) for x in v["key"]]
        out = DR.philox4x32(ctr, key)
        assert ["%08x" % int(w) for w in out] == v["out"]


@pytest.mark.parametrize("key,ctr", [((7, 9), (5, 0, 0, 0)), ((2**64 - 1, 3), (2**64 - 2, 1, 2, 3)),
                                     ((0x243F6A8885A308D3, 0x13198A2E03707344), (0, 0, 0, 0))])
def test_round_structure_matches_numpy_philox4x64(key, ctr):
    # numpy's Philox bit generator advances its 256-bit counter before every block of four
    # outputs: the first block of a generator set to counter c is Philox4x64-10(c + 1).
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                          counter=np.array(ctr, dtype=np.uint64))
    raw = [int(x) for x in bg.random_raw(8)]
    c = sum(int(w) << (64 * n) for n, w in enumerate(ctr))
    for blk in range(2):
        cn = (c + 1 + blk) % (1 << 256)
        words = [(cn >> (64 * n)) & ((1 << 64) - 1) for n in range(4)]
        assert list(DR.philox4x64(words, key)) == raw[4 * blk:4 * blk + 4]


def test_bytes_by_brute_force():
    seed, offset, bh = 0x1234567890ABCDEF, 3, 5
    u = DR.random_bytes(seed, offset, bh, 70, 90)
    g = np.random.default_rng(0)
    for _ in range(200):
        i, j = int(g.integers(70)), int(g.integers(90))
        rho = 16 * (i // 16) // 2 + i % 8
        kappa = 4 * (j // 32) + (j // 2) % 4
        words = DR.philox4x32([np.uint64(kappa), np.uint64(rho), np.uint64(bh), np.uint64(offset)],
                              (seed % 2**32, seed // 2**32))
        w = int(words[(j // 8) % 4])
        assert u[i, j] == (w >> (8 * (2 * ((i // 8) % 2) + j % 2))) & 0xFF


def test_bytes_do_not_depend_on_the_problem_size():
    big = DR.random_bytes(11, 0, 2, 200, 300)
    assert np.array_equal(DR.random_bytes(11, 0, 2, 37, 129), big[:37, :129])
    assert np.array_equal(DR.random_bytes(11, 0, 2, 1, 1), big[:1, :1])


def test_seed_offset_and_head_change_every_byte_stream():
    a = DR.random_bytes(1, 0, 0, 64, 64)
    for other in (DR.random_bytes(2, 0, 0, 64, 64), DR.random_bytes(1, 1, 0, 64, 64),
                  DR.random_bytes(1, 0, 1, 64, 64), DR.random_bytes(1 << 32, 0, 0, 64, 64)):
        assert (a == other).mean() < 0.02   # 1/256 expected


def test_bytes_are_uniform():
    u = DR.random_bytes(99, 0, 0, 1024, 1024).ravel()
    counts = np.bincount(u, minlength=256)
    expected = u.size / 256
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 255 + 8 * np.sqrt(2 * 255)   # 255 degrees of freedom, 8 sigma
    # neighbours inside one call (the two rows, adjacent keys) are not correlated
    v = DR.random_bytes(99, 0, 0, 256, 256).astype(np.float64)
    for a, b in ((v[0:8], v[8:16]), (v[:, 0::2], v[:, 1::2])):
        r = np.corrcoef(a.ravel(), b.ravel())[0, 1]
        assert abs(r) < 0.03


@pytest.mark.parametrize("t", [0, 1, 26, 128, 255])
def test_keep_fraction(t):
    z = DR.keep_drop_mask(5, 0, 0, 512, t)
    p_keep = 1 - t / 256
    sigma = np.sqrt(p_keep * (1 - p_keep) / z.size)
    assert abs(z.mean() - p_keep) <= 6 * sigma + 1e-12
    assert DR.keep_scale(t) == pytest.approx(1 / p_keep)


def test_threshold_range():
    with pytest.raises(ValueError):
        DR.keep_drop_mask(0, 0, 0, 4, 256)
    with pytest.raises(ValueError):
        DR.keep_drop_mask(0, 0, 0, 4, -1)


# ---------------------------------------------------------------- attention with dropout

def _inputs(n, d=4, dv=3, seed=5):
    g = np.random.default_rng(seed)
    return [g.standard_normal(s) for s in ((n, d), (n, d), (n, dv), (n, dv))]


def test_zero_threshold_is_the_plain_oracle():
    q, k, v, do = _inputs(23, 8, 8)
    for name, keep in _masks(23).items():
        z = DR.keep_drop_mask(1, 0, 0, 23, 0)
        assert z.all()
        o, lse, _ = DR.forward_head(q, k, v, 0.4, keep, z, 0)
        o0, lse0, _ = A.forward_head(q, k, v, 0.4, keep)
        assert np.array_equal(o, o0) and np.array_equal(lse, lse0), name
        for a, b in zip(DR.backward_head(q, k, v, do, 0.4, keep, z, 0),
                        A.backward_head(q, k, v, do, 0.4, keep)):
            np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14, err_msg=name)


def test_lse_does_not_depend_on_the_mask():
    q, k, v, _ = _inputs(40, 8, 8)
    keep = A.keep_mask(40, causal=True)
    _, lse0, _ = A.forward_head(q, k, v, 0.3, keep)
    for seed in (1, 2):
        z = DR.keep_drop_mask(seed, 0, 0, 40, 100)
        _, lse, _ = DR.forward_head(q, k, v, 0.3, keep, z, 100)
        assert np.array_equal(lse, lse0)


def test_expectation_over_masks_is_the_plain_output():
    # E[Z] = 1 - p, so E[O] = P V: averaging over many seeds converges to the plain O with
    # the standard error of the mean (the variance is computed from the exact P).
    n, t = 16, 64
    q, k, v, _ = _inputs(n, 4, 2, seed=7)
    keep = A.keep_mask(n, causal=True)
    o0, _, p = A.forward_head(q, k, v, 0.5, keep)
    seeds = 3000
    acc = np.zeros_like(o0)
    for s in range(seeds):
        z = DR.keep_drop_mask(s, 0, 0, n, t)
        acc += DR.forward_head(q, k, v, 0.5, keep, z, t)[0]
    mean = acc / seeds
    pk = 1 - t / 256
    var = (p * p) @ (v * v) * (1 - pk) / pk   # variance of one sample, per element
    se = np.sqrt(var / seeds) + 1e-15
    assert np.all(np.abs(mean - o0) <= 6 * se)


def _loss(q, k, v, do, scale, keep, z, t):
    return float((do * DR.forward_head(q, k, v, scale, keep, z, t)[0]).sum())


def _fd_error(backward_fn, keep, z, t, n=7, scale=0.6, h=1e-6):
    q, k, v, do = _inputs(n)
    grads = backward_fn(q, k, v, do, scale, keep, z, t)[:3]
    worst = 0.0
    for idx, x in enumerate((q, k, v)):
        num = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            args_p, args_m = [q, k, v], [q, k, v]
            xp, xm = x.copy(), x.copy()
            xp[pos] += h
            xm[pos] -= h
            args_p[idx], args_m[idx] = xp, xm
            num[pos] = (_loss(*args_p, do, scale, keep, z, t) -
                        _loss(*args_m, do, scale, keep, z, t)) / (2 * h)
        worst = max(worst, np.abs(grads[idx] - num).max() / max(np.abs(num).max(), 1e-30))
    return worst


@pytest.mark.parametrize("mode", ["dense", "causal", "padded", "block", "fully_masked_rows"])
@pytest.mark.parametrize("t", [64, 200])
def test_finite_differences(mode, t):
    n = 7
    keep = _masks(n)[mode]
    z = DR.keep_drop_mask(42, 0, 3, n, t)
    assert not z.all() and z.any()
    assert _fd_error(DR.backward_head, keep, z, t, n=n) < 1e-6


def test_D_two_ways_and_gradient_sums():
    n = 31
    q, k, v, do = _inputs(n, 6, 5, seed=9)
    for name, keep in _masks(n).items():
        z = DR.keep_drop_mask(8, 1, 0, n, 77)
        o, _, _ = DR.forward_head(q, k, v, 0.35, keep, z, 77)
        dq, dk, dv, D = DR.backward_head(q, k, v, do, 0.35, keep, z, 77)
        np.testing.assert_allclose(D, A.row_dot(do, o), rtol=1e-12, atol=1e-13, err_msg=name)
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12 * max(1, np.abs(dk).max()))
        live = keep.any(axis=1)
        assert np.all(dq[~live] == 0)


def test_batched_wrappers_match_heads():
    B, H, N, d = 2, 3, 20, 4
    g = np.random.default_rng(3)
    q, k, v, do = (g.standard_normal((B, H, N, d)) for _ in range(4))
    kv_len = np.array([9, 20])
    o, lse = DR.forward(q, k, v, 0.5, 90, seed=77, offset=2, kv_len=kv_len)
    dq, dk, dv, D = DR.backward(q, k, v, do, 0.5, 90, seed=77, offset=2, kv_len=kv_len)
    for b in range(B):
        for h in range(H):
            keep = A.keep_mask(N, kv_len=kv_len[b])
            z = DR.keep_drop_mask(77, 2, b * H + h, N, 90)
            ro, rl, _ = DR.forward_head(q[b, h], k[b, h], v[b, h], 0.5, keep, z, 90)
            assert np.array_equal(o[b, h], ro) and np.array_equal(lse[b, h], rl)
            for got, ref in zip((dq, dk, dv, D), DR.backward_head(q[b, h], k[b, h], v[b, h],
                                                                  do[b, h], 0.5, keep, z, 90)):
                assert np.array_equal(got[b, h], ref)


# A mistake planted in a copy of the backward must fail the finite-difference pin.
def _bwd_mask_missing_in_dP(q, k, v, do, scale, keep, z, t):
    _, _, p = DR.forward_head(q, k, v, scale, keep, z, t)
    ks = DR.keep_scale(t)
    dv = (p * z).T @ do * ks
    g = (do @ v.T) * ks               # planted: Z left out of dP
    D = (p * g).sum(axis=1)
    ds = p * (g - D[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), dv, D


def _bwd_unscaled_dV(q, k, v, do, scale, keep, z, t):
    dq, dk, dv, D = DR.backward_head(q, k, v, do, scale, keep, z, t)
    return dq, dk, dv / DR.keep_scale(t), D   # planted: 1 / (1 - p) left out of dV


@pytest.mark.parametrize("planted", [_bwd_mask_missing_in_dP, _bwd_unscaled_dV])
def test_planted_mistakes_fail_finite_differences(planted):
    keep = _masks(7)["causal"]
    z = DR.keep_drop_mask(42, 0, 3, 7, 64)
    assert _fd_error(planted, keep, z, 64, n=7) > 1e-3
