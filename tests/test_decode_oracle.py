"""Pins of the decode oracle (CPU): each check reaches the result by another route."""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(7)


def _rand(*shape):
    return RNG.standard_normal(shape)


def test_last_token_equals_the_causal_forward_row():
    # Token t with a cache of t + 1 keys is row t of causal attention over the sequence.
    B, H, N, d = 2, 3, 9, 8
    q, k, v = _rand(B, H, N, d), _rand(B, H, N, d), _rand(B, H, N, d)
    scale = 0.37
    o_full, lse_full = oracle.forward(q, k, v, scale, causal=True)
    for t in (0, 4, N - 1):
        cache_len = np.full(B, t + 1)
        o, lse = oracle.decode(q[:, :, t], k, v, scale, cache_len)
        np.testing.assert_allclose(o, o_full[:, :, t], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, lse_full[:, :, t], rtol=1e-12, atol=1e-12)


def test_grouped_heads_equal_repeated_key_value_heads():
    # Query head h reads K/V head h // G: repeating each K/V head G times must not change
    # anything (a wrong grouping such as h % Hkv fails this).
    B, Hq, Hkv, L, d = 2, 8, 2, 13, 4
    q, k, v = _rand(B, Hq, d), _rand(B, Hkv, L, d), _rand(B, Hkv, L, d)
    cache_len = np.array([13, 6])
    o, lse = oracle.decode(q, k, v, 0.5, cache_len)
    G = Hq // Hkv
    k_rep, v_rep = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    o2, lse2 = oracle.decode(q, k_rep, v_rep, 0.5, cache_len)
    np.testing.assert_allclose(o, o2, rtol=0, atol=0)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=0)
    # and each group really reads its own K/V head
    o_h0 = oracle.decode(q[:, :1], k[:, :1], v[:, :1], 0.5, cache_len)[0]
    o_h7 = oracle.decode(q[:, 7:], k[:, 1:], v[:, 1:], 0.5, cache_len)[0]
    np.testing.assert_allclose(o[:, 0], o_h0[:, 0], rtol=0, atol=0)
    np.testing.assert_allclose(o[:, 7], o_h7[:, 0], rtol=0, atol=0)


def test_identical_keys_give_the_mean_of_the_visible_values():
    B, Hq, Hkv, L, d = 1, 2, 1, 11, 5
    q = _rand(B, Hq, d)
    k = np.broadcast_to(_rand(1, 1, 1, d), (B, Hkv, L, d)).copy()
    v = _rand(B, Hkv, L, d)
    cache_len = np.array([7])
    o, lse = oracle.decode(q, k, v, 0.3, cache_len)
    np.testing.assert_allclose(o[0, 0], v[0, 0, :7].mean(axis=0), rtol=1e-12, atol=1e-12)
    s = 0.3 * q[0, 1] @ k[0, 0, 0]
    np.testing.assert_allclose(lse[0, 1], s + np.log(7), rtol=1e-12)


def test_one_key_cache_closed_form():
    B, Hq, Hkv, L, d = 2, 4, 2, 5, 3
    q, k, v = _rand(B, Hq, d), _rand(B, Hkv, L, d), _rand(B, Hkv, L, d)
    o, lse = oracle.decode(q, k, v, 0.7, np.array([1, 1]))
    for b in range(B):
        for h in range(Hq):
            g = h // 2
            np.testing.assert_allclose(o[b, h], v[b, g, 0], rtol=1e-12)
            np.testing.assert_allclose(lse[b, h], 0.7 * q[b, h] @ k[b, g, 0], rtol=1e-12)


def test_lse_matches_scipy_logsumexp():
    special = pytest.importorskip("scipy.special")
    B, Hq, Hkv, L, d = 3, 6, 3, 17, 8
    q, k, v = _rand(B, Hq, d), _rand(B, Hkv, L, d), _rand(B, Hkv, L, d)
    cache_len = np.array([17, 9, 2])
    _, lse = oracle.decode(q, k, v, 0.25, cache_len)
    for b in range(B):
        for h in range(Hq):
            s = 0.25 * k[b, h // 2, :cache_len[b]] @ q[b, h]
            assert abs(lse[b, h] - special.logsumexp(s)) < 1e-12


def test_rows_past_the_cache_length_do_not_matter():
    B, Hq, Hkv, L, d = 1, 2, 1, 6, 3
    q, k, v = _rand(B, Hq, d), _rand(B, Hkv, L, d), _rand(B, Hkv, L, d)
    o, lse = oracle.decode(q, k, v, 0.5, np.array([4]))
    k[:, :, 4:] = np.nan
    v[:, :, 4:] = np.inf
    o2, lse2 = oracle.decode(q, k, v, 0.5, np.array([4]))
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    o0, lse0 = oracle.decode(q, k, v, 0.5, np.array([0]))
    assert np.all(o0 == 0) and np.all(np.isneginf(lse0))
