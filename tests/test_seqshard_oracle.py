"""Pins of the sequence-sharded oracle (``oracle/seqshard.py``) on the CPU.

The merge of per-shard partial results must give the attention over all keys (the
reading guide's merge rule applied to (O, lse) pairs), and the per-shard backward with
the merged statistics must sum to the full backward.  Both are checked against the plain
oracle, which is pinned on its own in ``test_oracle.py``.
"""
import numpy as np
import pytest

from oracle import attention as A
from oracle import seqshard as SS


def rand(*shape, seed=0, scale=1.0):
    return scale * np.random.default_rng(seed).standard_normal(shape)


def _chunks(n, parts):
    edges = np.linspace(0, n, parts + 1).astype(int)
    return [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:])]


def _masks(n):
    return {"dense": A.keep_mask(n), "causal": A.keep_mask(n, causal=True),
            "padded": A.keep_mask(n, kv_len=n // 3),
            "block": A.keep_mask(n, blockmask=np.array([[1, 0], [1, 1]]), block=(n + 1) // 2)}


@pytest.mark.parametrize("parts", [1, 2, 3, 5])
@pytest.mark.parametrize("mode", ["dense", "causal", "padded", "block"])
def test_merged_partials_equal_the_full_forward(parts, mode):
    n, d = 23, 5
    q, k, v = rand(n, d, seed=1), rand(n, d, seed=2), rand(n, d, seed=3)
    keep = _masks(n)[mode]
    o_ref, lse_ref, _ = A.forward_head(q, k, v, 0.4, keep)
    os_, ls_ = [], []
    for a, b in _chunks(n, parts):
        o_k, lse_k, _ = A.forward_head(q, k[a:b], v[a:b], 0.4, keep[:, a:b])
        os_.append(o_k)
        ls_.append(lse_k)
    o, lse = SS.merge_partials(os_, ls_)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    dead = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), dead)
    np.testing.assert_allclose(lse[~dead], lse_ref[~dead], atol=1e-12)
    assert np.all(o[dead] == 0)


def test_merge_closed_forms():
    a, b = rand(4, 3, seed=4), rand(4, 3, seed=5)
    # part 1: one key (l = 1 at m = 0) -> lse = 0; part 2: l = 3 at m = 0 -> lse = ln 3.
    o, lse = SS.merge_partials([a, b], [np.zeros(4), np.full(4, np.log(3.0))])
    np.testing.assert_allclose(o, (a + 3 * b) / 4, atol=1e-15)
    np.testing.assert_allclose(lse, np.full(4, np.log(4.0)), atol=1e-15)
    # a single part is returned unchanged
    o1, l1 = SS.merge_partials([a], [np.array([0.5, -2.0, 7.0, 1e4])])
    np.testing.assert_array_equal(o1, a)
    np.testing.assert_allclose(l1, [0.5, -2.0, 7.0, 1e4])
    # a part with no visible key (lse = -inf) has weight 0; all parts empty -> O = 0, -inf
    o2, l2 = SS.merge_partials([a, b], [np.zeros(4), np.full(4, -np.inf)])
    np.testing.assert_array_equal(o2, a)
    np.testing.assert_array_equal(l2, np.zeros(4))
    o3, l3 = SS.merge_partials([a, b], [np.full(4, -np.inf)] * 2)
    assert np.all(o3 == 0) and np.all(np.isneginf(l3))
    # large logsumexps do not overflow
    o4, l4 = SS.merge_partials([a, b], [np.full(4, 1e4), np.full(4, 1e4 + np.log(3.0))])
    np.testing.assert_allclose(o4, (a + 3 * b) / 4, atol=1e-12)
    np.testing.assert_allclose(l4, 1e4 + np.log(4.0), rtol=1e-15)


def test_merge_does_not_depend_on_the_order_of_parts():
    os_ = [rand(6, 4, seed=10 + i) for i in range(4)]
    ls_ = [rand(6, seed=20 + i, scale=5.0) for i in range(4)]
    ls_[2][1] = -np.inf
    o, lse = SS.merge_partials(os_, ls_)
    perm = [2, 0, 3, 1]
    o_p, lse_p = SS.merge_partials([os_[i] for i in perm], [ls_[i] for i in perm])
    np.testing.assert_allclose(o_p, o, atol=1e-14)
    np.testing.assert_allclose(lse_p, lse, atol=1e-14)


@pytest.mark.parametrize("parts", [1, 2, 4])
@pytest.mark.parametrize("mode", ["dense", "causal", "padded", "block"])
def test_shard_backwards_sum_to_the_full_backward(parts, mode):
    n, d = 19, 4
    q, k, v, do = (rand(n, d, seed=s) for s in (30, 31, 32, 33))
    keep = _masks(n)[mode]
    dq_ref, dk_ref, dv_ref, _ = A.backward_head(q, k, v, do, 0.7, keep)
    o, lse, _ = A.forward_head(q, k, v, 0.7, keep)
    D = A.row_dot(do, o)
    dq = np.zeros_like(q)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    for a, b in _chunks(n, parts):
        gq, gk, gv = SS.backward_head_with_stats(q, k[a:b], v[a:b], do, lse, D, 0.7,
                                                 keep[:, a:b])
        dq += gq
        dk[a:b], dv[a:b] = gk, gv
    np.testing.assert_allclose(dq, dq_ref, atol=1e-12)
    np.testing.assert_allclose(dk, dk_ref, atol=1e-12)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-12)


def test_query_shards_of_a_key_shard_sum_to_its_gradient():
    # dK, dV of one key shard summed over query shards (each with its own rows' lse, D).
    n, d = 16, 3
    q, k, v, do = (rand(n, d, seed=s) for s in (40, 41, 42, 43))
    keep = A.keep_mask(n, causal=True)
    _, dk_ref, dv_ref, _ = A.backward_head(q, k, v, do, 0.5, keep)
    o, lse, _ = A.forward_head(q, k, v, 0.5, keep)
    D = A.row_dot(do, o)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    for qa, qb in _chunks(n, 4):
        for ka, kb in _chunks(n, 4):
            _, gk, gv = SS.backward_head_with_stats(q[qa:qb], k[ka:kb], v[ka:kb], do[qa:qb],
                                                    lse[qa:qb], D[qa:qb], 0.5,
                                                    keep[qa:qb, ka:kb])
            dk[ka:kb] += gk
            dv[ka:kb] += gv
    np.testing.assert_allclose(dk, dk_ref, atol=1e-12)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-12)


def test_shard_local_statistics_would_be_wrong():
    # Planted mistake: renormalising P within a shard (its own lse) instead of using the
    # merged lse.  The sum over shards then differs from the full backward.
    n, d = 12, 3
    q, k, v, do = (rand(n, d, seed=s) for s in (50, 51, 52, 53))
    keep = A.keep_mask(n)
    dq_ref, _, _, _ = A.backward_head(q, k, v, do, 0.5, keep)
    o, lse, _ = A.forward_head(q, k, v, 0.5, keep)
    D = A.row_dot(do, o)
    dq = np.zeros_like(q)
    for a, b in _chunks(n, 2):
        _, lse_local, _ = A.forward_head(q, k[a:b], v[a:b], 0.5, keep[:, a:b])
        dq += SS.backward_head_with_stats(q, k[a:b], v[a:b], do, lse_local, D, 0.5,
                                          keep[:, a:b])[0]
    assert np.abs(dq - dq_ref).max() > 1e-3
