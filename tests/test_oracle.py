"""Pins for the CPU fp64 oracle: facts fixed by the pages and by mathematics.

Each pin is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong sign or index, a transposed operand) fails at least one of them; the
``test_planted_*`` cases plant such mistakes in copies of the oracle's
functions and check that the pins catch them.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import attention as A
from oracle.online_softmax import tiled_forward_head

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand(*shape, scale=1.0, seed=None):
    g = np.random.default_rng(seed) if seed is not None else rng
    return g.standard_normal(shape) * scale


def masks_for(n, seed=0):
    """(name, keep) pairs covering every mask mode, block size 2 for tiny n."""
    g = np.random.default_rng(seed)
    nb = (n + 1) // 2
    bm = (g.random((nb, nb)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    bm_hole = bm.copy()
    bm_hole[0, :] = 0  # rows 0..1 see no key at all
    return [
        ("dense", A.keep_mask(n)),
        ("causal", A.keep_mask(n, causal=True)),
        ("padded", A.keep_mask(n, kv_len=max(1, n - 2))),
        ("block", A.keep_mask(n, blockmask=bm, block=2)),
        ("block_causal", A.keep_mask(n, causal=True, blockmask=bm, block=2)),
        ("fully_masked_rows", A.keep_mask(n, blockmask=bm_hole, block=2)),
    ]


# ---------------------------------------------------------------- forward pins

@pytest.mark.parametrize("n", [1, 7, 37])
def test_rows_of_P_sum_to_one(n):
    q, k, v = rand(n, 8), rand(n, 8), rand(n, 5)
    for name, keep in masks_for(n):
        _, lse, p = A.forward_head(q, k, v, 0.3, keep)
        live = keep.any(axis=1)
        assert np.all(np.abs(p[live].sum(axis=1) - 1.0) < 1e-12), name
        assert np.all(p[~live] == 0.0), name
        assert np.all(p[~keep] == 0.0), name
        assert np.all(np.isneginf(lse[~live])), name


def test_identical_keys_give_mean_of_values():
    n, d = 23, 6
    q = rand(n, d)
    k = np.tile(rand(1, d), (n, 1))
    v = rand(n, 4)
    o, _, _ = A.forward_head(q, k, v, 0.5, A.keep_mask(n))
    np.testing.assert_allclose(o, np.tile(v.mean(axis=0), (n, 1)), rtol=0, atol=1e-13)
    o, _, _ = A.forward_head(q, k, v, 0.5, A.keep_mask(n, kv_len=9))
    np.testing.assert_allclose(o, np.tile(v[:9].mean(axis=0), (n, 1)), rtol=0, atol=1e-13)
    o, _, _ = A.forward_head(q, k, v, 0.5, A.keep_mask(n, causal=True))
    cum = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o, cum, rtol=0, atol=1e-13)


def test_zero_queries_are_uniform_with_log_count_lse():
    n, d = 19, 4
    q = np.zeros((n, d))
    k, v = rand(n, d), rand(n, 3)
    o, lse, _ = A.forward_head(q, k, v, 1.0, A.keep_mask(n, causal=True))
    counts = np.arange(1, n + 1)
    np.testing.assert_allclose(lse, np.log(counts), rtol=0, atol=1e-14)
    np.testing.assert_allclose(o, np.cumsum(v, axis=0) / counts[:, None], atol=1e-13)


def test_single_token_closed_form():
    q, k, v, do = rand(1, 4), rand(1, 4), rand(1, 3), rand(1, 3)
    keep = A.keep_mask(1)
    o, lse, _ = A.forward_head(q, k, v, 0.7, keep)
    np.testing.assert_array_equal(o, v)
    assert lse[0] == pytest.approx(0.7 * float(q[0] @ k[0]), abs=1e-15)
    dq, dk, dv, _ = A.backward_head(q, k, v, do, 0.7, keep)
    np.testing.assert_array_equal(dv, do)
    assert np.all(dq == 0) and np.all(dk == 0)


def test_lse_matches_scipy_logsumexp():
    n = 41
    q, k, v = rand(n, 16, scale=3.0), rand(n, 16), rand(n, 2)
    for name, keep in masks_for(n):
        _, lse, _ = A.forward_head(q, k, v, 0.25, keep)
        s = 0.25 * (q @ k.T)
        ref = scipy.special.logsumexp(np.where(keep, s, -np.inf), axis=1)
        live = keep.any(axis=1)
        np.testing.assert_allclose(lse[live], ref[live], rtol=1e-14, atol=1e-13, err_msg=name)
        assert np.all(np.isneginf(lse[~live]) & np.isneginf(ref[~live]))


def test_two_key_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "two_key_example.json")))
    q, k, v, do = (np.array(g[x]) for x in ("q", "k", "v", "do"))
    for case, causal in (("non_causal", False), ("causal", True)):
        exp = g[case]
        keep = A.keep_mask(2, causal=causal)
        o, lse, _ = A.forward_head(q, k, v, g["scale"], keep)
        dq, dk, dv, _ = A.backward_head(q, k, v, do, g["scale"], keep)
        np.testing.assert_allclose(o, exp["o"], atol=1e-14)
        np.testing.assert_allclose(lse, exp["lse"], atol=1e-14)
        np.testing.assert_allclose(dq, exp["dq"], atol=1e-14)
        np.testing.assert_allclose(dk, exp["dk"], atol=1e-14)
        np.testing.assert_allclose(dv, exp["dv"], atol=1e-14)


def test_shift_of_keys_leaves_outputs_and_gradients_unchanged():
    # Adding c to every key adds scale*q_i.c to the whole row i of S: the
    # softmax is unchanged, hence O, dV, dK; rows of dS sum to zero, hence dQ.
    n, d = 17, 5
    q, k, v, do = rand(n, d), rand(n, d), rand(n, 3), rand(n, 3)
    c = rand(1, d, scale=4.0)
    for name, keep in masks_for(n):
        o1, lse1, _ = A.forward_head(q, k, v, 0.4, keep)
        o2, lse2, _ = A.forward_head(q, k + c, v, 0.4, keep)
        np.testing.assert_allclose(o1, o2, atol=1e-12, err_msg=name)
        live = keep.any(axis=1)
        np.testing.assert_allclose(lse2[live] - lse1[live], 0.4 * (q @ c.T)[live, 0], atol=1e-12)
        g1 = A.backward_head(q, k, v, do, 0.4, keep)
        g2 = A.backward_head(q, k + c, v, do, 0.4, keep)
        for a, b in zip(g1[:3], g2[:3]):
            np.testing.assert_allclose(a, b, atol=1e-11, err_msg=name)


# --------------------------------------------------------------- backward pins

def loss(q, k, v, do, scale, keep):
    o, _, _ = A.forward_head(q, k, v, scale, keep)
    return float((do * o).sum())


def fd_max_rel_error(backward_fn, n=7, d=4, dv_=3, seed=5, keep=None, scale=0.6, h=1e-6):
    g = np.random.default_rng(seed)
    q, k, v, do = (g.standard_normal(s) for s in ((n, d), (n, d), (n, dv_), (n, dv_)))
    keep = A.keep_mask(n) if keep is None else keep
    grads = backward_fn(q, k, v, do, scale, keep)[:3]
    worst = 0.0
    for idx, x in enumerate((q, k, v)):
        num = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[pos] += h
            xm[pos] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[idx] = xp
            args_m[idx] = xm
            num[pos] = (loss(*args_p, do, scale, keep) - loss(*args_m, do, scale, keep)) / (2 * h)
        denom = max(np.abs(num).max(), 1e-30)
        worst = max(worst, np.abs(grads[idx] - num).max() / denom)
    return worst


@pytest.mark.parametrize("mode", ["dense", "causal", "padded", "block", "block_causal",
                                  "fully_masked_rows"])
def test_finite_differences(mode):
    n = 7
    keep = dict(masks_for(n))[mode]
    assert fd_max_rel_error(A.backward_head, n=n, keep=keep) < 1e-6


def test_gradient_sums():
    n, d = 29, 6
    q, k, v, do = rand(n, d), rand(n, d), rand(n, 4), rand(n, 4)
    for name, keep in masks_for(n):
        dq, dk, dv, _ = A.backward_head(q, k, v, do, 0.35, keep)
        live = keep.any(axis=1)
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12 * max(1, np.abs(dk).max()))
        np.testing.assert_allclose(dv.sum(axis=0), do[live].sum(axis=0), rtol=1e-9, atol=1e-12)
        assert np.all(dq[~live] == 0)


def test_D_two_ways():
    n = 33
    q, k, v, do = rand(n, 8), rand(n, 8), rand(n, 8), rand(n, 8)
    for name, keep in masks_for(n):
        o, _, _ = A.forward_head(q, k, v, 0.3, keep)
        _, _, _, D = A.backward_head(q, k, v, do, 0.3, keep)
        np.testing.assert_allclose(D, A.row_dot(do, o), rtol=1e-12, atol=1e-13, err_msg=name)


def test_batched_wrappers_match_heads():
    B, H, N, d = 2, 3, 9, 4
    q, k, v, do = rand(B, H, N, d), rand(B, H, N, d), rand(B, H, N, d), rand(B, H, N, d)
    kv_len = np.array([4, 9])
    o, lse = A.forward(q, k, v, 0.5, causal=True, kv_len=kv_len)
    dq, dk, dv, D = A.backward(q, k, v, do, 0.5, causal=True, kv_len=kv_len)
    for b in range(B):
        for h in range(H):
            keep = A.keep_mask(N, causal=True, kv_len=kv_len[b])
            o1, l1, _ = A.forward_head(q[b, h], k[b, h], v[b, h], 0.5, keep)
            np.testing.assert_array_equal(o[b, h], o1)
            np.testing.assert_array_equal(lse[b, h], l1)
            g = A.backward_head(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, keep)
            np.testing.assert_array_equal(dk[b, h], g[1])
    sub_o, _ = A.forward(q, k, v, 0.5, heads=[(1, 2)])
    assert np.isnan(sub_o[0, 0]).all() and np.isfinite(sub_o[1, 2]).all()


def test_block_mask_indexing_explicit_matrix():
    # A 4 x 4 block mask over 2 x 2 blocks, written out element by element: the mask entry
    # [row block, column block] decides the query-row x key-column square it covers (a
    # transposed or shifted lookup fails here).
    bm = np.array([[1, 0, 0, 1],
                   [0, 1, 1, 0],
                   [1, 1, 0, 0],
                   [0, 0, 1, 1]], dtype=np.uint8)
    expected = np.array([
        [1, 1, 0, 0, 0, 0, 1, 1],
        [1, 1, 0, 0, 0, 0, 1, 1],
        [0, 0, 1, 1, 1, 1, 0, 0],
        [0, 0, 1, 1, 1, 1, 0, 0],
        [1, 1, 1, 1, 0, 0, 0, 0],
        [1, 1, 1, 1, 0, 0, 0, 0],
        [0, 0, 0, 0, 1, 1, 1, 1],
        [0, 0, 0, 0, 1, 1, 1, 1]], dtype=bool)
    np.testing.assert_array_equal(A.keep_mask(8, blockmask=bm, block=2), expected)
    # Ragged last block (n = 7): the last row and column of the mask cover one element.
    np.testing.assert_array_equal(A.keep_mask(7, blockmask=bm, block=2), expected[:7, :7])
    # Combined with the causal mask and a key length: the intersection, element by element.
    both = A.keep_mask(8, causal=True, blockmask=bm, kv_len=5, block=2)
    expected_both = np.array([
        [1, 0, 0, 0, 0, 0, 0, 0],
        [1, 1, 0, 0, 0, 0, 0, 0],
        [0, 0, 1, 0, 0, 0, 0, 0],
        [0, 0, 1, 1, 0, 0, 0, 0],
        [1, 1, 1, 1, 0, 0, 0, 0],
        [1, 1, 1, 1, 0, 0, 0, 0],
        [0, 0, 0, 0, 1, 0, 0, 0],
        [0, 0, 0, 0, 1, 0, 0, 0]], dtype=bool)
    np.testing.assert_array_equal(both, expected_both)
    # The default block is the pages' 128 x 128: one mask entry covers 128 x 128 pairs.
    bm2 = np.array([[1, 0], [1, 1]], dtype=np.uint8)
    keep = A.keep_mask(200, blockmask=bm2)
    assert keep[:128, :128].all() and not keep[:128, 128:].any()
    assert keep[128:, :].all()


# -------------------------------------------- independent online-softmax reference

@pytest.mark.parametrize("br,bc", [(1, 1), (16, 32), (128, 128), (None, None)])
def test_online_softmax_matches_direct_computation(br, bc):
    n, d = 150, 16
    q, k, v = rand(n, d, seed=3), rand(n, d, seed=4), rand(n, d, seed=5)
    br = br or n
    bc = bc or n
    for name, keep in [("dense", A.keep_mask(n)), ("causal", A.keep_mask(n, causal=True)),
                       ("padded", A.keep_mask(n, kv_len=97))]:
        o_ref, lse_ref, _ = A.forward_head(q, k, v, 0.25, keep)
        o, lse = tiled_forward_head(q, k, v, 0.25, keep, br, bc)
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12, err_msg=name)
        np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12, err_msg=name)


def test_online_softmax_block_size_does_not_matter():
    n, d = 70, 8
    q, k, v = rand(n, d, seed=6), rand(n, d, seed=7), rand(n, d, seed=8)
    keep = A.keep_mask(n, causal=True)
    outs = [tiled_forward_head(q, k, v, 0.5, keep, br, bc)[0]
            for br, bc in [(1, 1), (3, 5), (16, 32), (70, 70), (64, 1)]]
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-12)


def test_online_softmax_handles_large_logits():
    n, d = 40, 4
    q = rand(n, d, seed=9, scale=100.0)
    k = rand(n, d, seed=10, scale=100.0)  # |logits| up to ~1e4 and beyond
    v = rand(n, d, seed=11)
    for keep in (A.keep_mask(n), A.keep_mask(n, causal=True)):
        o, lse = tiled_forward_head(q, k, v, 1.0, keep, 8, 8)
        o_ref, lse_ref, _ = A.forward_head(q, k, v, 1.0, keep)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        assert np.all(np.isfinite(o_ref))
        assert np.abs(lse).max() > 1e3
        np.testing.assert_allclose(o, o_ref, atol=1e-9)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)


def test_fully_masked_blocks_and_rows_give_no_nan():
    n = 12
    q, k, v, do = rand(n, 4), rand(n, 4), rand(n, 4), rand(n, 4)
    keep = dict(masks_for(n))["fully_masked_rows"]
    dead = ~keep.any(axis=1)
    assert dead.any()
    o, lse = tiled_forward_head(q, k, v, 1.0, keep, 2, 2)
    o_ref, lse_ref, _ = A.forward_head(q, k, v, 1.0, keep)
    assert not np.isnan(o).any() and not np.isnan(o_ref).any()
    assert np.all(o[dead] == 0) and np.all(o_ref[dead] == 0)
    assert np.all(np.isneginf(lse[dead])) and np.all(np.isneginf(lse_ref[dead]))
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    dq, dk, dv, D = A.backward_head(q, k, v, do, 1.0, keep)
    for g in (dq, dk, dv, D):
        assert not np.isnan(g).any()
    assert np.all(dq[dead] == 0)


# --------------------------------------------------- library cross-check (optional)

def test_against_torch_sdpa_float64():
    torch = pytest.importorskip("torch")
    n, d = 33, 8
    q, k, v, do = rand(n, d), rand(n, d), rand(n, d), rand(n, d)
    for name, keep in masks_for(n)[:5]:
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(
            tq[None, None], tk[None, None], tv[None, None],
            attn_mask=torch.tensor(keep)[None, None], scale=0.3)[0, 0]
        out.backward(torch.tensor(do))
        o, _, _ = A.forward_head(q, k, v, 0.3, keep)
        dq, dk, dv, _ = A.backward_head(q, k, v, do, 0.3, keep)
        np.testing.assert_allclose(out.detach().numpy(), o, atol=1e-12, err_msg=name)
        np.testing.assert_allclose(tq.grad.numpy(), dq, atol=1e-11, err_msg=name)
        np.testing.assert_allclose(tk.grad.numpy(), dk, atol=1e-11, err_msg=name)
        np.testing.assert_allclose(tv.grad.numpy(), dv, atol=1e-11, err_msg=name)


# ------------------------------------------------------- planted mistakes are caught

def _bwd_transposed_dk(q, k, v, do, scale, keep):
    dq, dk, dv, D = A.backward_head(q, k, v, do, scale, keep)
    _, _, p = A.forward_head(q, k, v, scale, keep)
    dp = do @ v.T
    ds = p * (dp - (p * dp).sum(1)[:, None])
    return dq, scale * (ds @ q), dv, D            # should be ds.T @ q


def _bwd_dropped_D(q, k, v, do, scale, keep):
    _, _, p = A.forward_head(q, k, v, scale, keep)
    dp = do @ v.T
    ds = p * dp                                    # should be p * (dp - D)
    return scale * ds @ k, scale * ds.T @ q, p.T @ do, None


def _bwd_flipped_sign(q, k, v, do, scale, keep):
    _, _, p = A.forward_head(q, k, v, scale, keep)
    dp = do @ v.T
    ds = p * ((p * dp).sum(1)[:, None] - dp)      # sign flipped
    return scale * ds @ k, scale * ds.T @ q, p.T @ do, None


def _bwd_missing_scale(q, k, v, do, scale, keep):
    dq, dk, dv, D = A.backward_head(q, k, v, do, scale, keep)
    return dq, dk / scale, dv, D                   # dK without the 1/sqrt(d) factor


@pytest.mark.parametrize("planted", [_bwd_transposed_dk, _bwd_dropped_D, _bwd_flipped_sign, _bwd_missing_scale])
def test_planted_backward_mistakes_fail_finite_differences(planted):
    keep = A.keep_mask(7, causal=True)
    assert fd_max_rel_error(A.backward_head, keep=keep, dv_=4) < 1e-6
    assert fd_max_rel_error(planted, keep=keep, dv_=4) > 1e-2


def test_planted_forward_mistakes_fail_pins():
    n = 11
    q, k, v = rand(n, 4), rand(n, 4), rand(n, 4)
    keep = A.keep_mask(n)
    s = A.scores(q, k, 1.0, keep)
    # Forgetting to subtract the row max is harmless for small logits, but a
    # missing normalisation breaks the row-sum pin, and a transposed score
    # matrix breaks agreement with scipy's logsumexp.
    p_unnorm = np.exp(s - s.max(1, keepdims=True))
    assert np.abs(p_unnorm.sum(1) - 1).max() > 1e-3
    _, lse_t = A.softmax_rows(s.T)
    ref = scipy.special.logsumexp(s, axis=1)
    assert np.abs(lse_t - ref).max() > 1e-3
