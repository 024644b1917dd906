"""CPU fp64 oracle: exact scaled-dot-product attention by its plain definition.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the package's ``smoke()`` check and the
``cpu_baseline`` leg of the benchmark use it.  It shares no code with the CUDA
path and imports nothing from the package.

What it computes, one (batch, head) at a time, in float64, materialising the
full N x N score and probability matrices (the "standard attention" that the
pages set against FlashAttention):

* Forward -- "How FlashAttention works for training" (aivaro.ru answer 474),
  section 1: Attention(Q, K, V) = softmax(Q K^T / sqrt(d)) V; FlashAttention
  reading guide (arXiv 2205.14135), "Problem": S = Q K^T, P = softmax(S),
  O = P V.  The softmax is the safe form of the reading guide, "Method",
  step 2: subtract the row maximum before exponentiating.
* Saved statistic -- course week 13, step 2: the forward keeps only the output
  and the per-row logsumexp, lse_i = m_i + ln(l_i) (natural log).
* Masking -- course week 13, step 2 (causal: key j is visible to query i
  only when j <= i) and the reading guide's "Extension: block-sparse
  FlashAttention" (a 0/1 mask over 128 x 128 blocks; a 0 block is left out).
  Key padding: key j of sequence b is visible only when j < kv_len[b].
  Masked scores are -inf.  A row with no visible key has O = 0, lse = -inf
  and contributes no gradient.
* Backward -- the chain rule through O = P V and P = softmax(S).  The answer
  page's section 3 prints the gradient formulas garbled; only dV = P^T dO is
  right there.  The textbook softmax-Jacobian form is used instead:
      dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,
      dS = P o (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.
  D is also available as rowsum(dO o O) (``row_dot``), which is equal because
  rows of P sum to one and O = P V.

Pins (checked by the CPU tests, not by this file): rows of P sum to one,
identical keys give the mean of V, Q = 0 gives uniform weights with
lse = ln(#visible keys), N = 1 closed form, lse against scipy's logsumexp,
central finite differences of L = sum(dO o O), gradient sums
(sum_j dK_j = 0, sum_j dV_j = sum of dO over rows with a visible key), shift
invariance, a hand-derived two-key example, agreement with the independent
block-by-block online-softmax reference in ``online_softmax.py``.
"""
from __future__ import annotations

import numpy as np

BLOCK = 128


def keep_mask(n: int, causal: bool = False, blockmask=None, kv_len=None,
              block: int = BLOCK) -> np.ndarray:
    """Boolean [n, n]: True where query row i may attend key column j."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    keep = np.ones((n, n), dtype=bool)
    if causal:
        keep &= j <= i
    if kv_len is not None:
        keep &= j < int(kv_len)
    if blockmask is not None:
        bm = np.asarray(blockmask).astype(bool)
        keep &= bm[i // block, j // block]
    return keep


def scores(q: np.ndarray, k: np.ndarray, scale: float, keep: np.ndarray) -> np.ndarray:
    """S = scale * Q K^T with masked entries set to -inf."""
    s = scale * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)
    return np.where(keep, s, -np.inf)


def softmax_rows(s: np.ndarray):
    """Safe softmax of each row of S.

    Returns (P, lse).  Rows that are entirely -inf get P = 0 and lse = -inf.
    """
    m = s.max(axis=1)
    live = np.isfinite(m)
    p = np.zeros_like(s)
    p[live] = np.exp(s[live] - m[live, None])
    l = p.sum(axis=1)
    p[live] /= l[live, None]
    lse = np.full(s.shape[0], -np.inf)
    lse[live] = m[live] + np.log(l[live])
    return p, lse


def forward_head(q, k, v, scale: float, keep: np.ndarray):
    """One head: returns (O [n, d], lse [n], P [n, n])."""
    s = scores(q, k, scale, keep)
    p, lse = softmax_rows(s)
    o = p @ np.asarray(v, np.float64)
    return o, lse, p


def row_dot(do, o) -> np.ndarray:
    """D_i = sum_c dO_ic * O_ic."""
    return (np.asarray(do, np.float64) * np.asarray(o, np.float64)).sum(axis=1)


def backward_head(q, k, v, do, scale: float, keep: np.ndarray):
    """One head: returns (dQ, dK, dV, D) for the loss L = sum(dO o O)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    _, _, p = forward_head(q, k, v, scale, keep)
    dv = p.T @ do
    dp = do @ v.T
    D = (p * dp).sum(axis=1)
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, D


def _head_keep(n, causal, blockmask, kv_len, b):
    return keep_mask(n, causal, blockmask, None if kv_len is None else kv_len[b])


def forward(q, k, v, scale: float, causal: bool = False, blockmask=None, kv_len=None,
            heads=None):
    """All heads of [B, H, N, d] inputs.  Returns (O, lse) in float64.

    ``heads`` optionally restricts the work to a list of (b, h) pairs; other
    heads of the result are left as NaN.
    """
    q = np.asarray(q, np.float64)
    B, H, N, d = q.shape
    o = np.full((B, H, N, v.shape[-1]), np.nan)
    lse = np.full((B, H, N), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        keep = _head_keep(N, causal, blockmask, kv_len, b)
        o[b, h], lse[b, h], _ = forward_head(q[b, h], k[b, h], v[b, h], scale, keep)
    return o, lse


def backward(q, k, v, do, scale: float, causal: bool = False, blockmask=None, kv_len=None,
             heads=None):
    """All heads: returns (dQ, dK, dV, D) in float64 (NaN outside ``heads``)."""
    q = np.asarray(q, np.float64)
    B, H, N, d = q.shape
    dq = np.full(q.shape, np.nan)
    dk = np.full(q.shape, np.nan)
    dv = np.full((B, H, N, v.shape[-1]), np.nan)
    D = np.full((B, H, N), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        keep = _head_keep(N, causal, blockmask, kv_len, b)
        dq[b, h], dk[b, h], dv[b, h], D[b, h] = backward_head(
            q[b, h], k[b, h], v[b, h], do[b, h], scale, keep)
    return dq, dk, dv, D
