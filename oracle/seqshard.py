"""CPU fp64 oracle of attention split over key/value shards (sequence sharding).

TEST INFRASTRUCTURE ONLY (same rule as ``attention.py``): used by the tests, never by
the product path.

The FlashAttention reading guide (arXiv 2205.14135), "Method", merges the softmax
statistics of a vector split into parts: with m_k the maximum and l_k the sum of
exponentials of part k, the whole has m = max_k m_k and l = sum_k e^{m_k - m} l_k.  Its
"Limitations" names attention over several GPUs as open work; splitting the keys and
values of one sequence over shards is that setting.  Each shard k gives a normalised
partial output O_k = softmax(S_k) V_k over its own keys and the partial logsumexp
lse_k = m_k + ln l_k.  Since l_k e^{m_k} = e^{lse_k}, the merge rule reads, per row,

    lse = ln sum_k e^{lse_k},        O = sum_k e^{lse_k - lse} O_k,

which is the exact attention over the union of the keys (the weights e^{lse_k - lse} are
the shares l_k e^{m_k - m} / l of each part).  A part with lse_k = -inf (no visible key)
has weight 0; a row with no visible key in any part has O = 0 and lse = -inf.

The backward needs only the saved output and logsumexp (course week 13, step 2): with the
merged (global) lse and D = rowsum(dO o O) of the merged O, the probabilities of shard k
are P_k = exp(S_k - lse) (not renormalised within the shard), and

    dV_k = P_k^T dO,  dP_k = dO V_k^T,  dS_k = P_k o (dP_k - D),
    dQ  += scale dS_k K_k,  dK_k = scale dS_k^T Q,

so dQ is the sum of the shards' contributions and dK, dV of a shard come from that
shard alone (summed over the query shards that see it).
"""
from __future__ import annotations

import numpy as np


def merge_partials(o_parts, lse_parts):
    """Merge S partial results of the same query rows over disjoint key sets.

    o_parts [S, n, d] (each normalised over its own keys), lse_parts [S, n] (natural log,
    -inf where the part has no visible key).  Returns (O [n, d], lse [n]) in float64.
    """
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    m = lse_parts.max(axis=0)                      # [n]
    live = np.isfinite(m)
    w = np.zeros_like(lse_parts)
    w[:, live] = np.exp(lse_parts[:, live] - m[live])   # e^{lse_k - m}, 0 for -inf parts
    total = w.sum(axis=0)
    lse = np.full(m.shape, -np.inf)
    lse[live] = m[live] + np.log(total[live])
    w[:, live] /= total[live]                      # e^{lse_k - lse}
    o = np.einsum("kn,knd->nd", w, o_parts)
    return o, lse


def backward_head_with_stats(q, k, v, do, lse, D, scale: float, keep: np.ndarray):
    """Gradient contributions of one key/value shard for one head.

    q, do [n, d] (the query rows), k, v [m, d] (the shard's keys), lse, D [n] (the merged
    logsumexp and rowsum(dO o O) of the merged output), keep [n, m] the visibility of the
    shard's keys to the rows.  Returns (dQ contribution [n, d], dK [m, d], dV [m, d]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    lse = np.asarray(lse, np.float64)
    D = np.asarray(D, np.float64)
    s = scale * (q @ k.T)
    live = np.isfinite(lse)
    p = np.zeros_like(s)
    ok = keep & live[:, None]
    p[ok] = np.exp((s - np.where(live, lse, 0.0)[:, None])[ok])
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv
