"""Second CPU reference: the tiled forward with a running (m, l) state.

TEST INFRASTRUCTURE ONLY (same rule as ``attention.py``): used by the tests to
pin the oracle, never by the product path.

It follows the FlashAttention reading guide (arXiv 2205.14135), "Method":
the running statistics of a vector split into two parts merge as
m = max(m1, m2), l = e^{m1 - m} l1 + e^{m2 - m} l2, and for query block i and
key/value block j:

1. S_ij = Q_i K_j^T (scaled by 1/sqrt(d) as in the answer page, section 2.1);
2. m~_ij = rowmax(S_ij), P~_ij = exp(S_ij - m~_ij), l~_ij = rowsum(P~_ij);
3. m_i^new = max(m_i, m~_ij), l_i^new = e^{m_i - m_i^new} l_i + e^{m~_ij - m_i^new} l~_ij;
4. O_i <- diag(l_i^new)^-1 (diag(l_i) e^{m_i - m_i^new} O_i + e^{m~_ij - m_i^new} P~_ij V_j).

This is the renormalising form (O_i is kept normalised after every block).
The running maximum starts at -inf, not 0, and a block whose row is fully
masked (m~ = -inf) contributes nothing instead of producing
e^{-inf - (-inf)} = NaN: the two pitfalls the course page (week 13,
"typical mistakes") names.  Block sizes are free parameters: the result must
not depend on them.
"""
from __future__ import annotations

import numpy as np


def _exp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """e^{a - b} elementwise, taken as 0 where a = -inf (including -inf - -inf)."""
    a, b = np.broadcast_arrays(a, b)
    out = np.zeros(a.shape)
    ok = np.isfinite(a) & np.isfinite(b)
    out[ok] = np.exp(a[ok] - b[ok])
    return out


def tiled_forward_head(q, k, v, scale: float, keep: np.ndarray, br: int, bc: int):
    """One head, blocks of br query rows and bc key columns.  Returns (O, lse)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n = q.shape[0]
    o = np.zeros((n, v.shape[1]))
    l = np.zeros(n)
    m = np.full(n, -np.inf)
    for j0 in range(0, n, bc):
        j1 = min(n, j0 + bc)
        for i0 in range(0, n, br):
            i1 = min(n, i0 + br)
            s = scale * (q[i0:i1] @ k[j0:j1].T)
            s = np.where(keep[i0:i1, j0:j1], s, -np.inf)
            m_blk = s.max(axis=1)
            p_blk = _exp_diff(s, m_blk[:, None])
            l_blk = p_blk.sum(axis=1)
            m_old = m[i0:i1]
            l_old = l[i0:i1]
            m_new = np.maximum(m_old, m_blk)
            a_old = _exp_diff(m_old, m_new)
            a_blk = _exp_diff(m_blk, m_new)
            l_new = a_old * l_old + a_blk * l_blk
            num = (l_old * a_old)[:, None] * o[i0:i1] + a_blk[:, None] * (p_blk @ v[j0:j1])
            live = l_new > 0
            o_new = np.zeros_like(num)
            o_new[live] = num[live] / l_new[live, None]
            o[i0:i1] = o_new
            m[i0:i1] = m_new
            l[i0:i1] = l_new
    lse = np.full(n, -np.inf)
    live = l > 0
    lse[live] = m[live] + np.log(l[live])
    return o, lse
