"""Error bound of the FP8 forward's one extra rounding: P to e4m3 as the operand of P V.

The kernel computes, per query row, P_j = 2^(c s_j - m_ref) in fp32 with a reference
maximum m_ref that is at most the row's true maximum (it only ever takes a maximum seen so
far), rounds P_j to e4m3 for the product with V, and divides by l = sum_j P_j taken from the
unrounded values.  Against the exact result O = sum_j phat_j V_j (phat the normalised
probabilities) the error is  sum_j (e4m3(P_j) - P_j) / l * V_j.  Per key:
  * P_j >= 2^-6 (normal range): |e4m3(P_j) - P_j| <= 2^-4 P_j (half of the 2^-3 relative ulp);
  * P_j <  2^-6 (subnormal):    |e4m3(P_j) - P_j| <= 2^-10  (half of the 2^-9 step).
Dividing by l: P_j / l = phat_j, and l >= l_f = sum_j e^(s_j - m) (the same sum taken with
the true maximum, since m_ref <= m makes every P_j larger), so

    e_j = max(2^-4 phat_j, 2^-10 / l_f)

bounds key j's contribution per unit of |V_j|.  The deterministic bound is
sum_j e_j |V_jd| (+ 2^-12 sum_j phat_j |V_jd| for the fp32 exponentials and sums); treating
the roundings as independent and uniform within their bounds gives the variance
sum_j e_j^2 V_jd^2 / 3 used by the root-mean-square check.  The bf16 rounding of the
output (half an ulp, 2^-9 relative) comes on top.
"""
import numpy as np

import oracle


def head_terms(Q, K, V, scale, keep):
    """Exact O of one head and the two bound terms; all [N, dv] float64."""
    S = scale * (Q @ K.T)
    S = np.where(keep, S, -np.inf)
    live = keep.any(axis=1)
    m = np.where(live, S.max(axis=1), 0.0)
    Pf = np.where(keep, np.exp(S - m[:, None]), 0.0)
    lf = Pf.sum(axis=1)
    lf_safe = np.where(live, lf, 1.0)
    phat = Pf / lf_safe[:, None]
    e = np.where(keep, np.maximum(2.0 ** -4 * phat, 2.0 ** -10 / lf_safe[:, None]), 0.0)
    aV = np.abs(V)
    bound = e @ aV + 2.0 ** -12 * (phat @ aV)
    var = (e * e) @ (V * V) / 3.0
    o = phat @ V
    return o, bound, var


def check(o_lib, o_ref, Q, K, V, scale, keep, rms_factor=2.0):
    """Assert the bounds for the rows of one head (Q and keep may be a subset of the rows);
    ``o_ref`` is the oracle's exact O of those rows.  Returns (max error / bound, rms /
    predicted rms)."""
    _, bound, var = head_terms(Q, K, V, scale, keep)
    o = np.asarray(o_ref, np.float64)
    diff = np.abs(np.asarray(o_lib, np.float64) - o)
    out_round = 2.0 ** -9 * (np.abs(o) + bound)
    lim = bound + out_round + 1e-7
    worst = float((diff / lim).max()) if diff.size else 0.0
    assert np.all(diff <= lim), f"max error beyond the e4m3 P bound: ratio {worst:.3g}"
    pred = np.sqrt(np.mean(var + (2.0 ** -9 * o) ** 2 / 3.0)) + 1e-7
    rms = float(np.sqrt(np.mean(diff * diff)))
    assert rms <= rms_factor * pred, f"rms error {rms:.3g} > {rms_factor} x predicted {pred:.3g}"
    return worst, rms / pred


def keep_for(N, causal, blockmask, kv_len, b):
    L = None if kv_len is None else int(kv_len[b])
    return oracle.keep_mask(N, causal, blockmask, L)
