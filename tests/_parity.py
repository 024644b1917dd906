"""Shared helpers of the GPU parity tests: run the library, run the oracle, compare.

Tolerances (written here, used by every parity test):
  fp32: max|dO| <= 1e-4, max|dlse| <= 1e-4, max|dgrad| <= 1e-4 * max|grad|
  bf16: max|dO| <= 2e-2, max|dlse| <= 1e-3, max|dgrad| <= 2e-2 * max|grad|
where d denotes the difference between the library's output (upcast to fp64) and the
oracle's fp64 result on the same (bf16-rounded) inputs.  A gradient that is identically
zero in exact arithmetic (N = 1 gives dQ = dK = 0) has no scale to be relative to: there
the bound is absolute, max|grad| <= ZERO_GRAD_ABS.

With dropout, O = (P o Z) V / (1 - p): the kernel's roundings of P V (P to bf16 as the MMA
operand) and of O itself are both multiplied by the keep scale 1 / (1 - p), so the O bound
is the plain one times that scale (``o_scale``); lse does not depend on the mask and the
gradient bounds are already relative to max|grad|.
"""
import numpy as np
import torch

import oracle
from exact_io_aware_28_gb300 import fa

ZERO_GRAD_ABS = 1e-4
TOL = {
    "fp32": {"o": 1e-4, "lse": 1e-4, "grad": 1e-4},
    "bf16": {"o": 2e-2, "lse": 1e-3, "grad": 2e-2},
}


def np64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def run_library(x):
    o, lse = fa.forward(x.q, x.k, x.v, x.causal, x.blockmask, x.kv_len, x.scale)
    dq, dk, dv = fa.backward(x.q, x.k, x.v, o, lse, x.do, x.causal, x.blockmask, x.kv_len,
                             x.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_error() == fa.FA_OK
    return o, lse, dq, dk, dv


def run_oracle(x, heads=None):
    q, k, v, do = (np64(t) for t in (x.q, x.k, x.v, x.do))
    bm = None if x.blockmask is None else x.blockmask.cpu().numpy()
    kl = None if x.kv_len is None else x.kv_len.cpu().numpy()
    o, lse = oracle.forward(q, k, v, x.scale, x.causal, bm, kl, heads=heads)
    dq, dk, dv, _ = oracle.backward(q, k, v, do, x.scale, x.causal, bm, kl, heads=heads)
    return o, lse, dq, dk, dv


def compare(lib_out, ref_out, dtype, heads=None, o_scale=1.0):
    """Assert the tolerances; returns a dict of the measured errors."""
    tol = TOL[dtype]
    o, lse, dq, dk, dv = (np64(t) for t in lib_out)
    ro, rlse, rdq, rdk, rdv = ref_out
    if heads is not None:
        sel = tuple(np.array(h) for h in zip(*heads))
        o, lse, dq, dk, dv = (a[sel] for a in (o, lse, dq, dk, dv))
        ro, rlse, rdq, rdk, rdv = (a[sel] for a in (ro, rlse, rdq, rdk, rdv))
    errs = {}
    errs["o"] = float(np.abs(o - ro).max())
    dead = np.isneginf(rlse)
    assert np.array_equal(np.isneginf(lse), dead), "rows without a visible key differ"
    assert np.all(np.isfinite(lse[~dead]))
    errs["lse"] = float(np.abs(lse[~dead] - rlse[~dead]).max()) if (~dead).any() else 0.0
    for name, g, r in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
        assert np.all(np.isfinite(g)), name
        scale = float(np.abs(r).max())
        if scale < 1e-12:
            errs[name] = float(np.abs(g).max()) / ZERO_GRAD_ABS * tol["grad"]
        else:
            errs[name] = float(np.abs(g - r).max()) / scale
    assert errs["o"] <= tol["o"] * max(1.0, o_scale), errs
    assert errs["lse"] <= tol["lse"], errs
    for name in ("dq", "dk", "dv"):
        assert errs[name] <= tol["grad"], (name, errs)
    return errs
