"""CPU fp64 oracle for the FP8 (e4m3) forward: the input encoding and the attention it feeds.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute this
module: only the tests, the package's ``smoke()`` check and the benchmark's CPU legs use it.
It shares no code with the CUDA path and imports nothing from the package.

What it computes.  The pages name FP8 as one of the things the third FlashAttention adds
(answer page "How FlashAttention works for training", section 7 on FlashAttention-2 and -3;
course page "Week 13. GPU and FlashAttention", step 2, the bullet on FA2 and FA3); they say
nothing more about it.  The plainest reading, taken here:

* The operands of the two products, Q K^T and P V, are 8-bit floats, e4m3 (1 sign bit, 4
  exponent bits with bias 7, 3 mantissa bits, no infinities, largest finite value 448;
  "FP8 Formats for Deep Learning", Micikevicius et al. 2022, and the OCP 8-bit floating
  point specification).  A bf16 tensor is encoded with one power-of-two scale per block of
  128 rows (Q, K) or per head (V):  x = s * e4m3(x / s),  s = 2^k, k the smallest integer
  with amax <= 448 * 2^k (so x / s is exact and the largest element lands in e4m3's top
  binade).  Rounding is to nearest, ties to even; magnitudes above 448 saturate to 448.
* The attention itself is the exact definition of ``attention.py`` applied to the decoded
  inputs  Q = s_q * q8,  K = s_k * k8,  V = s_v * v8.  The one further rounding the kernel
  makes, P to e4m3 as the operand of P V, is not part of the definition: the tests bound it
  (half an e4m3 ulp per probability, 2^-4 relative, or 2^-10 absolute below 2^-6).

Pins (CPU tests): the decoder against every one of the 256 codes of torch.float8_e4m3fn;
the rounding against torch's cast on values inside the finite range; values the format
definition fixes (448, 2^-6, 2^-9, ties to even, saturation); the scale rule's boundary
cases; idempotence of the encoding; the forward on already-encoded inputs with scale 1
against the plain oracle.
"""
from __future__ import annotations

import numpy as np

from .attention import forward

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_STEP = 2.0 ** -9
ROW_BLOCK = 128


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 byte (uint8 array) from the format definition; NaN for S.1111.111."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * E4M3_SUBNORMAL_STEP, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def _round_half_even(x: np.ndarray) -> np.ndarray:
    return np.round(x)  # NumPy rounds halves to even


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even) of each element, saturating at +-448; float64 out.

    Works on the magnitude: below 2^-6 the spacing is the subnormal step 2^-9, in the
    binade [2^e, 2^(e+1)) it is 2^(e-3).  A value that rounds up to the next binade is still
    on the grid, so no renormalisation is needed.
    """
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # log2 of values just under a power of two can round up: correct the binade exactly.
    e = np.where(np.exp2(e) > a, e - 1, e)
    e = np.where(np.exp2(e + 1) <= a, e + 1, e)
    step = np.where(a < E4M3_MIN_NORMAL, E4M3_SUBNORMAL_STEP, np.exp2(e - 3))
    r = _round_half_even(a / step) * step
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def pow2_scale_exponent(amax) -> np.ndarray:
    """k of the scale s = 2^k: the smallest integer with amax <= 448 * 2^k, within
    [-126, 127]; k = 0 for amax = 0.  ``amax`` is exact (a bf16 value), so the comparison is
    exact: writing amax = f * 2^E with f in [0.5, 1), 448 = 0.875 * 2^9 gives
    k = E - 9 when f <= 0.875, else E - 8."""
    a = np.asarray(amax, np.float64)
    f, E = np.frexp(a)
    k = np.where(f <= 0.875, E - 9, E - 8).astype(np.int64)
    k = np.clip(k, -126, 127)
    return np.where(a > 0, k, 0)


def _encode(x: np.ndarray, s: np.ndarray) -> np.ndarray:
    return e4m3_round(x / s)  # x / 2^k is exact in float64


def quantize_blocks(x, rows: int = ROW_BLOCK):
    """x [B, H, N, d] -> (x8 [B, H, N, d] e4m3 values as float64, s [B, H, ceil(N/rows)]).

    One power-of-two scale per block of ``rows`` consecutive rows of each (b, h)."""
    x = np.asarray(x, np.float64)
    B, H, N, d = x.shape
    nb = (N + rows - 1) // rows
    s = np.empty((B, H, nb))
    x8 = np.empty_like(x)
    for i in range(nb):
        blk = x[:, :, i * rows:(i + 1) * rows, :]
        amax = np.abs(blk).max(axis=(2, 3)) if blk.size else np.zeros((B, H))
        si = np.exp2(pow2_scale_exponent(amax).astype(np.float64))
        s[:, :, i] = si
        x8[:, :, i * rows:(i + 1) * rows, :] = _encode(blk, si[:, :, None, None])
    return x8, s


def quantize_heads(x):
    """x [B, H, N, d] -> (x8 values, s [B, H]): one power-of-two scale per (b, h)."""
    x = np.asarray(x, np.float64)
    amax = np.abs(x).max(axis=(2, 3))
    s = np.exp2(pow2_scale_exponent(amax).astype(np.float64))
    return _encode(x, s[:, :, None, None]), s


def dequantize_blocks(x8, s, rows: int = ROW_BLOCK) -> np.ndarray:
    x8 = np.asarray(x8, np.float64)
    per_row = np.repeat(np.asarray(s, np.float64), rows, axis=2)[:, :, :x8.shape[2]]
    return x8 * per_row[..., None]


def forward_fp8(q8, q_scale, k8, k_scale, v8, v_scale, scale: float, causal: bool = False,
                blockmask=None, kv_len=None, heads=None):
    """Exact attention on the decoded e4m3 inputs.

    q8, k8 [B, H, N, d] with per-128-row-block scales [B, H, nb]; v8 [B, H, N, d] with
    per-head scales [B, H].  Returns (o, lse) in float64 as ``attention.forward``."""
    Q = dequantize_blocks(q8, q_scale)
    K = dequantize_blocks(k8, k_scale)
    V = np.asarray(v8, np.float64) * np.asarray(v_scale, np.float64)[:, :, None, None]
    return forward(Q, K, V, scale, causal, blockmask, kv_len, heads=heads)
