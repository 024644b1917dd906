"""Pins of the FP8 oracle (CPU): the e4m3 codec against the format definition and torch's
float8_e4m3fn, the power-of-two scale rule, and the bound the GPU tests use for the kernel's
e4m3 rounding of P, checked against a direct emulation of that rounding."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8

import _fp8_bound

RNG = np.random.default_rng(11)


def test_decoder_matches_every_code_of_torch_float8_e4m3fn():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = fp8.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    assert np.isnan(mine).sum() == 2  # S.1111.111 only: no infinities in e4m3
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])


def test_format_constants():
    v = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    v = v[~np.isnan(v)]
    assert v.max() == 448.0 and v.min() == -448.0
    pos = np.unique(v[v > 0])
    assert pos[0] == 2.0 ** -9                   # smallest subnormal
    assert pos[pos >= 2.0 ** -6][0] == 2.0 ** -6  # smallest normal
    assert len(pos) == 126                        # 7 subnormals + 15 binades x 8 - 1 (NaN)


def test_rounding_matches_torch_cast_inside_the_finite_range():
    x = np.concatenate([RNG.uniform(-448, 448, 50000), RNG.standard_normal(50000),
                        RNG.normal(0, 0.01, 50000), RNG.uniform(-2 ** -6, 2 ** -6, 50000)])
    grid = np.unique(np.abs(fp8.e4m3_decode(np.arange(127, dtype=np.uint8))))
    mids = (grid[1:] + grid[:-1]) / 2          # exact ties, both parities of the lower code
    x = np.concatenate([x, mids, -mids, grid, -grid]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(fp8.e4m3_round(x.astype(np.float64)), ref)


def test_rounding_fixed_by_the_format_definition():
    r = fp8.e4m3_round
    assert r(1.0 + 1 / 16) == 1.0          # tie between 1.000 and 1.001: even mantissa
    assert r(1.0 + 3 / 16) == 1.25         # tie between 1.001 and 1.010: even mantissa
    assert r(2.0 ** -10) == 0.0            # half the smallest subnormal: ties to even (0)
    assert r(3 * 2.0 ** -10) == 2.0 ** -8  # 1.5 subnormal steps: ties to even (2 steps)
    assert r(460.0) == 448.0 and r(1e6) == 448.0 and r(-1e6) == -448.0  # saturation
    assert r(0.0) == 0.0
    assert r(-0.3) == -0.3125


def test_scale_exponent_rule():
    k = fp8.pow2_scale_exponent(np.array([448.0, 449.0, 224.0, 1.0, 1.75, 1.7578125, 0.0]))
    assert list(k) == [0, 1, -1, -8, -8, -7, 0]
    amax = np.abs(RNG.standard_normal(2000) * np.exp2(RNG.integers(-60, 60, 2000)))
    k = fp8.pow2_scale_exponent(amax)
    s = np.exp2(k.astype(np.float64))
    assert np.all(amax / s <= 448.0)       # fits
    assert np.all(amax / s > 224.0)        # and uses the top binade (k is the smallest)


def test_quantize_blocks_and_heads():
    x = RNG.standard_normal((2, 3, 300, 16))
    x[0, 1, 128:256] *= 1e3      # one block with a much larger range
    x[1, 2, 256:] = 0.0          # an all-zero (partial) block: scale 1, codes 0
    x8, s = fp8.quantize_blocks(x)
    assert s.shape == (2, 3, 3)
    assert s[0, 1, 1] == 2.0 ** fp8.pow2_scale_exponent(np.abs(x[0, 1, 128:256]).max())
    assert s[1, 2, 2] == 1.0 and np.all(x8[1, 2, 256:] == 0)
    assert np.all(np.abs(x8) <= 448)
    assert np.array_equal(fp8.e4m3_round(x8), x8)          # values on the e4m3 grid
    xd = fp8.dequantize_blocks(x8, s)
    big = np.abs(x) >= 2.0 ** -6 * np.repeat(s, 128, axis=2)[:, :, :300, None]
    rel = np.abs(xd - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -4                           # half an ulp in the normal range
    # Idempotent on the decoded values (the codes may differ: an amax that rounds down to 224
    # halves the scale and doubles every code, exactly).
    x8b, sb = fp8.quantize_blocks(xd)
    assert np.array_equal(fp8.dequantize_blocks(x8b, sb), xd)
    v8, sv = fp8.quantize_heads(x)
    assert sv.shape == (2, 3) and sv[0, 1] == 2.0 ** fp8.pow2_scale_exponent(np.abs(x[0, 1]).max())


def test_forward_on_encoded_inputs_is_the_plain_forward():
    B, H, N, d = 1, 2, 70, 8
    q8 = fp8.e4m3_round(RNG.standard_normal((B, H, N, d)) * 8)
    k8 = fp8.e4m3_round(RNG.standard_normal((B, H, N, d)) * 8)
    v8 = fp8.e4m3_round(RNG.standard_normal((B, H, N, d)) * 8)
    ones_b, ones_h = np.ones((B, H, 1)), np.ones((B, H))
    o, lse = fp8.forward_fp8(q8, ones_b, k8, ones_b, v8, ones_h, 0.1, causal=True)
    o2, lse2 = oracle.forward(q8, k8, v8, 0.1, causal=True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # and the scales multiply the decoded operands: scaling k8's scale by 2 doubles the scores
    o3, lse3 = fp8.forward_fp8(q8, ones_b, k8, 2 * ones_b, v8, ones_h, 0.05, causal=True)
    np.testing.assert_allclose(o3, o, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shift", [0.0, 3.0, 7.9])
def test_p_rounding_bound_covers_an_emulation_of_the_kernel(shift):
    # Emulate the kernel's arithmetic for P: fp32 P_j = 2^(c s_j - m_ref) with a reference
    # maximum `shift` (log2 units) below the true one, rounded to e4m3, divided by the fp32
    # sum of the unrounded P.  The bound must hold elementwise and the rms must sit under
    # twice the predicted spread.
    N, d = 384, 64
    for logit_mult in (1.0, 4.0):
        Q = RNG.standard_normal((N, d)) * logit_mult
        K = RNG.standard_normal((N, d))
        V = RNG.standard_normal((N, d))
        scale = d ** -0.5
        keep = oracle.keep_mask(N, causal=True)
        S = np.where(keep, scale * Q @ K.T, -np.inf)
        m = S.max(axis=1, keepdims=True)
        log2e = 1.0 / np.log(2.0)
        Pk = np.where(keep, np.exp2(((S - m) * log2e + shift).astype(np.float32)), 0.0)
        Pk = Pk.astype(np.float32)
        lk = Pk.sum(axis=1, dtype=np.float32)
        Pq = fp8.e4m3_round(Pk.astype(np.float64))
        o_emu = (Pq @ V) / lk[:, None]
        o_ref = oracle.forward_head(Q, K, V, scale, keep)[0]
        worst, rms_ratio = _fp8_bound.check(o_emu, o_ref, Q, K, V, scale, keep)
        assert worst <= 1.0 and rms_ratio <= 2.0


def test_p_rounding_bound_detects_a_permuted_value_block():
    # The check must fail for a plausible kernel mistake: key blocks of V taken in the wrong
    # order within a 128-key tile.
    N, d = 256, 64
    Q, K, V = (RNG.standard_normal((N, d)) for _ in range(3))
    keep = oracle.keep_mask(N)
    scale = d ** -0.5
    perm = np.arange(N)
    perm[0:32], perm[32:64] = np.arange(32, 64), np.arange(0, 32)
    o_bad, _, _ = _fp8_bound.head_terms(Q, K, V[perm], scale, keep)
    o_ref = oracle.forward_head(Q, K, V, scale, keep)[0]
    with pytest.raises(AssertionError):
        _fp8_bound.check(o_bad, o_ref, Q, K, V, scale, keep)
