"""Pins for the NVFP4 encoding with a given per-tensor scale (oracle.nvfp4_quantize_scaled, CPU).

This is the single-pass form of the NVFP4 step of the kernel plan in
"NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md" (item 7): the caller supplies s_g, so only the block-scale and
element roundings remain.  Pinned to the two-pass quantiser (itself pinned in
test_oracle_nvfp4.py), to an exact rational brute force, and to closed forms."""
from fractions import Fraction

import numpy as np
import pytest

import oracle

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e4m3_values():
    """Non-negative finite E4M3FN values by code 0..0x7E, as exact fractions."""
    out = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        out.append(Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7))
    return out


E4M3 = e4m3_values()


def nearest_code(q: Fraction, values, top_saturates=True):
    """Index of the value nearest to q >= 0, ties to the even index, saturating at the top."""
    if top_saturates and q >= values[-1]:
        return len(values) - 1
    best = 0
    for c in range(1, len(values)):
        d, db = abs(q - values[c]), abs(q - values[best])
        if d < db or (d == db and c % 2 == 0):
            best = c
    return best


def brute_force(x: np.ndarray, sg: float):
    """Exact-rational reference of steps 2-4 for x (n % 16 == 0) and s_g > 0 finite."""
    s = Fraction(float(np.float32(sg)))
    e2 = [Fraction(v) for v in E2M1]
    codes = np.zeros(x.size // 2, np.uint8)
    scales = np.zeros(x.size // 16, np.uint8)
    for b in range(x.size // 16):
        blk = [float(v) for v in x[16 * b:16 * b + 16]]
        ab = max(Fraction(abs(v)) for v in blk)
        sc = nearest_code(ab / (6 * s), E4M3)
        scales[b] = sc
        den = E4M3[sc] * s
        for i, v in enumerate(blk):
            c = 0 if den == 0 else nearest_code(Fraction(abs(v)) / den, e2)
            if np.signbit(v):
                c |= 8
            e = 16 * b + i
            codes[e // 2] |= c << (4 * (e & 1))
    return codes, scales


def test_derived_scale_equals_two_pass():
    rng = np.random.default_rng(0)
    for trial in range(5):
        x = (rng.standard_normal(4096) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        c2, s2, sg = oracle.nvfp4_quantize(x)
        c1, s1 = oracle.nvfp4_quantize_scaled(x, sg)
        np.testing.assert_array_equal(c1, c2)
        np.testing.assert_array_equal(s1, s2)


@pytest.mark.parametrize("sg_factor", [1.0, 0.37, 3.1, 1e-3, 40.0])
def test_exact_rational_brute_force(sg_factor):
    """Random blocks (with exact midpoints planted) under scales that fit, saturate or underflow."""
    rng = np.random.default_rng(int(sg_factor * 1000))
    x = (rng.standard_normal(16 * 24) * np.repeat(10.0 ** rng.uniform(-2, 2, 24), 16)).astype(np.float32)
    sg = np.abs(x).max() / 2688.0 * sg_factor
    e = np.floor(np.log2(sg))
    sg = float(np.round(sg / 2.0 ** (e - 7)) * 2.0 ** (e - 7))   # 8 significant bits: midpoint products are exact
    # plant elements exactly on E2M1 midpoints of their block's scale (ties)
    c0, s0 = oracle.nvfp4_quantize_scaled(x, sg)
    planted = 0
    for b in range(0, 24, 3):
        den = oracle.e4m3_decode(int(s0[b])) * sg
        for i, mid in enumerate([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]):
            v = np.float32(mid * den)
            if float(v) == mid * den and abs(v) < np.abs(x[16 * b:16 * b + 16]).max():
                x[16 * b + 1 + i] = -v if i % 2 else v
                planted += 1
    assert planted >= 20
    codes, scales = oracle.nvfp4_quantize_scaled(x, sg)
    rc, rs = brute_force(x, sg)
    np.testing.assert_array_equal(scales, rs)
    np.testing.assert_array_equal(codes, rc)


def test_power_of_two_scale_invariance():
    """x*2^k with s_g*2^k gives the same encoding: every quotient in the definition is unchanged."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal(2048).astype(np.float32)
    sg = float(np.float32(np.abs(x).max() / 2688.0 * 0.8))
    c0, s0 = oracle.nvfp4_quantize_scaled(x, sg)
    for k in (-40, -7, 9, 60):
        c, s = oracle.nvfp4_quantize_scaled((x * np.float32(2.0 ** k)).astype(np.float32), sg * 2.0 ** k)
        np.testing.assert_array_equal(c, c0)
        np.testing.assert_array_equal(s, s0)


def test_saturation_closed_form():
    """With s_g far below amax / 2688 every non-zero block takes the largest scale (448) and every
    non-zero element the largest magnitude (6), sign kept."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal(1024).astype(np.float32)
    x[5] = 0.0
    x[6] = -0.0
    x[7] = 1e-3            # still far above 6 * den at this scale
    sg = 1e-12
    codes, scales = oracle.nvfp4_quantize_scaled(x, sg)
    assert np.all(scales == 0x7E)
    nib = np.stack([codes & 0xF, codes >> 4], 1).reshape(-1)
    want = np.where(x == 0, 0, 7) | np.where(np.signbit(x), 8, 0)
    np.testing.assert_array_equal(nib, want)


def test_underflow_closed_form():
    """With amax_b / (6 s_g) below half the smallest E4M3 subnormal (2^-10) every scale rounds to 0,
    and a zero scale encodes the block as zero."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal(512).astype(np.float32)
    sg = float(np.abs(x).max()) / 6.0 * 2.0 ** 10 * 1.01
    codes, scales = oracle.nvfp4_quantize_scaled(x, sg)
    assert np.all(scales == 0) and np.all(codes == 0)
    # exactly on 2^-10: a tie between codes 0 and 1 goes to the even code 0
    y = np.zeros(16, np.float32)
    y[3] = 6.0
    c, s = oracle.nvfp4_quantize_scaled(y, 2.0 ** 10)
    assert s[0] == 0
    c, s = oracle.nvfp4_quantize_scaled(y, 2.0 ** 10 * 0.99)
    assert s[0] == 1


@pytest.mark.parametrize("sg", [0.0, -1.0, float("inf"), float("-inf"), float("nan")])
def test_unusable_scale_encodes_zero(sg):
    x = np.random.default_rng(5).standard_normal(64).astype(np.float32)
    codes, scales = oracle.nvfp4_quantize_scaled(x, sg)
    assert np.all(codes == 0) and np.all(scales == 0)


def test_error_bound_without_saturation():
    """Where a block neither saturates nor underflows, every element is within one E2M1 step of
    the encoding: |x - dec| <= den (the largest half-gap of the E2M1 grid, between 4 and 6)."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal(8192).astype(np.float32)
    sg = float(np.float32(np.abs(x).max() / 2688.0 * 1.5))
    codes, scales = oracle.nvfp4_quantize_scaled(x, sg)
    deq = oracle.nvfp4_dequantize(codes, scales, sg)
    den = np.repeat([oracle.e4m3_decode(int(s)) for s in scales], 16) * sg
    ab = np.repeat(np.abs(x).reshape(-1, 16).max(1), 16)
    ok = (ab <= 6 * 448 * sg) & (den > 0)
    assert ok.mean() > 0.99
    assert np.all(np.abs(x[ok] - deq[ok]) <= den[ok] * (1 + 1e-12))
