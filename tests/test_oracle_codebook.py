"""Pins of the oracle's Lloyd-Max codebook and scalar quantizer.

The codebook is the precomputed Lloyd-Max scalar quantizer for a Gaussian that
the debugging post ("From 0% to 100%...", section 'Why this caught my eye') and
the aither-kvcache README (section 'Algorithm') describe.  It is pinned here
against things outside the oracle: scipy quadrature of the conditional means,
the closed form of the 1-bit quantizer, Max's 1960 table, an independent
numerical optimisation of the 2-bit quantizer, and the MSE values the README
prints.
"""
import math

import numpy as np
import pytest
from scipy import integrate, optimize, stats

import oracle


def _cond_mean(a, b):
    num = integrate.quad(lambda x: x * stats.norm.pdf(x), a, b, epsabs=1e-15, epsrel=1e-13, limit=200)[0]
    den = integrate.quad(lambda x: stats.norm.pdf(x), a, b, epsabs=1e-15, epsrel=1e-13, limit=200)[0]
    return num / den


def _distortion(c, t):
    edges = [-np.inf] + list(t) + [np.inf]
    tot = 0.0
    for k, ck in enumerate(c):
        tot += integrate.quad(lambda x: (x - ck) ** 2 * stats.norm.pdf(x), edges[k], edges[k + 1], epsabs=1e-15, limit=200)[0]
    return tot


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_fixed_point_conditions(bits):
    c, t, it = oracle.lloyd_max_f64(bits)
    assert np.all(np.diff(c) > 0)
    # midpoints are exactly the neighbour averages
    assert np.array_equal(t, 0.5 * (c[:-1] + c[1:]))
    edges = [-np.inf] + list(t) + [np.inf]
    for k in range(len(c)):
        assert abs(c[k] - _cond_mean(edges[k], edges[k + 1])) < 1e-11, (bits, k)
    # symmetric quantizer for a symmetric density
    assert np.array_equal(c, -c[::-1])


def test_one_bit_closed_form():
    c, t, _ = oracle.lloyd_max_f64(1)
    r = math.sqrt(2.0 / math.pi)
    assert abs(c[1] - r) < 1e-14 and abs(c[0] + r) < 1e-14
    assert t[0] == 0.0


@pytest.mark.parametrize("levels", ["2", "4", "8", "16"])
def test_matches_max_1960_table(golden, levels):
    g = golden("lloyd_max_gaussian.json")
    row = g["levels"][levels]
    tol = g["abs_tolerance_printed_digits"]
    bits = int(levels).bit_length() - 1
    c, t, _ = oracle.lloyd_max_f64(bits)
    L = len(c)
    np.testing.assert_allclose(c[L // 2:], row["outputs"], atol=tol)
    np.testing.assert_allclose(t[L // 2:], row["thresholds"], atol=tol)
    d = _distortion(c, t)
    # the table prints four significant digits
    assert abs(d - row["mse"]) <= 6e-4 * row["mse"]


def test_two_bit_independent_optimum():
    # minimise the exact 2-bit symmetric distortion over (inner, outer) levels
    def dist(p):
        a, b = p
        if not (0 < a < b):
            return 10.0
        return _distortion([-b, -a, a, b], [-(a + b) / 2, 0.0, (a + b) / 2])

    res = optimize.minimize(dist, x0=[0.5, 1.5], method="Nelder-Mead", options=dict(xatol=1e-10, fatol=1e-15, maxiter=4000))
    c, _, _ = oracle.lloyd_max_f64(2)
    np.testing.assert_allclose([c[2], c[3]], res.x, atol=2e-6)


def test_distortion_matches_validated_mse(golden):
    g = golden("validated_mse.json")
    for b in (2, 3, 4):
        c, t, _ = oracle.lloyd_max_f64(b)
        d = _distortion(c, t)
        assert abs(d - g["mse"][str(b)]) / g["mse"][str(b)] < 0.02, (b, d)
        assert d > 4.0 ** (-b)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_stored_codebook_is_fp16_rounding(bits):
    """Stored centroids are numpy's (correctly rounded, ties-to-even) fp16
    values of the fp64 fixed point; thresholds are the exact midpoints of
    neighbouring stored centroids."""
    c64, _, _ = oracle.lloyd_max_f64(bits)
    c32, t32 = oracle.make_codebook(bits)
    assert c32.dtype == np.float32 and t32.dtype == np.float32
    c16 = c64.astype(np.float16)
    assert np.array_equal(c32, c16.astype(np.float32))
    mid = 0.5 * (c16[:-1].astype(np.float64) + c16[1:].astype(np.float64))
    assert np.array_equal(t32.astype(np.float64), mid)  # exact in fp32
    assert np.array_equal(c32, -c32[::-1])
    assert np.all(np.diff(t32) > 0)
    # the rounding moves a centroid by at most half an fp16 ulp
    assert np.all(np.abs(c32 - c64) <= np.abs(c64) * 2.0 ** -11)


def test_round_to_half_matches_numpy():
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.standard_normal(2000) * 3, rng.standard_normal(500) * 1e-5, [0.5 * (1 + 2 ** -10), 1 + 3 * 2 ** -11,
                                                                                       6.103515625e-05, 2.0 ** -24 * 1.5, 65504.0, 65519.0, 65520.0]])
    for x in xs:
        with np.errstate(over="ignore"):
            want = float(np.float16(x))
        got = oracle.round_to_half(x)
        assert got == want or (np.isinf(want) and np.isinf(got)), (x, got, want)


def test_fp16_codebook_keeps_the_distortion(golden):
    """Storing the table at fp16 changes the Gaussian distortion by < 1e-4
    relative, so the validated MSE values still apply."""
    g = golden("validated_mse.json")
    for b in (2, 3, 4):
        c64, t64, _ = oracle.lloyd_max_f64(b)
        c32, t32 = oracle.make_codebook(b)
        d64 = _distortion(c64, t64)
        d16 = _distortion(c32.astype(np.float64), t32.astype(np.float64))
        assert d16 >= d64 - 1e-15  # the fp64 fixed point is the optimum
        assert (d16 - d64) / d64 < 1e-4, (b, d64, d16)
        assert abs(d16 - g["mse"][str(b)]) / g["mse"][str(b)] < 0.02


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_quantizer_count_rule_and_ties(bits):
    c, t = oracle.make_codebook(bits)
    rng = np.random.default_rng(bits)
    for u in rng.standard_normal(300) * 2:
        k = oracle.quantize_scalar(bits, t, u)
        # nearest centroid (distance), independent of the count rule
        assert k == int(np.argmin(np.abs(c.astype(np.float64) - u)))
    for k in range(len(t)):
        # a value exactly on a midpoint goes to the upper code
        assert oracle.quantize_scalar(bits, t, float(t[k])) == k + 1
        below = float(np.nextafter(t[k], np.float32(-np.inf)))
        assert oracle.quantize_scalar(bits, t, below) == k
    assert oracle.quantize_scalar(bits, t, -1e30) == 0
    assert oracle.quantize_scalar(bits, t, 1e30) == (1 << bits) - 1


def test_half_to_double_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[::97]])
    r = ref[::97]
    same = (got == r) | (np.isnan(got) & np.isnan(r))
    assert same.all()
    for b in (0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00):
        x = oracle.half_to_double(b)
        y = float(np.array([b], np.uint16).view(np.float16)[0])
        assert x == y and math.copysign(1, x) == math.copysign(1, y)
