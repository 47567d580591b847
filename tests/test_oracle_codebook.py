"""Pins for the oracle's coordinate density and Lloyd-Max codebook, each checked
against something other than the oracle's own formula: closed forms, the
uniform special case, the Gaussian limit (Max 1960), independent quadrature,
and the bound printed on the TurboQuant/MNN page (§2.3)."""
import math

import numpy as np
import pytest
from scipy import integrate

from conftest import golden_path, read_golden_kv
from oracle import tq_oracle as O


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_d3_is_uniform(bits):
    # d = 3: f(t) is uniform on [-1, 1] (Archimedes), so the Lloyd-Max
    # quantiser is the uniform one with centroids -1 + (2k+1)/2^b and
    # per-coordinate MSE = step^2 / 12.
    cb = O.lloyd_max_codebook(3, bits)
    K = 1 << bits
    want = -1.0 + (2 * np.arange(K) + 1) / K
    np.testing.assert_allclose(cb.centroids, want, atol=1e-13)
    step = 2.0 / K
    assert abs(O.codebook_mse(cb) - step * step / 12) < 1e-13


@pytest.mark.parametrize("d", [2, 3, 18, 32, 66, 128, 512])
def test_one_bit_closed_form(d):
    # b = 1: centroids are +-E|T| = +-Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2)).
    cb = O.lloyd_max_codebook(d, 1)
    want = math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
    np.testing.assert_allclose(cb.centroids, [-want, want], rtol=0, atol=1e-14)


def test_one_bit_values_at_128_and_32():
    assert abs(O.codebook(128, 1).centroids[1] - 0.0706616) < 5e-8
    assert abs(O.codebook(32, 1).centroids[1] - 0.1421535) < 5e-8


def _levels():
    out = {}
    with open(golden_path("max1960_gaussian_levels.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                b, *lv = line.split()
                out[int(b)] = np.array([float(x) for x in lv])
    return out


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_gaussian_limit_max1960(bits):
    # As d grows sqrt(d) T -> N(0,1): the scaled centroids approach Max's
    # Gaussian Lloyd-Max levels (printed to 4 significant digits).
    lv = _levels()[bits]
    cb = O.lloyd_max_codebook(200000, bits)
    pos = np.sqrt(200000) * cb.centroids[(1 << bits) // 2:]
    np.testing.assert_allclose(pos, lv, rtol=2.5e-3, atol=6e-4)


def _quad_cell(lo, hi, a):
    # Independent quadrature with t = sin(theta): (1-t^2)^a dt = cos^(2a+1) dtheta,
    # smooth for a >= -1/2 (no singular end points).
    th0, th1 = math.asin(lo), math.asin(hi)
    m0 = integrate.quad(lambda th: math.cos(th) ** (2 * a + 1), th0, th1, epsabs=0, epsrel=1e-13, limit=200)[0]
    m1 = integrate.quad(lambda th: math.sin(th) * math.cos(th) ** (2 * a + 1), th0, th1,
                        epsabs=0, epsrel=1e-13, limit=200)[0]
    return m0, m1


@pytest.mark.parametrize("d,bits", [(128, 3), (128, 4), (32, 3), (32, 4), (2, 3), (24, 1), (18, 2), (20, 3), (66, 4)])
def test_centroid_and_midpoint_conditions(d, bits):
    cb = O.codebook(d, bits)
    a = (d - 3) / 2
    # midpoint condition
    np.testing.assert_allclose(cb.boundaries, 0.5 * (cb.centroids[:-1] + cb.centroids[1:]), atol=1e-15)
    # centroid condition by independent quadrature of the unnormalised density
    edges = np.concatenate(([-1.0], cb.boundaries, [1.0]))
    for k in range(1 << bits):
        m0, m1 = _quad_cell(edges[k], edges[k + 1], a)
        assert abs(m1 / m0 - cb.centroids[k]) < 1e-11, (k, m1 / m0, cb.centroids[k])


@pytest.mark.parametrize("d,bits", [(128, 3), (32, 4), (66, 4), (2, 2)])
def test_symmetry(d, bits):
    cb = O.codebook(d, bits)
    np.testing.assert_allclose(cb.centroids, -cb.centroids[::-1], atol=1e-15)
    assert cb.boundaries[len(cb.boundaries) // 2] == 0.0 or abs(cb.boundaries[len(cb.boundaries) // 2]) < 1e-16
    assert np.all(np.diff(cb.centroids) > 0)


def test_density_exponent_pins_the_density():
    # The exponent (d-3)/2: the probability mass of |T| <= x must equal the
    # fraction of the sphere's area in that band, which for d = 3 is x
    # (Archimedes' hat-box theorem) and for d = 4 is (2/pi)(asin x + x sqrt(1-x^2)).
    for x in (0.1, 0.5, 0.9):
        assert abs(O.coord_cdf(x, 3) - O.coord_cdf(-x, 3) - x) < 1e-14
        want4 = (2 / math.pi) * (math.asin(x) + x * math.sqrt(1 - x * x))
        assert abs(O.coord_cdf(x, 4) - O.coord_cdf(-x, 4) - want4) < 1e-14


def test_std_at_128_matches_page():
    pages = read_golden_kv("pages_numbers.txt")
    # Var T = 1/d for a coordinate of a uniform point on the sphere.
    var = O.cell_second_moment(-1.0, 1.0, 128)
    assert abs(var - 1 / 128) < 1e-15
    assert abs(math.sqrt(var) - float(pages["coord_std_128"][0])) < 5e-4


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [32, 128])
def test_mse_bound_page(d, bits):
    # [TQ-MNN §2.3]: unit-vector MSE <= 2.7 / 4^b, information-theoretic floor 1/4^b.
    pages = read_golden_kv("pages_numbers.txt")
    mse_unit = d * O.codebook_mse(O.codebook(d, bits))
    assert mse_unit <= float(pages["mse_bound_const"][0]) / 4 ** bits
    assert mse_unit >= 1.0 / 4 ** bits


def test_mse_by_monte_carlo():
    # Gaussian vectors are rotation invariant, so after any fixed orthogonal R
    # the normalised coordinates follow f(t); the empirical reconstruction MSE
    # of unit vectors matches the closed form.
    rng = np.random.default_rng(7)
    d, bits = 128, 3
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    spec = O.spec_wht128(signs, bits)
    x = rng.standard_normal((4000, d))
    idx, nrm, _ = O.quantize(x, spec, "f32")
    xr = O.dequantize(idx, nrm.astype(np.float64), spec)
    rel = np.sum((xr - x) ** 2, axis=1) / np.sum(x * x, axis=1)
    want = d * O.codebook_mse(O.codebook(d, bits))
    assert abs(rel.mean() - want) < 0.03 * want


@pytest.mark.parametrize("bits,key", [(3, "ip_shrink_3bit"), (4, "ip_shrink_4bit")])
def test_inner_product_shrink_matches_page(bits, key):
    # [TQ-MNN §2.4]: the MSE quantiser shrinks inner products by about 4% (3 bits)
    # and 1% (4 bits).  Measured as 1 - E<x_hat, x>/||x||^2 on Gaussian vectors.
    pages = read_golden_kv("pages_numbers.txt")
    rng = np.random.default_rng(11)
    d = 128
    spec = O.spec_wht128(np.ones(d), bits)
    x = rng.standard_normal((4000, d))
    idx, nrm, _ = O.quantize(x, spec, "f32")
    xr = O.dequantize(idx, nrm.astype(np.float64), spec)
    shrink = 1 - np.mean(np.sum(xr * x, axis=1) / np.sum(x * x, axis=1))
    page = float(pages[key][0])
    assert 0.5 * page < shrink < 1.5 * page
