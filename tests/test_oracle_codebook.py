"""Pins of the oracle codebook against facts independent of its own formulas.

* Textbook Lloyd-Max quantizers of N(0,1) (Max 1960): the sphere marginal
  tends to N(0, 1/d) ([Reconstruction] §5 Step 3), so sqrt(d) * c must
  approach them as d grows.
* Monte Carlo on uniform points of the sphere (drawn with numpy's own
  generator, normalised Gaussian vectors): cell probabilities, conditional
  means (the Lloyd-Max centroid condition) and the quantizer MSE.
* [README] §Paper Validation: the ratio of the measured MSE to the Theorem 1
  bound is 0.70x at 2 bits and 0.82x at 3 bits.
"""

import math

import numpy as np
import pytest

from oracle import codebook as cb

GAUSS_LM = {  # positive output levels and MSE of the N(0,1) Lloyd-Max quantizer
    1: ([0.7979], 0.3634),
    2: ([0.4528, 1.5104], 0.1175),
    3: ([0.2451, 0.7560, 1.3439, 2.1519], 0.03455),
    4: ([0.1284, 0.3881, 0.6568, 0.9423, 1.2562, 1.6180, 2.0690, 2.7326], 0.009497),
}


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_gaussian_limit(bits):
    levels, mse = GAUSS_LM[bits]
    c = cb.lloyd_max(4096, bits)
    pos = c.centroids[len(c.centroids) // 2:].astype(np.float64)
    np.testing.assert_allclose(pos, levels, atol=3e-3)
    assert abs(c.mse_unit - mse) < 3e-3 * mse + 2e-5
    # finite d sits below the Gaussian values and moves toward them as d grows
    c128 = cb.lloyd_max(128, bits)
    c256 = cb.lloyd_max(256, bits)
    e128 = np.max(np.abs(c128.centroids[len(c128.centroids) // 2:] - levels))
    e256 = np.max(np.abs(c256.centroids[len(c256.centroids) // 2:] - levels))
    assert e256 < e128 < 0.03 * max(levels)


@pytest.mark.parametrize("d,bits", [(128, 1), (128, 2), (128, 3), (256, 2), (256, 4)])
def test_monte_carlo_sphere(d, bits):
    rng = np.random.default_rng(1234 + d + bits)
    n = 400_000 // d * 64
    g = rng.standard_normal((n // 64, d))
    x = (g / np.linalg.norm(g, axis=1, keepdims=True))[:, :64].ravel()  # coordinates of sphere points
    c = cb.lloyd_max(d, bits)
    t = c.boundaries.astype(np.float64) / math.sqrt(d)
    idx = np.searchsorted(t, x, side="right")
    cen = c.centroids_f64
    # cell probabilities
    edges = np.concatenate([[-1.0], t, [1.0]])
    for j in range(len(cen)):
        sel = idx == j
        p_mc = sel.mean()
        a, b = edges[j], edges[j + 1]
        if a >= 0:
            p = cb.cell_mass(d, a, b)
        elif b <= 0:
            p = cb.cell_mass(d, -b, -a)
        else:
            p = cb.cell_mass(d, 0, -a) + cb.cell_mass(d, 0, b)
        se = math.sqrt(p * (1 - p) / x.size)
        assert abs(p_mc - p) < 5 * se + 1e-12
        # centroid condition: conditional mean of the cell
        m_mc = x[sel].mean()
        se_m = x[sel].std() / math.sqrt(sel.sum())
        assert abs(m_mc - cen[j]) < 5 * se_m
    # MSE of the quantizer per coordinate, times d, is the unit-vector MSE
    mse_mc = d * np.mean((x - cen[idx]) ** 2)
    se = d * np.std((x - cen[idx]) ** 2) / math.sqrt(x.size)
    assert abs(mse_mc - c.mse_unit) < 5 * se


def test_one_bit_mean_abs():
    # b = 1: the centroid is E|X| of the sphere marginal
    d = 128
    rng = np.random.default_rng(7)
    g = rng.standard_normal((20000, d))
    x = (g / np.linalg.norm(g, axis=1, keepdims=True)).ravel()
    c = cb.lloyd_max(d, 1)
    assert abs(np.abs(x).mean() - c.centroids_f64[1]) < 5 * np.abs(x).std() / math.sqrt(x.size)
    assert abs(c.mse_unit - (1 - d * c.centroids_f64[1] ** 2)) < 1e-12


def test_symmetry_and_boundaries():
    for d in (128, 256):
        for bits in (1, 2, 3, 4):
            c = cb.lloyd_max(d, bits)
            L = 1 << bits
            assert c.centroids.dtype == np.float32 and c.boundaries.dtype == np.float32
            assert np.all(c.centroids[::-1] == -c.centroids)
            assert np.all(np.diff(c.centroids) > 0)
            assert c.boundaries[L // 2 - 1] == 0.0
            mid = ((c.centroids[:-1] + c.centroids[1:]) * np.float32(0.5)).astype(np.float32)
            assert np.array_equal(c.boundaries, mid)


def test_theorem1_ratios_match_readme():
    # [README] §Paper Validation, Thm 3 row: 2-bit = 0.70x, 3-bit = 0.82x of the bound
    d = 256
    r = {b: cb.lloyd_max(d, b).mse_unit / cb.theorem1_bound(b) for b in (1, 2, 3, 4)}
    assert abs(r[2] - 0.70) < 0.03
    assert abs(r[3] - 0.82) < 0.03
    assert all(v < 1.0 for v in r.values())
    for b in (1, 2, 3):
        ratio = cb.lloyd_max(d, b).mse_unit / cb.lloyd_max(d, b + 1).mse_unit
        assert 3.0 <= ratio <= 4.5


def test_fixed_point_by_adaptive_quadrature():
    """Centroid condition and MSE re-derived with adaptive quadrature of the
    unnormalised density (1 - x^2)^((d-3)/2), normalised numerically: this
    checks the closed-form first moment, the Beta-function cell masses and
    the density constant used by the solver."""
    from scipy.integrate import quad

    for d in (128, 256):
        e = (d - 3) / 2.0
        f = lambda x: (1.0 - x * x) ** e
        Z = 2.0 * quad(f, 0.0, 1.0, epsabs=0, epsrel=1e-13, limit=200)[0]
        for bits in (1, 2, 3, 4):
            c = cb.lloyd_max(d, bits)
            mu = c.centroids_f64[len(c.centroids_f64) // 2:]
            edges = np.concatenate([[0.0], 0.5 * (mu[:-1] + mu[1:]), [1.0]])
            mse = 0.0
            for j in range(len(mu)):
                a, b = edges[j], edges[j + 1]
                m0 = quad(f, a, b, epsabs=0, epsrel=1e-12, limit=200)[0] / Z
                m1 = quad(lambda x: x * f(x), a, b, epsabs=0, epsrel=1e-12, limit=200)[0] / Z
                assert abs(m1 / m0 - mu[j]) < 1e-9 * max(1.0, mu[j])
                mse += 2.0 * m0 * mu[j] ** 2
            assert abs((1.0 - d * mse) - c.mse_unit) < 1e-9
