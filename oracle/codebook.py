"""Lloyd-Max codebook for one coordinate of a randomly rotated unit vector.

[Reconstruction] §5 Step 2 says a coordinate of a randomly rotated unit vector
follows a "scaled Beta" law (the formula itself is a lost image); Step 3 says
it tends to N(0, 1/d); Step 4 says the codebook is the continuous k-means
(Lloyd-Max) solution on that density for 2^b buckets, computed offline.

Reading taken for the lost formula: the marginal of one coordinate X of a
uniform point on the unit sphere S^{d-1}, whose density on [-1, 1] is

    f_d(x) = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) * (1 - x^2)^((d-3)/2),

equivalently X^2 ~ Beta(1/2, (d-1)/2) with a symmetric random sign.

Cell probabilities use the regularised incomplete Beta function (scipy);
the cell first moment has the closed form

    int_a^b x f_d(x) dx = C_d / (d-1) * [(1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)].

The solver works on the positive half only, so the codebook is exactly
symmetric and the middle boundary is exactly 0.

Stored form (the reading of "RMS-scaled" keys): the
centroids are multiplied by sqrt(d) (unit-RMS coordinates, ~N(0,1)) and
rounded to float32; the decision boundaries are the float32 midpoints
(c_j + c_{j+1}) * 0.5f computed in float32 from the float32 centroids, and
these float32 boundaries are the ones every code decision uses.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
from scipy.special import betainc


@dataclass
class Codebook:
    d: int
    bits: int
    centroids: np.ndarray      # float32 [2^bits], ascending, RMS scale (sqrt(d) * c)
    boundaries: np.ndarray     # float32 [2^bits - 1], float32 midpoints
    centroids_f64: np.ndarray  # float64 [2^bits], unit-sphere scale (not RMS scaled)
    mse_unit: float            # E||u - u_hat||^2 for a unit vector u (float64 centroids)
    iterations: int


def pdf_constant(d: int) -> float:
    """C_d = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) for the sphere marginal."""
    return math.exp(math.lgamma(d / 2.0) - 0.5 * math.log(math.pi) - math.lgamma((d - 1) / 2.0))


def cell_mass(d: int, a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """P(a <= X <= b) for 0 <= a <= b <= 1 (X^2 ~ Beta(1/2, (d-1)/2), X symmetric)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return 0.5 * (betainc(0.5, (d - 1) / 2.0, b * b) - betainc(0.5, (d - 1) / 2.0, a * a))


def cell_first_moment(d: int, a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """int_a^b x f_d(x) dx (closed form)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    e = (d - 1) / 2.0
    return pdf_constant(d) / (d - 1) * ((1.0 - a * a) ** e - (1.0 - b * b) ** e)


def lloyd_max(d: int, bits: int, tol: float = 1e-13, max_iter: int = 100_000) -> Codebook:
    """Lloyd-Max iteration ([Reconstruction] §5 Step 4) on the sphere marginal.

    Alternates the two optimality conditions on the positive half-line:
    boundary = midpoint of neighbouring centroids, centroid = conditional mean
    of its cell.  Stops when the largest centroid change, in RMS units
    (sqrt(d) * c), is below ``tol``.
    """
    if d < 4 or bits < 1 or bits > 8:
        raise ValueError("need d >= 4 and 1 <= bits <= 8")
    half = 1 << (bits - 1)
    # start from Gaussian-limit quantiles of N(0, 1/d) on the positive side
    from scipy.stats import norm

    probs = 0.5 + (np.arange(half) + 0.5) / (2.0 * half)
    mu = norm.ppf(probs) / math.sqrt(d)
    it = 0
    for it in range(1, max_iter + 1):
        edges = np.concatenate([[0.0], 0.5 * (mu[:-1] + mu[1:]), [1.0]])
        new = cell_first_moment(d, edges[:-1], edges[1:]) / cell_mass(d, edges[:-1], edges[1:])
        delta = np.max(np.abs(new - mu)) * math.sqrt(d)
        mu = new
        if delta < tol:
            break
    else:
        raise RuntimeError("Lloyd-Max did not converge")
    edges = np.concatenate([[0.0], 0.5 * (mu[:-1] + mu[1:]), [1.0]])
    mass = cell_mass(d, edges[:-1], edges[1:])
    # MSE per unit vector: d * (E[X^2] - sum P_j mu_j^2), E[X^2] = 1/d, both halves
    mse_unit = 1.0 - d * 2.0 * float(np.sum(mass * mu * mu))

    full = np.concatenate([-mu[::-1], mu])
    c32 = (full * math.sqrt(d)).astype(np.float32)
    t32 = ((c32[:-1] + c32[1:]) * np.float32(0.5)).astype(np.float32)
    return Codebook(d=d, bits=bits, centroids=c32, boundaries=t32,
                    centroids_f64=full, mse_unit=mse_unit, iterations=it)


def theorem1_bound(bits: int) -> float:
    """Upper bound on the unit-vector MSE of TurboQuant_mse.

    The constant is a lost image in [Reconstruction] §5 ("Distortion-Rate
    Result"); the reading taken is sqrt(3)*pi/2 * 4^-b, whose ratios to the
    Lloyd-Max MSE reproduce the 2- and 3-bit figures of [README] §Paper
    Validation (0.70x, 0.82x).
    """
    return math.sqrt(3.0) * math.pi / 2.0 * 4.0 ** (-bits)
