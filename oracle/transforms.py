"""Random rotations and the QJL matrix, drawn from the oracle's own SplitMix64.

* Dense rotation Pi ([Reconstruction] §5 Step 2: "a dense, random orthogonal
  matrix ... typically via the QR decomposition of a standard Gaussian
  matrix"): G is d x d i.i.d. N(0,1) filled row-major; G = QR; the columns of
  Q are multiplied by sign(R_jj) so that Pi is Haar distributed; y = Pi u.
* Structured rotation ([Design study] §Dense and structured transform
  comparison; [Reconstruction] §9 "Fast Walsh-Hadamard + Rademacher", §13
  reference logic: signs first, then the Walsh-Hadamard butterfly, then
  division by sqrt(d)):  Pi u = H (sigma * u) / sqrt(d), H the unnormalised
  Sylvester-ordered Walsh-Hadamard matrix H_ij = (-1)^popcount(i & j).
* QJL matrix S ([Reconstruction] §6 "The 1-Bit QJL Transform": i.i.d. standard
  normal entries), d x d (m = d rows; reading of the lost row count, matching
  the sqrt(pi/2)/d constant of the estimator), row-major, float32.
* Structured QJL matrix (next-row option; [Design study] §Candidate key and
  value algorithms, the structured key arm with an optional residual QJL
  stage, "another transform-domain residual stage" costing p log p): the
  subsampled-randomised-Hadamard form with all d rows kept,
  S = H diag(sigma_S), entries +-1, rows orthogonal with squared norm d like
  the expected squared norm of a Gaussian row.  Reading: the estimator keeps
  its Gaussian constant sqrt(pi/2)/d; for a residual spread over the
  coordinates (the rotated basis) the Rademacher sums <s_i, r> are close to
  Gaussian, so the estimate is close to unbiased, not exactly unbiased (a
  residual on one coordinate is over-estimated by sqrt(pi/2), pinned).

Roles: 0 = key rotation, 1 = value rotation, 2 = QJL matrix S, 3 = the signs
sigma_S of the structured QJL matrix.
Stored forms are float32: Pi as d*d row-major, sigma as d values of +-1.
"""

from __future__ import annotations

import numpy as np

from .rng import SplitMix64, stream_state

DENSE = 0
FWHT = 1

ROLE_KEY_ROT = 0
ROLE_VALUE_ROT = 1
ROLE_QJL = 2
ROLE_QJL_SIGNS = 3


def gaussian_matrix(d: int, seed: int, layer: int, head: int, role: int) -> np.ndarray:
    g = SplitMix64(stream_state(seed, layer, head, role))
    return g.normals(d * d).reshape(d, d)


def haar_rotation_f64(d: int, seed: int, layer: int, head: int, role: int) -> np.ndarray:
    """Dense Haar rotation in float64 (before the float32 cast)."""
    G = gaussian_matrix(d, seed, layer, head, role)
    Q, R = np.linalg.qr(G)
    s = np.sign(np.diag(R))
    s[s == 0] = 1.0
    return Q * s[None, :]


def rademacher_signs(d: int, seed: int, layer: int, head: int, role: int) -> np.ndarray:
    g = SplitMix64(stream_state(seed, layer, head, role))
    return g.rademacher(d)


def walsh_hadamard(d: int) -> np.ndarray:
    """Unnormalised Sylvester Walsh-Hadamard matrix from its definition."""
    if d & (d - 1):
        raise ValueError("d must be a power of two")
    i = np.arange(d)
    parity = np.zeros((d, d), dtype=np.int64)
    a = i[:, None] & i[None, :]
    while np.any(a):
        parity ^= a & 1
        a = a >> 1
    return np.where(parity == 1, -1.0, 1.0)


def build_transform(kind: int, d: int, seed: int, layer: int, head: int, role: int) -> np.ndarray:
    """The stored float32 array for (kind, role): d*d matrix or d signs."""
    if role == ROLE_QJL:
        return gaussian_matrix(d, seed, layer, head, role).astype(np.float32)
    if role == ROLE_QJL_SIGNS:
        return rademacher_signs(d, seed, layer, head, role).astype(np.float32)
    if kind == DENSE:
        return haar_rotation_f64(d, seed, layer, head, role).astype(np.float32)
    if kind == FWHT:
        return rademacher_signs(d, seed, layer, head, role).astype(np.float32)
    raise ValueError("unknown transform kind")


def rotation_matrix(kind: int, stored: np.ndarray, d: int) -> np.ndarray:
    """The d x d rotation Pi (float64) represented by a stored float32 array."""
    if kind == DENSE:
        return np.asarray(stored, dtype=np.float64).reshape(d, d)
    sigma = np.asarray(stored, dtype=np.float64).reshape(d)
    return walsh_hadamard(d) * sigma[None, :] / np.sqrt(d)


def rotate(kind: int, stored: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y = Pi x for the rows of x ([..., d]) in float64."""
    d = x.shape[-1]
    return np.asarray(x, dtype=np.float64) @ rotation_matrix(kind, stored, d).T


def rotate_inverse(kind: int, stored: np.ndarray, y: np.ndarray) -> np.ndarray:
    """x = Pi^T y for the rows of y ([..., d]) in float64."""
    d = y.shape[-1]
    return np.asarray(y, dtype=np.float64) @ rotation_matrix(kind, stored, d)


def structured_qjl_matrix(stored_signs: np.ndarray, d: int) -> np.ndarray:
    """S = H diag(sigma_S) (float64, entries +-1) from the stored d signs."""
    sigma = np.asarray(stored_signs, dtype=np.float64).reshape(d)
    return walsh_hadamard(d) * sigma[None, :]
