"""Pins of the oracle's generator and rotations.

* SplitMix64: the published first outputs of the reference generator for
  seed 0.
* Box-Muller: moments of the standard normal.
* Dense rotation: orthogonality, and Haar-ness (the column-sign fix of the
  QR factor): the first column of a Haar matrix is uniform on the sphere.
* Walsh-Hadamard: the Sylvester recursion H_2k = [[H, H], [H, -H]] built
  independently by Kronecker products, H H = d I, and the golden vector of
  [Reconstruction] §13 (the basis vector e_1 spreads to +-1/sqrt(d) in every
  coordinate).
"""

import math

import numpy as np
import pytest

from oracle import rng as R
from oracle import transforms as T


def test_splitmix64_published_outputs():
    g = R.SplitMix64(0)
    got = [g.next_u64() for _ in range(4)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]
    g2 = R.SplitMix64(0)
    assert [int(x) for x in g2.outputs(4)] == got
    assert g2.state == g.state


def test_box_muller_moments():
    z = R.SplitMix64(R.stream_state(3, 0, 0, 0)).normals(1 << 20)
    n = z.size
    assert abs(z.mean()) < 5 / math.sqrt(n)
    assert abs(z.var() - 1) < 5 * math.sqrt(2 / n)
    assert abs(np.mean(z ** 4) - 3) < 5 * math.sqrt(96 / n)
    assert abs(np.mean(z ** 3)) < 5 * math.sqrt(15 / n)


def test_uniform_range_and_rademacher_balance():
    g = R.SplitMix64(R.stream_state(5, 1, 2, 3))
    u = g.uniforms(1 << 18)
    assert u.min() >= 0 and u.max() < 1
    s = R.SplitMix64(R.stream_state(5, 1, 2, 3)).rademacher(1 << 18)
    assert set(np.unique(s)) == {-1.0, 1.0}
    assert abs(s.mean()) < 5 / math.sqrt(s.size)


@pytest.mark.parametrize("d", [32, 128, 256])
def test_dense_rotation_orthogonal(d):
    P = T.haar_rotation_f64(d, 0, 0, 1, 0)
    assert np.max(np.abs(P.T @ P - np.eye(d))) < 1e-13
    P32 = T.build_transform(T.DENSE, d, 0, 0, 1, 0).astype(np.float64)
    assert np.max(np.abs(P32.T @ P32 - np.eye(d))) < 1e-6


def test_dense_rotation_is_haar():
    # Pi e_1 (first column) must be uniform on the sphere: E x_1 = 0,
    # E x_1^2 = 1/d, E x_1^4 = 3 / (d (d + 2)).  Without the sign fix of the
    # QR factor, x_1 = Pi_11 would be biased.
    d, n = 16, 6000
    x = np.array([T.haar_rotation_f64(d, s, 0, 0, 0)[:, 0] for s in range(n)])
    m1 = x[:, 0].mean()
    assert abs(m1) < 5 * math.sqrt(1 / d / n)
    assert abs(np.mean(x ** 2) - 1 / d) < 0.03 / d
    assert abs(np.mean(x ** 4) - 3 / (d * (d + 2))) < 0.06 * 3 / (d * (d + 2))
    # all diagonal entries unbiased
    diag = np.array([np.diag(T.haar_rotation_f64(d, s, 0, 0, 0)) for s in range(2000)])
    assert np.max(np.abs(diag.mean(axis=0))) < 5 * math.sqrt(1 / d / 2000)


@pytest.mark.parametrize("d", [2, 8, 128, 256])
def test_walsh_hadamard_matches_sylvester(d):
    H = np.array([[1.0]])
    while H.shape[0] < d:
        H = np.kron(np.array([[1.0, 1.0], [1.0, -1.0]]), H)
    assert np.array_equal(T.walsh_hadamard(d), H)
    assert np.array_equal(H @ H, d * np.eye(d))


@pytest.mark.parametrize("d", [128, 256])
def test_fwht_rotation_golden_basis_vector(d):
    sig = T.build_transform(T.FWHT, d, 0, 0, 0, 0)
    assert set(np.unique(sig)) <= {-1.0, 1.0}
    e1 = np.zeros(d)
    e1[0] = 1.0
    y = T.rotate(T.FWHT, sig, e1[None])[0]
    np.testing.assert_array_equal(np.abs(y), np.full(d, 1 / math.sqrt(d)))
    assert np.all(np.sign(y) == sig[0])
    # orthogonal and exactly invertible on integers (H H = d I)
    P = T.rotation_matrix(T.FWHT, sig, d)
    assert np.max(np.abs(P.T @ P - np.eye(d))) < 1e-14
    x = np.random.default_rng(0).integers(-50, 50, size=(4, d)).astype(np.float64)
    back = T.rotate_inverse(T.FWHT, sig, T.rotate(T.FWHT, sig, x))
    assert np.max(np.abs(back - x)) < 1e-12


def test_seed_determinism_and_streams():
    a = T.build_transform(T.DENSE, 64, 7, 3, 1, 0)
    b = T.build_transform(T.DENSE, 64, 7, 3, 1, 0)
    assert np.array_equal(a, b)
    for other in [(8, 3, 1, 0), (7, 4, 1, 0), (7, 3, 2, 0), (7, 3, 1, 1)]:
        assert not np.array_equal(a, T.build_transform(T.DENSE, 64, *other))
    S = T.build_transform(T.FWHT, 64, 7, 3, 1, T.ROLE_QJL)
    assert S.shape == (64, 64) and S.dtype == np.float32
    assert abs(S.astype(np.float64).var() - 1) < 0.1


@pytest.mark.parametrize("d", [64, 128])
def test_structured_qjl_matrix(d):
    """S = H diag(sigma_S): entries +-1 and S S^T = d I exactly; the signs come from their own stream."""
    sig = T.build_transform(T.FWHT, d, 3, 2, 1, T.ROLE_QJL_SIGNS)
    assert sig.shape == (d,) and set(np.unique(sig)) <= {-1.0, 1.0}
    assert not np.array_equal(sig, T.build_transform(T.FWHT, d, 3, 2, 1, T.ROLE_KEY_ROT))
    assert np.array_equal(sig, T.build_transform(T.DENSE, d, 3, 2, 1, T.ROLE_QJL_SIGNS))
    S = T.structured_qjl_matrix(sig, d)
    assert np.array_equal(np.abs(S), np.ones((d, d)))
    assert np.array_equal(S @ S.T, d * np.eye(d))
    # column j is sigma_j times column j of the Sylvester matrix
    H = T.walsh_hadamard(d)
    assert np.array_equal(S[:, 5], sig[5] * H[:, 5])
