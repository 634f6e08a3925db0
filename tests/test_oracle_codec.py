"""Pins of the oracle codec (TurboQuant_mse / TurboQuant_prod, packing).

* Packing: a hand-worked fixture and exact round trips.
* Zero-vector guard and the golden vectors of [Reconstruction] §13.
* MSE distortion: Monte Carlo E||u - u_hat||^2 over random unit vectors and
  random rotations equals the codebook's unit MSE (a wrong index mapping, a
  transposed rotation or a dropped sqrt(d) would inflate it) and stays below
  the Theorem 1 bound ([README] §Paper Validation: "within bounds").
* QJL ([Reconstruction] §6, [README] §Paper Validation "Relative bias <
  0.1%"): over 2^17 independent Gaussian S the residual estimate is unbiased
  to < 1e-3 relative, and its variance matches the closed form
  ||q||^2 ||r||^2 (pi/2 - rho^2) / d within 3% (which pins sqrt(pi/2)/d).
* Value cosine at d = 256, 2 bits: 0.940 ([README] §TQ Quantization
  Quality); sqrt(1 - D) for an MSE-optimal code.
"""

import math
import os

import numpy as np
import pytest

from oracle import codebook as CB
from oracle import codec as C
from oracle import transforms as T

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "packing_sign_magnitude.txt")


def test_golden_packing():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    for row in rows:
        bits = int(row[0])
        words = [int(w, 16) for w in row[2:]]
        if row[1] == "*":
            idx = np.zeros(32, dtype=np.int64)
            idx[[0, 5, 31]] = 1
        else:
            idx = np.arange(32) % int(row[1])
        packed = C.pack_codes(idx[None], bits)[0]
        assert packed.shape == (bits, 1)
        assert [int(w) for w in packed[:, 0]] == words
        assert np.array_equal(C.unpack_codes(packed[None], bits, 32)[0], idx)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [32, 128, 256])
def test_pack_round_trip(bits, d):
    idx = np.random.default_rng(bits * d).integers(0, 1 << bits, size=(50, d))
    w = C.pack_codes(idx, bits)
    assert w.dtype == np.uint32 and w.shape == (50, bits, d // 32)
    assert np.array_equal(C.unpack_codes(w, bits, d), idx)
    b = np.random.default_rng(1).integers(0, 2, size=(7, d)).astype(np.uint8)
    assert np.array_equal(C.unpack_bits(C.pack_bits(b), d), b)


def test_bucketize_ties_go_up():
    cb = CB.lloyd_max(128, 2)
    t = cb.boundaries.astype(np.float64)
    z = np.concatenate([t, np.nextafter(t, -np.inf), [-10.0, 10.0]])
    idx = C.bucketize(z, cb.boundaries)
    assert list(idx[:3]) == [1, 2, 3]
    assert list(idx[3:6]) == [0, 1, 2]
    assert list(idx[6:]) == [0, 3]


def _setup(d=128, kb=2, vb=2, kind=T.DENSE, seed=0):
    return {"kcb": CB.lloyd_max(d, kb), "vcb": CB.lloyd_max(d, vb),
            "rot": T.build_transform(kind, d, seed, 0, 0, 0),
            "S": T.build_transform(kind, d, seed, 0, 0, 2), "kind": kind}


def test_zero_vector_guard():
    s = _setup()
    x = np.zeros((2, 128))
    x[1, 3] = 5e-8  # below the 1e-7 threshold
    rec = C.quantize_prod(x, s["kind"], s["rot"], s["kcb"], s["S"])
    assert np.all(rec["norm"] == 0) and np.all(rec["rnorm"] == 0)
    assert np.all(rec["signs"])
    assert np.all(rec["idx"] == 2)  # code of z = 0 (ties go up)
    kh = C.dequantize_prod(rec["norm"], rec["rnorm"], rec["idx"], rec["signs"], s["kind"], s["rot"],
                           s["kcb"], s["S"])
    assert np.all(kh == 0)


def test_golden_vectors_fwht():
    # [Reconstruction] §13: e_1 spreads evenly; the outlier vector keeps its norm
    d = 128
    s = _setup(kind=T.FWHT)
    e1 = np.zeros((1, d))
    e1[0, 0] = 1.0
    rec = C.quantize_mse(e1, T.FWHT, s["rot"], s["kcb"])
    np.testing.assert_allclose(np.abs(rec["z"]), 1.0, rtol=0, atol=1e-15)
    out = np.full((1, d), 0.01)
    out[0, 0] = 100.0
    rec = C.quantize_mse(out, T.FWHT, s["rot"], s["kcb"])
    assert abs(rec["norm_f64"][0] - math.sqrt(100.0 ** 2 + 127 * 1e-4)) < 1e-12
    xh = C.dequantize_mse(rec["norm"], rec["idx"], T.FWHT, s["rot"], s["kcb"])
    err = np.sum((xh - out) ** 2) / np.sum(out ** 2)
    assert err < 3 * s["kcb"].mse_unit


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("kind", [T.DENSE, T.FWHT])
def test_mse_distortion_matches_codebook(bits, kind):
    d = 128
    cb = CB.lloyd_max(d, bits)
    rng = np.random.default_rng(100 + bits)
    errs = []
    for seed in range(8):
        rot = T.build_transform(kind, d, seed, 0, 0, 1)
        x = rng.standard_normal((1500, d)) * rng.lognormal(0, 1, size=(1500, 1))
        rec = C.quantize_mse(x, kind, rot, cb)
        xh = C.dequantize_mse(rec["norm"], rec["idx"], kind, rot, cb)
        errs.append(np.sum((xh - x) ** 2, axis=1) / np.sum(x ** 2, axis=1))
    e = np.concatenate(errs)
    se = e.std() / math.sqrt(e.size)
    assert abs(e.mean() - cb.mse_unit) < 5 * se + 1e-6 * 0
    assert e.mean() < CB.theorem1_bound(bits)


def test_qjl_unbiased_and_variance():
    d = 32
    rng = np.random.default_rng(42)
    r = rng.standard_normal(d)
    r *= 0.3 / np.linalg.norm(r)
    q = r / np.linalg.norm(r) * 2.0 + 0.05 * rng.standard_normal(d)  # rho close to 1
    true = float(q @ r)
    est = []
    for _ in range(64):
        S = rng.standard_normal((2048, d, d))
        signs = C.sketch(r, S) >= 0
        est.append(C.qjl_estimate(q, np.linalg.norm(r), signs, S))
    est = np.concatenate(est)
    assert est.size == 1 << 17
    rel_bias = est.mean() / true - 1
    assert abs(rel_bias) < 1e-3
    rho = true / (np.linalg.norm(q) * np.linalg.norm(r))
    var = (q @ q) * (r @ r) * (math.pi / 2 - rho ** 2) / d
    assert abs(est.var() / var - 1) < 0.03


def test_key_estimator_unbiased_through_quantize_prod():
    # E_S[<q', y_hat> + sqrt(pi/2)/d gamma <S q', s>] = <q', y> for a fixed key
    d = 32
    s = _setup(d=d, kb=2)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, d))
    q = rng.standard_normal(d)
    rec = C.quantize_mse(x, T.DENSE, s["rot"], s["kcb"])
    r = rec["y"][0] - rec["yhat"][0]
    qr = T.rotate(T.DENSE, s["rot"], q[None])[0]
    est = []
    for _ in range(16):
        S = rng.standard_normal((4096, d, d))
        recs = C.quantize_prod(np.repeat(x, 1, 0), T.DENSE, s["rot"], s["kcb"], S[0])
        assert np.array_equal(recs["signs"][0], C.sketch(r, S[0]) >= 0)
        est.append(qr @ rec["yhat"][0] + C.qjl_estimate(qr, np.linalg.norm(r), C.sketch(r, S) >= 0, S))
    est = np.concatenate(est)
    true = qr @ rec["y"][0]
    se = est.std() / math.sqrt(est.size)
    assert abs(est.mean() - true) < 5 * se


def test_value_cosine_two_bits_d256():
    d = 256
    cb = CB.lloyd_max(d, 2)
    rot = T.build_transform(T.FWHT, d, 0, 0, 0, 1)
    x = np.random.default_rng(9).standard_normal((4000, d))
    rec = C.quantize_mse(x, T.FWHT, rot, cb)
    xh = C.dequantize_mse(rec["norm"], rec["idx"], T.FWHT, rot, cb)
    cos = np.sum(x * xh, 1) / np.linalg.norm(x, axis=1) / np.linalg.norm(xh, axis=1)
    assert abs(cos.mean() - 0.940) < 0.0015
    cb4 = CB.lloyd_max(d, 4)
    rec = C.quantize_mse(x, T.FWHT, rot, cb4)
    xh = C.dequantize_mse(rec["norm"], rec["idx"], T.FWHT, rot, cb4)
    cos4 = np.sum(x * xh, 1) / np.linalg.norm(x, axis=1) / np.linalg.norm(xh, axis=1)
    assert 0.994 < cos4.mean() < 0.998  # [README] reports 0.997 for its own 4-bit value codec


# ----------------------------------------------------------------------------- EDEN / renormalized keys

def _pair(rng, n, d, rho):
    """n pairs (y, q') of unit vectors with <y, q'> = rho and (y, q') uniform
    over such pairs: the joint law of (Pi x, Pi q) under a Haar rotation."""
    y = rng.standard_normal((n, d))
    y /= np.linalg.norm(y, axis=1, keepdims=True)
    w = rng.standard_normal((n, d))
    w -= np.sum(w * y, axis=1, keepdims=True) * y
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    return y, rho * y + math.sqrt(1 - rho * rho) * w


def test_length_renormalized_keys_are_unbiased():
    """TurboVec's per-vector correction norm / <y, y_hat> ([Reconstruction] §12
    item 2, §13 step 6) restores unbiasedness: over uniformly rotated pairs of
    correlation rho the mean estimate n s <q', y_hat> equals n rho, where the
    uncorrected code shrinks it.  Checked for 1 to 3 bits and a key norm of 3."""
    d, n, rho = 64, 20000, 0.6
    rng = np.random.default_rng(7)
    y, q = _pair(rng, n, d, rho)
    for bits in (1, 2, 3):
        cb = CB.lloyd_max(d, bits)
        rec = C.quantize_scaled(3.0 * y, T.DENSE, np.eye(d), cb, C.KEY_RENORM)
        np.testing.assert_allclose(rec["norm_f64"], 3.0, rtol=1e-12)
        est = rec["norm_f64"] * rec["scale"] * np.sum(q * rec["yhat"], axis=1)
        assert abs(est.mean() - 3.0 * rho) < 4 * est.std() / math.sqrt(n), bits
        plain = rec["norm_f64"] * np.sum(q * rec["yhat"], axis=1)
        assert 3.0 * rho - plain.mean() > 10 * plain.std() / math.sqrt(n), bits
    z = C.quantize_scaled(np.zeros((1, d)), T.FWHT, T.build_transform(T.FWHT, d, 0, 0, 0, 0),
                          CB.lloyd_max(d, 2), C.KEY_RENORM)
    assert z["scale"][0] == 0 and z["norm"][0] == 0


def test_length_renormalization_is_the_eden_scale():
    """The page relates TurboVec's correction to EDEN's unbiased scalar: with the
    norm kept in its own field both stored scales agree on arbitrary keys."""
    d = 128
    cb = CB.lloyd_max(d, 2)
    rot = T.build_transform(T.FWHT, d, 0, 0, 0, 0)
    x = np.random.default_rng(4).standard_normal((64, d)) * np.exp(np.random.default_rng(5).standard_normal(d))
    a = C.quantize_scaled(x, T.FWHT, rot, cb, C.KEY_RENORM)
    b = C.quantize_scaled(x, T.FWHT, rot, cb, C.KEY_EDEN)
    np.testing.assert_allclose(a["scale"], b["scale"], rtol=1e-12)


def test_eden_scale_is_unbiased_and_plain_code_is_not():
    """E <q', s y_hat> = <q', y> over random rotations (rotation = identity on
    a uniformly rotated pair); the same code with s = 1 underestimates."""
    d, n, rho = 64, 20000, 0.6
    rng = np.random.default_rng(5)
    y, q = _pair(rng, n, d, rho)
    cb = CB.lloyd_max(d, 2)
    eye = np.eye(d)
    rec = C.quantize_scaled(y, T.DENSE, eye, cb, C.KEY_EDEN)
    est = np.sum(q * rec["scale"][:, None] * rec["yhat"], axis=1)
    se = est.std() / math.sqrt(n)
    assert abs(est.mean() - rho) < 4 * se
    plain = np.sum(q * rec["yhat"], axis=1)
    assert rho - plain.mean() > 10 * plain.std() / math.sqrt(n)


def test_one_bit_eden_has_275x_lower_variance_than_qjl():
    """1-bit estimators of <q, x> for orthogonal unit q, x: EDEN (1-bit code,
    unbiased scale) has variance (pi/2 - 1)/d, the QJL sign sketch of the whole
    vector pi/2/d, a ratio of 2.75 ([Reconstruction] §12.2)."""
    d, n = 128, 3000
    rng = np.random.default_rng(6)
    y, q = _pair(rng, n, d, 0.0)
    cb = CB.lloyd_max(d, 1)
    rec = C.quantize_scaled(y, T.DENSE, np.eye(d), cb, C.KEY_EDEN)
    eden = np.sum(q * rec["scale"][:, None] * rec["yhat"], axis=1)
    S = rng.standard_normal((n, d, d))
    qjl = C.qjl_estimate(q, 1.0, C.sketch(y, S) >= 0, S)
    assert abs(eden.var() * d / (math.pi / 2 - 1) - 1) < 0.08
    assert abs(qjl.var() * d / (math.pi / 2) - 1) < 0.08
    assert 2.45 < qjl.var() / eden.var() < 3.05


def test_structured_sketch_estimator():
    """S = H diag(sigma_S): a residual on one coordinate e_k gives the closed form sqrt(pi/2) q_k
    (sign(S e_k) is column k of S and S^T S = d I); for spread (Gaussian) residuals the estimate is
    unbiased -- Sr / sqrt(d) is then an orthonormal transform of a Gaussian vector -- and with
    orthogonal rows its distortion stays below the dense Gaussian sketch's."""
    d = 128
    rng = np.random.default_rng(5)
    sig = T.build_transform(T.FWHT, d, 1, 0, 0, T.ROLE_QJL_SIGNS)
    S = T.structured_qjl_matrix(sig, d)
    q = rng.standard_normal(d)
    for k in (0, 7, 100):
        e = np.zeros(d)
        e[k] = 1.0
        est = C.qjl_estimate(q, 1.0, (S @ e) >= 0, S)
        assert abs(est - math.sqrt(math.pi / 2) * q[k]) < 1e-12
    n = 20000
    r = rng.standard_normal((n, d))
    qq = r + 2.0 * rng.standard_normal((n, d))
    true = np.sum(qq * r, axis=1)
    dist = {}
    for name, M in (("srht", S), ("gauss", T.build_transform(T.FWHT, d, 1, 0, 0, T.ROLE_QJL).astype(np.float64))):
        signs = (r @ M.T) >= 0
        est = C.qjl_constant(d) * np.linalg.norm(r, axis=1) * np.sum((qq @ M.T) * np.where(signs, 1.0, -1.0), axis=1)
        slope = np.sum(est * true) / np.sum(true * true)
        err = (est - true) ** 2 / (np.sum(qq * qq, axis=1) * np.sum(r * r, axis=1))
        dist[name] = d * err.mean()
        se = math.sqrt(np.mean((est - slope * true) ** 2) / np.sum(true * true))
        assert abs(slope - 1.0) < 5 * se + 1e-3, (name, slope, se)
    assert dist["srht"] < dist["gauss"]
