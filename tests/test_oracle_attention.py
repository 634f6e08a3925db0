"""Pins of the oracle decode attention.

* Window only (all tokens float16, unrotated): equals textbook softmax
  attention to 1e-12.
* Two routes: scoring in the rotated domain ([Design study] §Transform
  placement, q^T k = (T q)^T (T k); value accumulation in the transform
  domain with one inverse transform per head) equals textbook attention over
  explicitly dequantized keys k_hat = n Pi^T (y_hat + sqrt(pi/2)/d gamma S^T s)
  and values v_hat = m Pi_v^T y_hat, with GQA written as repeated KV heads.
* Quality against exact attention improves with the bit width
  ([Reconstruction] §15 Experiment A: attention-distribution KL divergence).
"""

import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import codebook as CB
from oracle import codec as C
from oracle import transforms as T


def _params(d, Hkv, kind, kb, vb, seed=0):
    return {
        "kind": kind,
        "k_rot": [T.build_transform(kind, d, seed, 0, h, 0) for h in range(Hkv)],
        "v_rot": [T.build_transform(kind, d, seed, 0, h, 1) for h in range(Hkv)],
        "qjl_s": [T.build_transform(kind, d, seed, 0, h, 2) for h in range(Hkv)],
        "k_cb": CB.lloyd_max(d, kb), "v_cb": CB.lloyd_max(d, vb), "key_qjl": True,
    }


def _compress(K, V, p):
    Hkv = K.shape[0]
    comp = {k: [] for k in ("knorm", "krnorm", "kidx", "ksigns", "vnorm", "vidx")}
    for g in range(Hkv):
        kr = C.quantize_prod(K[g], p["kind"], p["k_rot"][g], p["k_cb"], p["qjl_s"][g])
        vr = C.quantize_mse(V[g], p["kind"], p["v_rot"][g], p["v_cb"])
        comp["knorm"].append(kr["norm"]); comp["krnorm"].append(kr["rnorm"])
        comp["kidx"].append(kr["idx"]); comp["ksigns"].append(kr["signs"])
        comp["vnorm"].append(vr["norm"]); comp["vidx"].append(vr["idx"])
    return {k: np.stack(v) for k, v in comp.items()}


def _explicit(comp, p):
    Hkv = comp["knorm"].shape[0]
    Kh = np.stack([C.dequantize_prod(comp["knorm"][g], comp["krnorm"][g], comp["kidx"][g], comp["ksigns"][g],
                                     p["kind"], p["k_rot"][g], p["k_cb"], p["qjl_s"][g]) for g in range(Hkv)])
    Vh = np.stack([C.dequantize_mse(comp["vnorm"][g], comp["vidx"][g], p["kind"], p["v_rot"][g], p["v_cb"])
                   for g in range(Hkv)])
    return Kh, Vh


def _textbook(q, K, V, scale):
    Hq = q.shape[0]
    G = Hq // K.shape[0]
    Ke, Ve = np.repeat(K, G, axis=0), np.repeat(V, G, axis=0)
    l = scale * np.einsum("htd,hd->ht", Ke, q)
    m = l.max(axis=1, keepdims=True)
    e = np.exp(l - m)
    return {"out": np.einsum("ht,htd->hd", e / e.sum(1, keepdims=True), Ve),
            "lse": m[:, 0] + np.log(e.sum(1)), "scores": l}


def test_window_only_is_exact_attention():
    rng = np.random.default_rng(0)
    Hkv, Hq, Tw, d = 2, 6, 40, 64
    K = rng.standard_normal((Hkv, Tw, d)).astype(np.float16)
    V = rng.standard_normal((Hkv, Tw, d)).astype(np.float16)
    q = rng.standard_normal((Hq, d))
    p = _params(d, Hkv, T.FWHT, 2, 2)
    got = A.decode_one(q, None, K, V, p, 1 / math.sqrt(d))
    ref = _textbook(q, K.astype(np.float64), V.astype(np.float64), 1 / math.sqrt(d))
    for k in ("out", "lse", "scores"):
        np.testing.assert_allclose(got[k], ref[k], rtol=0, atol=1e-12)
    ex = A.exact_attention(q, K, V, 1 / math.sqrt(d))
    np.testing.assert_allclose(ex["out"], ref["out"], rtol=0, atol=1e-12)


def test_zero_padded_head_is_the_unpadded_attention():
    """A head shorter than the transform size, zero-padded (keys, values and
    query): scores, lse and the first head_dim output coordinates are those of
    textbook attention on the unpadded vectors; the padded outputs are zero;
    and padding keeps norms and inner products."""
    from oracle import codec as C

    rng = np.random.default_rng(3)
    Hkv, Hq, Tw, dh, d = 2, 6, 30, 40, 64
    K = rng.standard_normal((Hkv, Tw, dh)).astype(np.float16)
    V = rng.standard_normal((Hkv, Tw, dh)).astype(np.float16)
    q = rng.standard_normal((Hq, dh))
    Kp, Vp, qp = (C.pad_head(x, d) for x in (K, V, q))
    assert Kp.shape == (Hkv, Tw, d) and not Kp[..., dh:].any()
    np.testing.assert_array_equal(np.linalg.norm(Kp, axis=-1), np.linalg.norm(K.astype(np.float64), axis=-1))
    p = _params(d, Hkv, T.FWHT, 2, 2)
    got = A.decode_one(qp, None, Kp.astype(np.float16), Vp.astype(np.float16), p, 1 / math.sqrt(dh))
    ref = _textbook(q, K.astype(np.float64), V.astype(np.float64), 1 / math.sqrt(dh))
    for k in ("lse", "scores"):
        np.testing.assert_allclose(got[k], ref[k], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["out"][:, :dh], ref["out"], rtol=0, atol=1e-12)
    assert not got["out"][:, dh:].any()
    with pytest.raises(ValueError):
        C.pad_head(np.zeros((2, 70)), 64)


@pytest.mark.parametrize("kind", [T.DENSE, T.FWHT])
@pytest.mark.parametrize("bits", [(2, 2), (3, 4)])
def test_rotated_domain_equals_explicit_dequantization(kind, bits):
    rng = np.random.default_rng(1)
    Hkv, Hq, Tc, Tw, d = 2, 4, 96, 7, 128
    K = rng.standard_normal((Hkv, Tc + Tw, d)) * np.exp(rng.standard_normal((Hkv, 1, d)))
    V = rng.standard_normal((Hkv, Tc + Tw, d))
    q = rng.standard_normal((Hq, d))
    p = _params(d, Hkv, kind, *bits)
    comp = _compress(K[:, :Tc], V[:, :Tc], p)
    wk, wv = K[:, Tc:].astype(np.float16), V[:, Tc:].astype(np.float16)
    got = A.decode_one(q, comp, wk, wv, p, 1 / math.sqrt(d))
    Kh, Vh = _explicit(comp, p)
    ref = _textbook(q, np.concatenate([Kh, wk.astype(np.float64)], 1),
                    np.concatenate([Vh, wv.astype(np.float64)], 1), 1 / math.sqrt(d))
    for k in ("out", "lse", "scores"):
        np.testing.assert_allclose(got[k], ref[k], rtol=0, atol=1e-9)


def test_quality_improves_with_bits():
    rng = np.random.default_rng(2)
    Hkv, Hq, Tc, d = 2, 4, 512, 128
    K = rng.standard_normal((Hkv, Tc, d))
    V = rng.standard_normal((Hkv, Tc, d))
    q = rng.standard_normal((Hq, d)) * 2
    ex = A.exact_attention(q, K, V, 1 / math.sqrt(d))
    errs, kls = [], []
    for b in (2, 3, 4):
        p = _params(d, Hkv, T.FWHT, b, b)
        got = A.decode_one(q, _compress(K, V, p), None, None, p, 1 / math.sqrt(d))
        errs.append(np.max(np.abs(got["out"] - ex["out"])))
        lp = got["scores"] - got["lse"][:, None]
        le = ex["scores"] - ex["lse"][:, None]
        kls.append(np.mean(np.sum(np.exp(le) * (le - lp), axis=1)))
    assert errs[0] > errs[1] > errs[2]
    assert kls[0] > kls[1] > kls[2] >= 0
