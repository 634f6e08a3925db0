"""Pins of the KIVI-like control arm ([Design study] §Candidate key and value
algorithms, arm 3: per-channel keys, per-token values, FP16 window).

* Worked examples of asymmetric min-max codes (exact grids, ties up).
* A constant group has scale 0 and reconstructs to its float16 value.
* Every reconstruction lies within half a step plus the float16 roundings
  of zero and scale.
* Keys group by channel, values by token: the key quantizer of a page is the
  value quantizer of its transpose.
* Packing round trips and the record size of the page format.
* Decode over a KIVI cache equals textbook attention over the dequantized
  keys and values plus the float16 window.
"""

import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import kivi as KV


def test_worked_examples():
    r = KV.quantize_values(np.array([[0.0, 1.0, 2.0, 3.0]]), 2)
    assert r["scale"][0] == 1.0 and r["zero"][0] == 0.0
    assert r["codes"][0].tolist() == [0, 1, 2, 3]
    assert np.array_equal(KV.dequantize_values(r), [[0.0, 1.0, 2.0, 3.0]])
    r = KV.quantize_values(np.array([[0.0, 0.5, 1.0, 1.5, 3.0]]), 2)   # s = 1: 0.5 and 1.5 are ties, up
    assert r["codes"][0].tolist() == [0, 1, 1, 2, 3]
    assert r["margin"][0, 1] == 0 and r["margin"][0, 3] == 0
    r = KV.quantize_values(np.array([[-2.0, 0.0, 13.0]]), 4)   # s = 1, z = -2
    assert r["codes"][0].tolist() == [0, 2, 15]
    r = KV.quantize_values(np.array([[1.0, 2.0, 1.4, 1.6]]), 1)  # s = 1: codes 0 / 1 around 1.5
    assert r["codes"][0].tolist() == [0, 1, 0, 1]


def test_constant_group_and_scale_rounding():
    x = np.full((1, 8), 0.1)
    r = KV.quantize_values(x, 2)
    assert r["scale"][0] == 0 and np.all(r["codes"] == 0)
    assert np.all(KV.dequantize_values(r) == np.float64(np.float16(0.1)))
    # the scale is formed in float32, then rounded to float16
    mn, mx = np.float32(0.1), np.float32(1.7)
    s, z = KV.scale_zero(np.array([mn]), np.array([mx]), 2)
    assert s[0] == np.float16(np.float32(mx - mn) / np.float32(3)) and z[0] == np.float16(mn)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_reconstruction_error_bound(bits):
    rng = np.random.default_rng(bits)
    X = rng.standard_normal((400, 128)) * rng.lognormal(0, 1, (400, 1))
    r = KV.quantize_values(X, bits)
    err = np.abs(KV.dequantize_values(r) - X)
    bound = KV.error_bound(X, r["scale"][:, None], r["zero"][:, None], X.min(1, keepdims=True),
                           X.max(1, keepdims=True), bits)
    assert np.all(err <= bound * (1 + 1e-12))
    assert r["codes"].min() == 0 and r["codes"].max() == (1 << bits) - 1
    # within the range the error is at most half a step (codes strictly inside the clamps)
    inner = (r["codes"] > 0) & (r["codes"] < (1 << bits) - 1)
    assert np.all(err[inner] <= r["scale"][:, None].astype(np.float64).repeat(128, 1)[inner] / 2 + 1e-12)


def test_keys_group_by_channel_values_by_token():
    rng = np.random.default_rng(0)
    K = rng.standard_normal((16, 128)) * np.exp(rng.standard_normal(128))
    kr = KV.quantize_key_page(K, 2)
    vr = KV.quantize_values(K.T, 2)
    assert np.array_equal(kr["scale"], vr["scale"]) and np.array_equal(kr["zero"], vr["zero"])
    assert np.array_equal(kr["codes"], vr["codes"].T)
    with pytest.raises(ValueError):
        KV.quantize_keys(K[:15], 2)


@pytest.mark.parametrize("d,kb,vb", [(128, 2, 2), (256, 4, 2), (128, 1, 4)])
def test_page_layout_and_round_trip(d, kb, vb):
    lay = KV.subblock_layout(d, kb, vb)
    assert all(v % 16 == 0 for v in lay.values())
    assert lay["bytes"] == 16 * KV.record_bytes(d, kb, vb)
    rng = np.random.default_rng(d + kb)
    H, npg = 2, 3
    pool = np.zeros(npg * H * lay["bytes"], np.uint8)
    truth = {}
    for p in range(npg):
        for h in range(H):
            K = rng.standard_normal((16, d))
            V = rng.standard_normal((16, d))
            kr, vr = KV.quantize_key_page(K, kb), KV.quantize_values(V, vb)
            truth[p, h] = (kr, vr)
            KV.write_page(pool, lay, H, p, h, d, kb, vb, kr, vr)
    for (p, h), (kr, vr) in truth.items():
        g = KV.read_page(pool, lay, H, p, h, d, kb, vb)
        assert np.array_equal(g["kscale"], kr["scale"]) and np.array_equal(g["kzero"], kr["zero"])
        assert np.array_equal(g["kcodes"], kr["codes"]) and np.array_equal(g["vcodes"], vr["codes"])
        assert np.array_equal(g["vscale"], vr["scale"]) and np.array_equal(g["vzero"], vr["zero"])
    # 2-bit keys and values at d = 128: 100 bytes a token-head (32 of them the page's key scales and zeros)
    assert KV.record_bytes(128, 2, 2) == 100


def test_packing_worked_example():
    c = np.array([[3, 0, 1, 2] * 8])                     # 2 bits: code j at bits 2 j
    w = KV.pack_codes(c, 2)
    assert w.shape == (1, 2) and int(w[0, 0]) == int(w[0, 1]) == 0x93939393
    assert np.array_equal(KV.unpack_codes(w, 2, 32), c)


def test_decode_is_textbook_attention_over_the_dequantized_cache():
    rng = np.random.default_rng(7)
    Hkv, Hq, Tc, Tw, d = 2, 6, 48, 5, 128
    K = rng.standard_normal((Hkv, Tc + Tw, d)) * 2
    V = rng.standard_normal((Hkv, Tc + Tw, d))
    q = rng.standard_normal((Hq, d))
    Kh = np.stack([KV.dequantize_keys(KV.quantize_keys(K[g, :Tc], 2)) for g in range(Hkv)])
    Vh = np.stack([KV.dequantize_values(KV.quantize_values(V[g, :Tc], 2)) for g in range(Hkv)])
    wk, wv = K[:, Tc:].astype(np.float16), V[:, Tc:].astype(np.float16)
    got = KV.decode_one(q, Kh, Vh, wk, wv, 1 / math.sqrt(d))
    G = Hq // Hkv
    Ke = np.repeat(np.concatenate([Kh, wk.astype(np.float64)], 1), G, 0)
    Ve = np.repeat(np.concatenate([Vh, wv.astype(np.float64)], 1), G, 0)
    l = np.einsum("htd,hd->ht", Ke, q) / math.sqrt(d)
    p = np.exp(l - l.max(1, keepdims=True))
    np.testing.assert_allclose(got["out"], np.einsum("ht,htd->hd", p / p.sum(1, keepdims=True), Ve), atol=1e-12)
    np.testing.assert_allclose(got["scores"], l, atol=1e-12)
    # against exact attention the 4-bit cache errs far less than the 2-bit one
    ex = A.exact_attention(q, K, V, 1 / math.sqrt(d))
    Kh4 = np.stack([KV.dequantize_keys(KV.quantize_keys(K[g, :Tc], 4)) for g in range(Hkv)])
    Vh4 = np.stack([KV.dequantize_values(KV.quantize_values(V[g, :Tc], 4)) for g in range(Hkv)])
    got4 = KV.decode_one(q, Kh4, Vh4, wk, wv, 1 / math.sqrt(d))
    e2, e4 = np.abs(got["out"] - ex["out"]).max(), np.abs(got4["out"] - ex["out"]).max()
    assert e4 < e2 / 3 and e2 > 1e-2
