"""Pins of the mixed-channel key rate and the byte (u8 log) key norm.

[Design study] §Packed format and complete bit accounting: fractional rates
come from channel allocation (3.5 bits per channel = 64 channels at 3 bits
and 64 at 4 for d = 128), and a u8 norm adds 8 / d = 0.0625 bits per channel
at d = 128.  Reading: the rotated coordinates 0 .. d/2 - 1 carry the wider
code; the byte norm is uniform in log2 over a per-layer range.

* With the same book on both halves the mixed quantizer is the uniform one;
  with two books each half equals the uniform quantizer of its own book.
* Distortion E||u - u_hat||^2 is the mean of the two books' Lloyd-Max unit
  MSEs (each half holds half the coordinates, all with the same law).
* Packing: a hand-worked sign-magnitude example; round trips; the record
  sizes the page's bit accounting gives.
* Byte norm: grid points decode exactly, the round trip stays within the
  half-step bound 2^(step/2) - 1, codes are monotone, clamped, 0 = zero vector.
* Decode attention over mixed keys with byte norms equals textbook attention
  over explicitly dequantized keys.
"""

import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import codebook as CB
from oracle import codec as C
from oracle import paging as PG
from oracle import transforms as T


@pytest.mark.parametrize("kind", [T.DENSE, T.FWHT])
def test_same_book_on_both_halves_is_the_uniform_quantizer(kind):
    d = 128
    cb = CB.lloyd_max(d, 3)
    rot = T.build_transform(kind, d, 5, 0, 0, 0)
    x = np.random.default_rng(0).standard_normal((200, d))
    a = C.quantize_mse(x, kind, rot, cb)
    b = C.quantize_mse(x, kind, rot, cb, cb_hi=cb)
    for k in ("idx", "yhat", "margin", "norm"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("kind", [T.DENSE, T.FWHT])
@pytest.mark.parametrize("bits", [1, 2, 3])
def test_each_half_is_its_own_uniform_quantizer(kind, bits):
    d = 128
    lo, hi = CB.lloyd_max(d, bits), CB.lloyd_max(d, bits + 1)
    rot = T.build_transform(kind, d, 7, 1, 0, 0)
    x = np.random.default_rng(bits).standard_normal((300, d)) * np.exp(np.random.default_rng(9).standard_normal(d))
    mixed = C.quantize_mse(x, kind, rot, lo, cb_hi=hi)
    u_lo = C.quantize_mse(x, kind, rot, lo)
    u_hi = C.quantize_mse(x, kind, rot, hi)
    h = d // 2
    assert np.array_equal(mixed["idx"][:, :h], u_hi["idx"][:, :h])
    assert np.array_equal(mixed["idx"][:, h:], u_lo["idx"][:, h:])
    np.testing.assert_array_equal(mixed["yhat"][:, :h], u_hi["yhat"][:, :h])
    np.testing.assert_array_equal(mixed["yhat"][:, h:], u_lo["yhat"][:, h:])
    assert mixed["idx"][:, :h].max() < 1 << (bits + 1) and mixed["idx"][:, h:].max() < 1 << bits
    xh = C.dequantize_mse(mixed["norm"], mixed["idx"], kind, rot, lo, hi)
    yh = T.rotate(kind, rot, xh / np.asarray(mixed["norm"], np.float64)[:, None])
    # the stored dense rotation is float32, orthogonal to ~1e-7
    np.testing.assert_allclose(yh, mixed["yhat"], rtol=0, atol=1e-6)


@pytest.mark.parametrize("bits", [2, 3])
def test_mixed_distortion_is_the_mean_of_the_two_books(bits):
    d = 128
    lo, hi = CB.lloyd_max(d, bits), CB.lloyd_max(d, bits + 1)
    rng = np.random.default_rng(30 + bits)
    errs = []
    for seed in range(6):
        rot = T.build_transform(T.DENSE, d, seed, 0, 0, 0)
        x = rng.standard_normal((1500, d))
        rec = C.quantize_mse(x, T.DENSE, rot, lo, cb_hi=hi)
        xh = C.dequantize_mse(rec["norm"], rec["idx"], T.DENSE, rot, lo, hi)
        errs.append(np.sum((xh - x) ** 2, axis=1) / np.sum(x ** 2, axis=1))
    e = np.concatenate(errs)
    expect = 0.5 * (lo.mse_unit + hi.mse_unit)
    assert abs(e.mean() - expect) < 5 * e.std() / math.sqrt(e.size)
    assert hi.mse_unit < e.mean() < lo.mse_unit


def test_split_packing_worked_example():
    # d = 64, base 1 bit: coordinates 0..31 take 2-bit codes j mod 4, 32..63 1-bit codes j mod 2.
    # 2-bit sign-magnitude (half = 2): 0 -> sign 0, m 1; 1 -> 0, 0; 2 -> 1, 0; 3 -> 1, 1.
    # Plane 0 of word 0: bits set where j mod 4 in {2, 3} -> 0xCCCCCCCC; the top plane where
    # j mod 4 in {0, 3} -> 0x99999999.  1-bit codes: sign bit set for code 1 -> 0xAAAAAAAA.
    d = 64
    idx = np.concatenate([np.arange(32) % 4, np.arange(32) % 2])[None]
    words, extra = C.pack_codes_split(idx, 1)
    assert words.shape == (1, 1, 2) and extra.shape == (1, 1)
    assert [int(w) for w in words[0, 0]] == [0xCCCCCCCC, 0xAAAAAAAA]
    assert int(extra[0, 0]) == 0x99999999
    assert np.array_equal(C.unpack_codes_split(words, extra, 1, d), idx)


@pytest.mark.parametrize("d,bits", [(128, 1), (128, 2), (128, 3), (256, 3)])
def test_split_packing_round_trip_and_size(d, bits):
    rng = np.random.default_rng(d * bits)
    idx = np.concatenate([rng.integers(0, 1 << (bits + 1), (50, d // 2)), rng.integers(0, 1 << bits, (50, d // 2))],
                         axis=1)
    words, extra = C.pack_codes_split(idx, bits)
    assert np.array_equal(C.unpack_codes_split(words, extra, bits, d), idx)
    # (bits + 1/2) bits per channel: 64 channels at 3 bits and 64 at 4 = 56 bytes at d = 128
    assert 4 * (words[0].size + extra[0].size) * 8 == (2 * bits + 1) * d // 2
    # the shared planes mean the same in both halves: planes 0..bits-1 of the wide half equal those
    # of the wide codes
    wide = C.code_planes(idx[:, : d // 2], bits + 1)
    assert np.array_equal(C.unpack_bits(words, d)[:, :, : d // 2], wide[:, :bits])


def test_bit_accounting_of_the_recommended_key_mode():
    # keys 3.5 bits per channel + u8 log-norm, no sketch; values 3 bits with a float32 norm
    d = 128
    key_bytes = PG.record_bytes(d, 3, 0, 3, key_split=1, key_norm_u8=1) - (4 + 3 * d // 8)
    assert key_bytes == 1 + 56
    assert key_bytes * 8 / d == 3.5 + 0.0625
    lay = PG.subblock_layout(d, 3, 0, 3, key_split=1, key_norm_u8=1)
    assert lay["bytes"] == 16 * PG.record_bytes(d, 3, 0, 3, key_split=1, key_norm_u8=1)
    assert all(v % 16 == 0 for v in lay.values())
    with pytest.raises(ValueError):
        PG.subblock_layout(d, 3, 1, 3, key_split=1)


@pytest.mark.parametrize("lo,hi", [(-4.0, 12.0), (2.0, 8.0)])
def test_byte_norm_grid_bound_and_order(lo, hi):
    step = C.norm_u8_step(lo, hi)
    k = np.arange(255)
    codes, _ = C.norm_u8_encode(np.exp2(lo + k * step), lo, hi)
    assert np.array_equal(codes, k + 1)
    np.testing.assert_allclose(C.norm_u8_decode(codes, lo, hi), np.exp2(lo + k * step), rtol=1e-14)
    rng = np.random.default_rng(3)
    n = np.sort(np.exp2(rng.uniform(lo, hi, 20000)))
    codes, margin = C.norm_u8_encode(n, lo, hi)
    assert np.all(np.diff(codes.astype(int)) >= 0)
    assert np.all(margin <= 0.5 + 1e-12)
    rel = np.abs(C.norm_u8_decode(codes, lo, hi) / n - 1.0)
    assert rel.max() <= 2.0 ** (step / 2) - 1.0 + 1e-12
    assert rel.max() > 0.9 * (2.0 ** (step / 2) - 1.0)  # the bound is reached
    c, m = C.norm_u8_encode(np.array([0.0, 5e-8, 2.0 ** (lo - 3), 2.0 ** (hi + 3)]), lo, hi)
    assert c.tolist() == [0, 0, 1, 255]
    assert C.norm_u8_decode(c, lo, hi)[:2].tolist() == [0.0, 0.0]
    assert m[0] == np.inf and m[1] == np.inf


def test_byte_norm_ties_go_up():
    lo, hi = 0.0, 508.0  # step 2: n = 2^e with e odd sits exactly on the decision point t = e / 2
    e = np.arange(1, 40, 2)
    codes, margin = C.norm_u8_encode(np.exp2(e.astype(np.float64)), lo, hi)
    assert np.array_equal(codes, 1 + (e + 1) // 2)
    assert np.all(margin == 0)


@pytest.mark.parametrize("kind", [T.DENSE, T.FWHT])
@pytest.mark.parametrize("corr", [C.KEY_MSE, C.KEY_EDEN, C.KEY_RENORM])
def test_attention_over_mixed_keys_equals_explicit_dequantization(kind, corr):
    rng = np.random.default_rng(11)
    Hkv, Hq, Tc, Tw, d = 2, 4, 64, 5, 128
    lo_r, hi_r = -2.0, 10.0
    K = rng.standard_normal((Hkv, Tc + Tw, d)) * np.exp(rng.standard_normal((Hkv, 1, d)))
    V = rng.standard_normal((Hkv, Tc + Tw, d))
    q = rng.standard_normal((Hq, d))
    kcb, kcb_hi, vcb = CB.lloyd_max(d, 3), CB.lloyd_max(d, 4), CB.lloyd_max(d, 3)
    p = {"kind": kind, "k_rot": [T.build_transform(kind, d, 3, 0, h, 0) for h in range(Hkv)],
         "v_rot": [T.build_transform(kind, d, 3, 0, h, 1) for h in range(Hkv)], "qjl_s": None,
         "k_cb": kcb, "k_cb_hi": kcb_hi, "v_cb": vcb, "key_qjl": corr}
    comp = {k: [] for k in ("knorm", "krnorm", "kidx", "vnorm", "vidx")}
    Kh, Vh = [], []
    for g in range(Hkv):
        if corr == C.KEY_MSE:
            kr = C.quantize_mse(K[g, :Tc], kind, p["k_rot"][g], kcb, cb_hi=kcb_hi)
            s = np.ones(Tc)
        else:
            kr = C.quantize_scaled(K[g, :Tc], kind, p["k_rot"][g], kcb, corr, cb_hi=kcb_hi)
            s = kr["rnorm"].astype(np.float64)
        code, _ = C.norm_u8_encode(kr["norm_f64"], lo_r, hi_r)
        nhat = C.norm_u8_decode(code, lo_r, hi_r)
        vr = C.quantize_mse(V[g, :Tc], kind, p["v_rot"][g], vcb)
        comp["knorm"].append(nhat); comp["krnorm"].append(s.astype(np.float32)); comp["kidx"].append(kr["idx"])
        comp["vnorm"].append(vr["norm"]); comp["vidx"].append(vr["idx"])
        Kh.append(C.dequantize_scaled(nhat, s.astype(np.float32), kr["idx"], kind, p["k_rot"][g], kcb, kcb_hi))
        Vh.append(C.dequantize_mse(vr["norm"], vr["idx"], kind, p["v_rot"][g], vcb))
    comp = {k: np.stack(v) for k, v in comp.items()}
    wk, wv = K[:, Tc:].astype(np.float16), V[:, Tc:].astype(np.float16)
    got = A.decode_one(q, comp, wk, wv, p, 1 / math.sqrt(d))
    Ke = np.repeat(np.concatenate([np.stack(Kh), wk.astype(np.float64)], 1), Hq // Hkv, axis=0)
    Ve = np.repeat(np.concatenate([np.stack(Vh), wv.astype(np.float64)], 1), Hq // Hkv, axis=0)
    l = np.einsum("htd,hd->ht", Ke, q) / math.sqrt(d)
    e = np.exp(l - l.max(1, keepdims=True))
    np.testing.assert_allclose(got["scores"], l, rtol=0, atol=1e-9)
    np.testing.assert_allclose(got["out"], np.einsum("ht,htd->hd", e / e.sum(1, keepdims=True), Ve), rtol=0, atol=1e-9)


def test_mixed_page_round_trip_with_byte_norms():
    d, kb, vb, H = 128, 3, 3, 2
    rng = np.random.default_rng(4)
    lay = PG.subblock_layout(d, kb, 2, vb, key_split=1, key_norm_u8=1)
    pool = np.zeros(3 * H * lay["bytes"], np.uint8)
    truth = {}
    for page in range(3):
        for h in range(H):
            for slot in range(16):
                idx = np.concatenate([rng.integers(0, 16, d // 2), rng.integers(0, 8, d // 2)])
                words, extra = C.pack_codes_split(idx[None], kb)
                rec = dict(code=int(rng.integers(0, 256)), s=rng.random(), idx=idx, vn=rng.random(),
                           vidx=rng.integers(0, 8, d))
                truth[page, h, slot] = rec
                PG.write_page(pool, lay, H, page, h, slot, d, kb, 2, vb, rec["code"], rec["s"], words[0], None,
                              rec["vn"], C.code_planes(rec["vidx"][None], vb)[0], kxcode_words=extra[0],
                              key_norm_u8=1)
    for page in range(3):
        for h in range(H):
            got = PG.read_page(pool, lay, H, page, h, d, kb, 2, vb, key_split=1, norm_range=(-4.0, 12.0))
            for slot in range(16):
                rec = truth[page, h, slot]
                assert got["knorm_code"][slot] == rec["code"]
                assert got["knorm"][slot] == C.norm_u8_decode(rec["code"], -4.0, 12.0)
                assert np.array_equal(got["kidx"][slot], rec["idx"])
                assert got["krnorm"][slot] == np.float32(rec["s"])
                assert np.array_equal(got["vidx"][slot], rec["vidx"])


def test_scalar_corrections_with_mixed_books():
    """With mixed-rate books both scalar corrections keep the estimate unbiased
    (uniformly rotated unit pairs with correlation rho, identity rotation): the
    EDEN scale and TurboVec's length-renormalized correction norm / <y, y_hat>,
    where the plain mixed code shrinks it."""
    d = 128
    lo, hi = CB.lloyd_max(d, 2), CB.lloyd_max(d, 3)
    n, rho = 20000, 0.6
    rng = np.random.default_rng(6)
    g = rng.standard_normal((n, d))
    y = g / np.linalg.norm(g, axis=1, keepdims=True)
    h = rng.standard_normal((n, d))
    h -= np.sum(h * y, axis=1, keepdims=True) * y
    h /= np.linalg.norm(h, axis=1, keepdims=True)
    q = rho * y + math.sqrt(1 - rho * rho) * h
    for mode in (C.KEY_EDEN, C.KEY_RENORM):
        rec = C.quantize_scaled(2.0 * y, T.DENSE, np.eye(d), lo, mode, cb_hi=hi)
        est = rec["norm_f64"] * rec["scale"] * np.sum(q * rec["yhat"], axis=1)
        assert abs(est.mean() - 2.0 * rho) < 4 * est.std() / math.sqrt(n), mode
    plain = np.sum(q * rec["yhat"], axis=1)
    assert rho - plain.mean() > 10 * plain.std() / math.sqrt(n)
