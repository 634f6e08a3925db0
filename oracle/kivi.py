"""KIVI-like asymmetric control arm: per-channel keys, per-token values.

[Design study] §Candidate key and value algorithms, arm 3 ("control baseline
arm"): a KIVI-style per-channel K / per-token V baseline with an FP16 recent
window; the source table's KIVI entry: asymmetric K/V handling, 2-bit
tuning-free quantization, a configurable FP16 residual window.  The pages
give no formulas; the reading taken is plain asymmetric min-max integer
quantization with b bits (b in {1, 2, 4}):

  group g of values x:  mn = min g, mx = max g;
  scale s = float16( float32(float32(mx) - float32(mn)) / float32(2^b - 1) )
      (the scale, a stored quantity, is formed in float32 on both sides, so
      its float16 rounding is the same decision everywhere);
  zero  z = float16(mn);
  code  c = min(2^b - 1, max(0, floor((x - z) / s + 1/2)))   (ties up),
        c = 0 where s == 0;
  x_hat = z + s c.

Groups: a key group is one channel of one head over the 16 tokens of one
page (the page is the fixed token group of the page format); a value group
is one token of one head over its d channels.  The most recent tokens stay
float16 (the window of the TurboQuant path, same flush rule).

Page sub-block of one (page, kv head), token-major codes packed as integers
(code j of a token at bits (j b) mod 32 of word (j b) / 32):
  key scales   float16[d]                      2 d
  key zeros    float16[d]                      2 d
  key codes    uint32[16][d b_k / 32]          2 d b_k
  value scales float16[16]                     32
  value zeros  float16[16]                     32
  value codes  uint32[16][d b_v / 32]          2 d b_v
"""

from __future__ import annotations

import math

import numpy as np

PAGE = 16
KIVI_BITS = (1, 2, 4)


def scale_zero(mn: np.ndarray, mx: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """(s, z) as float16 from the group minimum and maximum."""
    rng32 = np.asarray(mx, np.float32) - np.asarray(mn, np.float32)
    s = (rng32 / np.float32((1 << bits) - 1)).astype(np.float16)
    z = np.asarray(mn, np.float32).astype(np.float16)
    return s, z


def codes_of(x: np.ndarray, s: np.ndarray, z: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """Codes of x under (s, z) (broadcast), and each code decision's margin: the
    distance of (x - z) / s from the nearest rounding point k + 1/2 (inf where
    s == 0 or the value is clamped far outside the range)."""
    x = np.asarray(x, np.float64)
    s64 = np.asarray(s, np.float64)
    z64 = np.asarray(z, np.float64)
    top = (1 << bits) - 1
    live = s64 > 0
    t = np.where(live, (x - z64) / np.where(live, s64, 1.0), 0.0)
    c = np.clip(np.floor(t + 0.5), 0, top)
    c = np.where(live, c, 0).astype(np.int64)
    k = np.clip(np.round(t - 0.5), 0, top - 1)
    margin = np.where(live, np.abs(t - (k + 0.5)), np.inf)
    return c, margin


def dequantize(c: np.ndarray, s: np.ndarray, z: np.ndarray) -> np.ndarray:
    return np.asarray(z, np.float64) + np.asarray(s, np.float64) * np.asarray(c, np.float64)


def quantize_key_page(K: np.ndarray, bits: int) -> dict:
    """Keys of one page and head, K [n <= 16, d] -> per-channel (s, z) [d], codes [n, d]."""
    K = np.asarray(K, np.float64)
    s, z = scale_zero(K.min(axis=0), K.max(axis=0), bits)
    c, margin = codes_of(K, s[None, :], z[None, :], bits)
    return {"scale": s, "zero": z, "codes": c, "margin": margin}


def quantize_values(V: np.ndarray, bits: int) -> dict:
    """Values V [n, d] -> per-token (s, z) [n], codes [n, d]."""
    V = np.asarray(V, np.float64)
    s, z = scale_zero(V.min(axis=1), V.max(axis=1), bits)
    c, margin = codes_of(V, s[:, None], z[:, None], bits)
    return {"scale": s, "zero": z, "codes": c, "margin": margin}


def quantize_keys(K: np.ndarray, bits: int) -> dict:
    """Keys [T, d] of one head, T a multiple of 16, page by page; scale and zero [T/16, d]."""
    T, d = K.shape
    if T % PAGE:
        raise ValueError("keys are quantized in whole pages")
    pages = [quantize_key_page(K[p:p + PAGE], bits) for p in range(0, T, PAGE)]
    return {"scale": np.stack([r["scale"] for r in pages]), "zero": np.stack([r["zero"] for r in pages]),
            "codes": np.concatenate([r["codes"] for r in pages]),
            "margin": np.concatenate([r["margin"] for r in pages])}


def dequantize_keys(rec: dict) -> np.ndarray:
    s = np.repeat(np.asarray(rec["scale"], np.float64), PAGE, axis=0)
    z = np.repeat(np.asarray(rec["zero"], np.float64), PAGE, axis=0)
    return z + s * rec["codes"]


def dequantize_values(rec: dict) -> np.ndarray:
    return dequantize(rec["codes"], rec["scale"][:, None], rec["zero"][:, None])


# ----------------------------------------------------------------------------- page layout

def subblock_layout(d: int, key_bits: int, value_bits: int) -> dict:
    if key_bits not in KIVI_BITS or value_bits not in KIVI_BITS:
        raise ValueError("KIVI bits must be 1, 2 or 4")
    off, o = {}, 0
    off["key_scale"] = o; o += 2 * d
    off["key_zero"] = o; o += 2 * d
    off["key_codes"] = o; o += 4 * PAGE * (d * key_bits // 32)
    off["value_scale"] = o; o += 2 * PAGE
    off["value_zero"] = o; o += 2 * PAGE
    off["value_codes"] = o; o += 4 * PAGE * (d * value_bits // 32)
    off["bytes"] = o
    return off


def record_bytes(d: int, key_bits: int, value_bits: int) -> float:
    """Bytes per (token, kv head), the key scales and zeros shared by a page's 16 tokens."""
    return (4 * d + PAGE * d * key_bits // 8 + 4 * PAGE + PAGE * d * value_bits // 8) / PAGE


def pack_codes(c: np.ndarray, bits: int) -> np.ndarray:
    """[n, d] codes -> uint32 [n, d b / 32], code j at bits (j b) mod 32 of word (j b) / 32."""
    n, d = c.shape
    per = 32 // bits
    c = np.asarray(c, np.uint64).reshape(n, d // per, per)
    sh = (np.arange(per, dtype=np.uint64) * np.uint64(bits))
    return (c << sh).sum(axis=-1).astype(np.uint32)


def unpack_codes(w: np.ndarray, bits: int, d: int) -> np.ndarray:
    per = 32 // bits
    w = np.asarray(w, np.uint64)[..., None]
    sh = np.arange(per, dtype=np.uint64) * np.uint64(bits)
    c = (w >> sh) & np.uint64((1 << bits) - 1)
    return c.reshape(w.shape[:-2] + (d,)).astype(np.int64)


def write_page(pool: np.ndarray, lay: dict, n_heads: int, page: int, head: int, d: int, key_bits: int,
               value_bits: int, krec: dict, vrec: dict) -> None:
    """One full page (16 tokens) of one head: krec from quantize_key_page, vrec from quantize_values."""
    base = (page * n_heads + head) * lay["bytes"]
    sb = pool[base: base + lay["bytes"]]
    sb[lay["key_scale"]: lay["key_scale"] + 2 * d] = np.asarray(krec["scale"], np.float16).view(np.uint8)
    sb[lay["key_zero"]: lay["key_zero"] + 2 * d] = np.asarray(krec["zero"], np.float16).view(np.uint8)
    kw = pack_codes(krec["codes"], key_bits)
    sb[lay["key_codes"]: lay["key_codes"] + kw.nbytes] = kw.view(np.uint8).ravel()
    sb[lay["value_scale"]: lay["value_scale"] + 2 * PAGE] = np.asarray(vrec["scale"], np.float16).view(np.uint8)
    sb[lay["value_zero"]: lay["value_zero"] + 2 * PAGE] = np.asarray(vrec["zero"], np.float16).view(np.uint8)
    vw = pack_codes(vrec["codes"], value_bits)
    sb[lay["value_codes"]: lay["value_codes"] + vw.nbytes] = vw.view(np.uint8).ravel()


def read_page(pool: np.ndarray, lay: dict, n_heads: int, page: int, head: int, d: int, key_bits: int,
              value_bits: int) -> dict:
    base = (page * n_heads + head) * lay["bytes"]
    sb = np.ascontiguousarray(pool[base: base + lay["bytes"]])
    kw = sb[lay["key_codes"]: lay["key_codes"] + 4 * PAGE * (d * key_bits // 32)].view(np.uint32)
    vw = sb[lay["value_codes"]: lay["value_codes"] + 4 * PAGE * (d * value_bits // 32)].view(np.uint32)
    return {"kscale": sb[lay["key_scale"]: lay["key_scale"] + 2 * d].view(np.float16).copy(),
            "kzero": sb[lay["key_zero"]: lay["key_zero"] + 2 * d].view(np.float16).copy(),
            "kcodes": unpack_codes(kw.reshape(PAGE, -1), key_bits, d),
            "vscale": sb[lay["value_scale"]: lay["value_scale"] + 2 * PAGE].view(np.float16).copy(),
            "vzero": sb[lay["value_zero"]: lay["value_zero"] + 2 * PAGE].view(np.float16).copy(),
            "vcodes": unpack_codes(vw.reshape(PAGE, -1), value_bits, d)}


# ----------------------------------------------------------------------------- decode

def decode_one(q: np.ndarray, Khat: np.ndarray | None, Vhat: np.ndarray | None, win_k: np.ndarray | None,
               win_v: np.ndarray | None, scale: float) -> dict:
    """Attention of one sequence over its dequantized pages and float16 window:
    q [Hq, d]; Khat, Vhat [Hkv, Tc, d] (float64 dequantized); window [Hkv, Tw, d]."""
    from .attention import exact_attention

    parts_k = [x for x in (Khat, None if win_k is None else np.asarray(win_k, np.float64)) if x is not None]
    parts_v = [x for x in (Vhat, None if win_v is None else np.asarray(win_v, np.float64)) if x is not None]
    K = np.concatenate(parts_k, axis=1)
    V = np.concatenate(parts_v, axis=1)
    return exact_attention(q, K, V, scale)


def error_bound(x: np.ndarray, s: np.ndarray, z: np.ndarray, mn: np.ndarray, mx: np.ndarray, bits: int) -> np.ndarray:
    """Bound on |x - x_hat| for a group: half a step inside the range, plus the float16 rounding of the zero
    and of the scale times the top code at the clamped ends."""
    s64, z64 = np.asarray(s, np.float64), np.asarray(z, np.float64)
    top = (1 << bits) - 1
    return (s64 / 2 + np.abs(np.asarray(mn, np.float64) - z64)
            + np.abs(np.asarray(mx, np.float64) - np.asarray(mn, np.float64) - top * s64) + 0 * x)
