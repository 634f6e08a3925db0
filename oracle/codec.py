"""Per-vector TurboQuant_mse (values) and TurboQuant_prod (keys), and packing.

TurboQuant_mse ([Reconstruction] §5 Steps 1-5):
  1. norm separation: n = ||x||, u = x / n; n stored as float32 (§8 storage
     formula: "Norm: 1 float32");
  2. rotation: y = Pi u;
  4./5. each coordinate is mapped to the index of its Lloyd-Max bucket; the
     reconstruction is x_hat = n Pi^T c[idx].
  Zero guard ([Reconstruction] §11 item 2, §13 reference logic): if
  n < 1e-7 the record is a zero code with norm 0.
  "RMS-scaled" (reading): the decision variable is z = sqrt(d) * y, compared
  against the float32 boundaries of the RMS-scaled codebook; ties go up,
  idx_j = #{i : z_j >= t_i}.

TurboQuant_prod for keys ([Reconstruction] §6 "The Residual and
Bit-Splitting", "The 1-Bit QJL Transform", "The Asymmetric Unbiased
Estimator"): a (b-1)-bit MSE code, the residual r, its norm gamma = ||r||
stored as float32, and the sign sketch sign(S r) with S d x d i.i.d. N(0,1).
Reading: the residual is taken in the rotated basis, r = y - y_hat with
y_hat = c[idx] / sqrt(d); <q, r_original> = <Pi q, r> for orthogonal Pi, and
S Pi^T is again an i.i.d. Gaussian matrix, so the estimator's law is the one
stated on the page.  sign(0) = +1.  For a zero vector gamma = 0 and all sign
bits are +1.

Packing (reading; [README] §How It Works packs nibbles, [Design study]
§Packed format asks for a bit-packed code stream): sign-magnitude bit planes.
Per vector and b-bit code: plane 0 holds the sign side (bit = 1 iff
idx >= 2^(b-1)); planes 1..b-1 hold the magnitude m (LSB first), where
m = idx - 2^(b-1) on the non-negative side and m = 2^(b-1) - 1 - idx on the
negative side.  Coordinate j sits at bit (j mod 32) of 32-bit word j // 32.
The QJL sketch is one plane, bit = 1 iff (S r)_j >= 0.

Mixed-channel rate ([Design study] §Packed format and complete bit
accounting: fractional rates by channel allocation, e.g. 3.5 bits per channel
= half the channels at 3 bits and half at 4, fixed offsets, no decoder
state).  Reading: the rotated coordinates 0 .. d/2 - 1 take the (b+1)-bit
Lloyd-Max book and the rest the b-bit book (the page does not say which
half; after the rotation every coordinate has the same law).  Byte norms
(same section, "u8 log-norm"): see norm_u8_encode.
"""

from __future__ import annotations

import math

import numpy as np

from . import transforms as T
from .codebook import Codebook

ZERO_NORM = 1e-7


def pad_head(x: np.ndarray, d: int) -> np.ndarray:
    """Zero-pad the last axis (a head of head_dim <= d coordinates) to the
    transform size d: [Design study] §Dense and structured transform
    comparison treats non-power-of-two head sizes by temporary zero-padding
    during append and query transform.  Inner products are unchanged."""
    x = np.asarray(x, dtype=np.float64)
    if x.shape[-1] == d:
        return x
    if x.shape[-1] > d:
        raise ValueError("head longer than the transform size")
    pad = [(0, 0)] * (x.ndim - 1) + [(0, d - x.shape[-1])]
    return np.pad(x, pad)


def qjl_constant(d: int) -> float:
    """sqrt(pi/2) / d: the QJL estimator constant for m = d sketch rows."""
    return math.sqrt(math.pi / 2.0) / d


def bucketize(z: np.ndarray, boundaries: np.ndarray) -> np.ndarray:
    """idx = #{i : z >= t_i} in float64 against the float32 boundaries."""
    t = np.asarray(boundaries, dtype=np.float32).astype(np.float64)
    return (z[..., None] >= t).sum(axis=-1).astype(np.int64)


def boundary_margin(z: np.ndarray, boundaries: np.ndarray) -> np.ndarray:
    t = np.asarray(boundaries, dtype=np.float32).astype(np.float64)
    return np.min(np.abs(z[..., None] - t), axis=-1)


def centroid_values(idx: np.ndarray, cb: Codebook, cb_hi: Codebook | None = None) -> np.ndarray:
    """Float64 copies of the float32 RMS-scaled centroids C[idx], per coordinate.
    Mixed-channel rate (cb_hi given): coordinates 0 .. d/2 - 1 read cb_hi."""
    book = lambda c: np.asarray(c.centroids, dtype=np.float32).astype(np.float64)
    if cb_hi is None:
        return book(cb)[idx]
    h = idx.shape[-1] // 2
    return np.concatenate([book(cb_hi)[idx[..., :h]], book(cb)[idx[..., h:]]], axis=-1)


def quantize_mse(x: np.ndarray, kind: int, rot: np.ndarray, cb: Codebook, cb_hi: Codebook | None = None) -> dict:
    """TurboQuant_mse of the rows of x ([N, d]); everything in float64.
    cb_hi (mixed-channel rate): rotated coordinates 0 .. d/2 - 1 are coded
    with cb_hi, the rest with cb (see centroid_values)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    n = np.sqrt(np.sum(x * x, axis=-1))
    zero = n < ZERO_NORM
    u = np.where(zero[:, None], 0.0, x / np.where(zero, 1.0, n)[:, None])
    y = T.rotate(kind, rot, u)
    z = math.sqrt(d) * y
    if cb_hi is None:
        idx = bucketize(z, cb.boundaries)
        margin = boundary_margin(z, cb.boundaries)
    else:
        h = d // 2
        idx = np.concatenate([bucketize(z[:, :h], cb_hi.boundaries), bucketize(z[:, h:], cb.boundaries)], axis=-1)
        margin = np.concatenate([boundary_margin(z[:, :h], cb_hi.boundaries),
                                 boundary_margin(z[:, h:], cb.boundaries)], axis=-1)
    yhat = centroid_values(idx, cb, cb_hi) / math.sqrt(d)
    norm32 = np.where(zero, 0.0, n).astype(np.float32)
    return {"norm": norm32, "norm_f64": np.where(zero, 0.0, n), "idx": idx, "y": y, "z": z,
            "yhat": yhat, "zero": zero, "margin": margin}


def quantize_prod(x: np.ndarray, kind: int, rot: np.ndarray, cb: Codebook, S: np.ndarray) -> dict:
    """TurboQuant_prod of the rows of x: MSE code + residual norm + QJL signs
    (uniform rate only: the mixed-channel key mode carries no sketch)."""
    rec = quantize_mse(x, kind, rot, cb)
    r = rec["y"] - rec["yhat"]
    gamma = np.sqrt(np.sum(r * r, axis=-1))
    Sr = sketch(r, S)
    signs = Sr >= 0.0
    zero = rec["zero"]
    gamma = np.where(zero, 0.0, gamma)
    signs[zero] = True
    rec.update({"r": r, "rnorm": gamma.astype(np.float32), "rnorm_f64": gamma, "signs": signs,
                "Sr": Sr, "sign_margin": np.where(zero[:, None], np.inf, np.abs(Sr))})
    return rec


# ----------------------------------------------------------------------------- packing

# Key corrections.  QJL is TurboQuant_prod's residual sketch; the two others
# spend no bit on a residual and keep one float32 scale s per key instead
# (the "next" correction variants), so that the key is reconstructed as
# n s Pi^T y_hat:
#  * EDEN's unbiased scale ([Reconstruction] §10, §12.2: TurboQuant_mse is
#    EDEN/DRIVE with a fixed scale; the unbiased EDEN scalar has 2.75x lower
#    1-bit variance than QJL): the scale that makes <y, s y_hat> = ||y||^2,
#    s = ||y||^2 / <y, y_hat>, with y the rotated unit vector (||y|| = 1);
#  * TurboVec's length-renormalized correction ([Reconstruction] §12 item 2,
#    §13 reference logic, step 6): one scalar per vector computed at
#    ingestion, the vector's norm divided by the inner product of the
#    rotated unit vector with its reconstruction, norm / <y, y_hat>; the
#    page says it restores unbiasedness.  The record keeps the norm n in its
#    own field, so the stored scale is that scalar divided by n.  Both
#    readings give the same number: the page notes that TurboVec mirrors the
#    EDEN strategy.
KEY_MSE, KEY_QJL, KEY_EDEN, KEY_RENORM = 0, 1, 2, 3


def quantize_scaled(x: np.ndarray, kind: int, rot: np.ndarray, cb: Codebook, mode: int,
                    cb_hi: Codebook | None = None) -> dict:
    """TurboQuant_mse code of the rows of x plus the scale s of the key
    correction `mode` (KEY_EDEN or KEY_RENORM), stored as float32 in the
    record's "rnorm" slot; the key is reconstructed as n s Pi^T y_hat.  For a
    zero vector s = 0 (its norm is 0, so its score is 0 whatever s is).
    cb_hi: mixed-channel rate as in quantize_mse."""
    rec = quantize_mse(x, kind, rot, cb, cb_hi)
    y, yhat, zero = rec["y"], rec["yhat"], rec["zero"]
    dot = np.where(zero, 1.0, np.sum(y * yhat, axis=-1))
    if mode == KEY_EDEN:
        s = np.sum(y * y, axis=-1) / dot
    elif mode == KEY_RENORM:
        n = rec["norm_f64"]
        correction = n / dot                       # norm / <y, y_hat>
        s = correction / np.where(zero, 1.0, n)    # the norm is stored separately
    else:
        raise ValueError("mode must be KEY_EDEN or KEY_RENORM")
    s = np.where(zero, 0.0, s)
    rec.update({"rnorm": s.astype(np.float32), "rnorm_f64": s, "scale": s})
    return rec


def dequantize_scaled(norm, scale, idx, kind, rot, cb, cb_hi=None) -> np.ndarray:
    """k_hat = n s Pi^T y_hat for the EDEN / length-renormalized keys."""
    return np.asarray(scale, dtype=np.float64)[:, None] * dequantize_mse(norm, idx, kind, rot, cb, cb_hi)


def code_planes(idx: np.ndarray, bits: int) -> np.ndarray:
    """Sign-magnitude planes as 0/1 arrays: [..., bits, d]."""
    half = 1 << (bits - 1)
    pos = idx >= half
    mag = np.where(pos, idx - half, half - 1 - idx)
    planes = [pos.astype(np.uint8)]
    for k in range(bits - 1):
        planes.append(((mag >> k) & 1).astype(np.uint8))
    return np.stack(planes, axis=-2)


def planes_to_idx(planes: np.ndarray) -> np.ndarray:
    bits = planes.shape[-2]
    half = 1 << (bits - 1)
    mag = np.zeros(planes.shape[:-2] + planes.shape[-1:], dtype=np.int64)
    for k in range(bits - 1):
        mag |= planes[..., k + 1, :].astype(np.int64) << k
    pos = planes[..., 0, :].astype(bool)
    return np.where(pos, half + mag, half - 1 - mag)


def pack_bits(b: np.ndarray) -> np.ndarray:
    """0/1 array [..., d] -> uint32 words [..., d // 32], coordinate j at bit j % 32."""
    d = b.shape[-1]
    if d % 32:
        raise ValueError("d must be a multiple of 32")
    w = b.reshape(b.shape[:-1] + (d // 32, 32)).astype(np.uint64)
    return (w << np.arange(32, dtype=np.uint64)).sum(axis=-1).astype(np.uint32)


def unpack_bits(w: np.ndarray, d: int) -> np.ndarray:
    w = np.asarray(w, dtype=np.uint64)[..., None]
    b = (w >> np.arange(32, dtype=np.uint64)) & np.uint64(1)
    return b.reshape(w.shape[:-2] + (d,)).astype(np.uint8)


def pack_codes(idx: np.ndarray, bits: int) -> np.ndarray:
    """[N, d] code indices -> uint32 [N, bits, d // 32]."""
    return pack_bits(code_planes(idx, bits))


def unpack_codes(words: np.ndarray, bits: int, d: int) -> np.ndarray:
    return planes_to_idx(unpack_bits(words, d))


# ----------------------------------------------------------------------------- reconstruction

def dequantize_mse(norm: np.ndarray, idx: np.ndarray, kind: int, rot: np.ndarray, cb: Codebook,
                   cb_hi: Codebook | None = None) -> np.ndarray:
    """x_hat = n Pi^T c[idx] / sqrt(d)  ([Reconstruction] §5 Step 5)."""
    d = idx.shape[-1]
    yhat = centroid_values(idx, cb, cb_hi) / math.sqrt(d)
    return np.asarray(norm, dtype=np.float64)[:, None] * T.rotate_inverse(kind, rot, yhat)


def dequantize_prod(norm, rnorm, idx, signs, kind, rot, cb, S) -> np.ndarray:
    """Explicit key the estimator is an inner product with:
    k_hat = n Pi^T (y_hat + sqrt(pi/2)/d * gamma * S^T (2 s - 1))."""
    d = idx.shape[-1]
    yhat = np.asarray(cb.centroids, dtype=np.float32).astype(np.float64)[idx] / math.sqrt(d)
    pm = np.where(np.asarray(signs, dtype=bool), 1.0, -1.0)
    corr = pm @ np.asarray(S, dtype=np.float32).astype(np.float64)
    ytil = yhat + qjl_constant(d) * np.asarray(rnorm, dtype=np.float64)[:, None] * corr
    return np.asarray(norm, dtype=np.float64)[:, None] * T.rotate_inverse(kind, rot, ytil)


def sketch(v: np.ndarray, S: np.ndarray) -> np.ndarray:
    """S v for v [..., d] and S [..., d, d] (broadcast), float64."""
    S = np.asarray(S)
    S = S.astype(np.float64) if S.dtype != np.float64 else S
    return np.matmul(S, np.asarray(v, dtype=np.float64)[..., None])[..., 0]


def qjl_estimate(q: np.ndarray, r_norm, signs: np.ndarray, S: np.ndarray) -> np.ndarray:
    """Residual inner-product estimate sqrt(pi/2)/d * ||r|| * <S q, sign(S r)>
    ([Reconstruction] §6 "The Asymmetric Unbiased Estimator"); broadcasts
    over leading axes of S / signs."""
    d = q.shape[-1]
    pm = np.where(np.asarray(signs, dtype=bool), 1.0, -1.0)
    return qjl_constant(d) * np.asarray(r_norm, dtype=np.float64) * np.sum(sketch(q, S) * pm, axis=-1)


# ----------------------------------------------------------------------------- mixed-channel rate, byte norms

def pack_codes_split(idx: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """Mixed-channel rate ([Design study] §Packed format: 3.5 bits per
    channel = half the channels at 3 bits, half at 4): coordinates 0 .. d/2-1
    hold (bits + 1)-bit codes, the rest bits-bit codes, both sign-magnitude.
    Planes 0 .. bits-1 mean the same in both halves (sign, then magnitude
    bits LSB first) and cover all d coordinates; plane `bits` (the top
    magnitude bit of the wider codes) exists for the first half only.
    Returns (uint32 [N, bits, d/32], uint32 [N, d/64])."""
    d = idx.shape[-1]
    h = d // 2
    hi = code_planes(idx[..., :h], bits + 1)
    lo = code_planes(idx[..., h:], bits)
    main = np.concatenate([hi[..., :bits, :], lo], axis=-1)
    return pack_bits(main), pack_bits(hi[..., bits, :])


def unpack_codes_split(words: np.ndarray, extra: np.ndarray, bits: int, d: int) -> np.ndarray:
    h = d // 2
    planes = unpack_bits(words, d)                        # [..., bits, d]
    top = unpack_bits(extra, h)[..., None, :]             # [..., 1, d/2]
    hi = np.concatenate([planes[..., :, :h], top], axis=-2)
    return np.concatenate([planes_to_idx(hi), planes_to_idx(planes[..., :, h:])], axis=-1)


NORM_U8_LEVELS = 255  # codes 1..255; code 0 marks a zero vector


def norm_u8_step(lo: float, hi: float) -> float:
    """log2 spacing of the byte norm codes over [2^lo, 2^hi]."""
    return (hi - lo) / (NORM_U8_LEVELS - 1)


def norm_u8_encode(n: np.ndarray, lo: float, hi: float) -> tuple[np.ndarray, np.ndarray]:
    """u8 log-norm ([Design study] §Packed format: one byte per token-head
    for the key norm, 8 / d bits per channel).  Reading: codes 1..255 are
    uniform in log2 over [lo, hi] (a per-layer range), round to nearest with
    ties up, clamped at both ends; code 0 is the zero vector (n < 1e-7).
      t = (log2 n - lo) / step,  code = 1 + min(254, max(0, floor(t + 1/2))).
    Returns (codes uint8, margin): margin is |t - decision point| in code
    units for the nearest of the 254 decision points t = k + 1/2."""
    n = np.asarray(n, dtype=np.float64)
    zero = n < ZERO_NORM
    t = (np.log2(np.where(zero, 1.0, n)) - lo) / norm_u8_step(lo, hi)
    k = np.clip(np.floor(t + 0.5), 0, NORM_U8_LEVELS - 1)
    codes = np.where(zero, 0, 1 + k).astype(np.uint8)
    kd = np.clip(np.round(t - 0.5), 0, NORM_U8_LEVELS - 2)
    margin = np.where(zero, np.inf, np.abs(t - (kd + 0.5)))
    return codes, margin


def norm_u8_decode(codes: np.ndarray, lo: float, hi: float) -> np.ndarray:
    """n_hat = 2^(lo + (code - 1) step); 0 for code 0."""
    c = np.asarray(codes, dtype=np.float64)
    return np.where(c == 0, 0.0, np.exp2(lo + (c - 1.0) * norm_u8_step(lo, hi)))
