"""Fixed-size cache pages, the fp16 recent window and the append policy.

[Design study] §Packed format and complete bit accounting: a fixed-token page
per layer, token-major append order, head-major inner layout; body order
ring marker -> key norms -> key code stream -> key residual sign stream ->
(outlier sidecar) -> value norms -> value code stream -> padding to 16 bytes.
[Design study] §Paging, lifecycle: page-wise growth ("fixed-page append until
full").  The 64-byte header, ring marker and outlier sidecars are not part of
the hot path and are not stored (the sidecar is deferred by the page itself:
"no outlier sidecar initially").

Sub-block of one (page, kv head), P = 16 tokens, in this order (byte sizes):
  key norms          float32[P]  (uint8[P] as byte codes)     4 P  (P)
  key residual norms float32[P]          (only with QJL)      4 P
  key code planes    uint32[b_k][P][d/32]  token-major        b_k P d / 8
  key top plane      uint32[P][d/64]  (mixed-channel rate)    P d / 16
  key sign plane     uint32[P][d/32]       (only with QJL)    P d / 8
  value norms        float32[P]                               4 P
  value code planes  uint16[b_v][d]        coordinate-major:  b_v P d / 8
                     bit t of entry (p, j) is plane p of token t, coordinate j
Every size is a multiple of 16 bytes for d >= 32, so the sub-block needs no
padding.  The pool is [n_pages][n_kv_heads][sub-block].

Window ([Design study] §Executive summary, §Packed format "Recent tokens"):
the last W tokens stay float16 for both K and V.  Reading of the flush rule:
whole pages; the number of compressed tokens at length T is
n_c(T) = P * floor(max(0, T - W) / P), so the window holds T - n_c(T) tokens,
between W and W + P - 1 once T >= W.  The ring has W + P slots per
(sequence, kv head); a flushed page is quantized from the float16 window
contents.
"""

from __future__ import annotations

import numpy as np

PAGE = 16


def n_compressed(T: int, W: int, P: int = PAGE) -> int:
    return P * (max(0, T - W) // P)


def subblock_layout(d: int, key_bits: int, key_qjl: int, value_bits: int, P: int = PAGE,
                    key_split: int = 0, key_norm_u8: int = 0) -> dict:
    """key_qjl: key correction (0 none, 1 QJL: scale slot + sign plane, 2 / 3 EDEN / length-renormalized: scale slot).
    key_split: mixed-channel key rate (the first d/2 coordinates carry one more plane, stored after the
    key_bits full planes as uint32 [P][d/64]).  key_norm_u8: key norms as one byte per token."""
    if P != PAGE:
        raise ValueError("page size is fixed at 16 tokens")
    if key_split and (key_qjl == 1 or d % 64):
        raise ValueError("the mixed-channel key rate needs d % 64 == 0 and no QJL sketch")
    w = d // 32
    off = {}
    o = 0
    off["key_norm"] = o; o += (1 if key_norm_u8 else 4) * P
    off["key_rnorm"] = o; o += 4 * P if key_qjl else 0
    off["key_codes"] = o; o += 4 * key_bits * P * w
    off["key_xcodes"] = o; o += 4 * P * (w // 2) if key_split else 0
    off["key_signs"] = o; o += 4 * P * w if key_qjl == 1 else 0
    off["value_norm"] = o; o += 4 * P
    off["value_codes"] = o; o += 2 * value_bits * d
    off["bytes"] = o
    return off


def record_bytes(d: int, key_bits: int, key_qjl: bool, value_bits: int, key_split: int = 0,
                 key_norm_u8: int = 0) -> int:
    """Bytes per (token, kv head): the D1 + D2 storage formulas of
    [Reconstruction] §8 with float32 norms, or the [Design study] bit
    accounting with a byte key norm and mixed-channel key rates."""
    kb = (1 if key_norm_u8 else 4) + (4 if key_qjl else 0) + key_bits * d // 8 + (d // 16 if key_split else 0)
    kb += d // 8 if key_qjl == 1 else 0
    vb = 4 + value_bits * d // 8
    return kb + vb


def write_page(pool: np.ndarray, lay: dict, n_heads: int, page: int, head: int, slot: int,
               d: int, key_bits: int, key_qjl: bool, value_bits: int,
               knorm, krnorm, kcode_words, ksign_words, vnorm, vcode_planes_bits,
               kxcode_words=None, key_norm_u8: int = 0) -> None:
    """Write one token record into the byte pool (uint8 [n_pages * n_heads * bytes]).

    kcode_words: uint32 [key_bits, d/32]; ksign_words: uint32 [d/32];
    vcode_planes_bits: uint8 0/1 [value_bits, d]; kxcode_words: uint32 [d/64]
    (mixed-channel keys); knorm: the float32 norm, or its byte code with key_norm_u8.
    """
    base = (page * n_heads + head) * lay["bytes"]
    sb = pool[base: base + lay["bytes"]]
    w = d // 32
    if key_norm_u8:
        sb[lay["key_norm"] + slot] = np.uint8(knorm)
    else:
        sb[lay["key_norm"] + 4 * slot: lay["key_norm"] + 4 * slot + 4] = np.array([knorm], np.float32).view(np.uint8)
    if key_qjl:
        sb[lay["key_rnorm"] + 4 * slot: lay["key_rnorm"] + 4 * slot + 4] = np.array([krnorm], np.float32).view(np.uint8)
    for p in range(key_bits):
        o = lay["key_codes"] + 4 * ((p * PAGE + slot) * w)
        sb[o: o + 4 * w] = np.asarray(kcode_words[p], np.uint32).view(np.uint8)
    if kxcode_words is not None:
        o = lay["key_xcodes"] + 4 * slot * (w // 2)
        sb[o: o + 4 * (w // 2)] = np.asarray(kxcode_words, np.uint32).view(np.uint8)
    if key_qjl == 1:
        o = lay["key_signs"] + 4 * slot * w
        sb[o: o + 4 * w] = np.asarray(ksign_words, np.uint32).view(np.uint8)
    sb[lay["value_norm"] + 4 * slot: lay["value_norm"] + 4 * slot + 4] = np.array([vnorm], np.float32).view(np.uint8)
    o = lay["value_codes"]
    vc = sb[o: o + 2 * value_bits * d].view(np.uint16).reshape(value_bits, d)
    bit = np.uint16(1 << slot)
    vc &= np.uint16(~bit & 0xFFFF)
    vc |= (np.asarray(vcode_planes_bits, np.uint16) << np.uint16(slot)).astype(np.uint16)


def read_page(pool: np.ndarray, lay: dict, n_heads: int, page: int, head: int,
              d: int, key_bits: int, key_qjl: bool, value_bits: int,
              key_split: int = 0, norm_range: tuple[float, float] | None = None) -> dict:
    """Decode all P records of one (page, head) sub-block back to arrays.
    norm_range = (lo, hi): key norms are byte codes (kept as "knorm_code",
    decoded into "knorm")."""
    from .codec import norm_u8_decode, planes_to_idx, unpack_bits, unpack_codes_split

    base = (page * n_heads + head) * lay["bytes"]
    sb = np.ascontiguousarray(pool[base: base + lay["bytes"]])
    w = d // 32
    if norm_range is not None:
        code = sb[lay["key_norm"]: lay["key_norm"] + PAGE].copy()
        out = {"knorm_code": code, "knorm": norm_u8_decode(code, *norm_range)}
    else:
        out = {"knorm": sb[lay["key_norm"]: lay["key_norm"] + 4 * PAGE].view(np.float32).copy()}
    if key_qjl:
        out["krnorm"] = sb[lay["key_rnorm"]: lay["key_rnorm"] + 4 * PAGE].view(np.float32).copy()
    if key_qjl == 1:
        sw = sb[lay["key_signs"]: lay["key_signs"] + 4 * PAGE * w].view(np.uint32).reshape(PAGE, w)
        out["ksigns"] = unpack_bits(sw, d).astype(bool)
    cw = sb[lay["key_codes"]: lay["key_codes"] + 4 * key_bits * PAGE * w].view(np.uint32).reshape(key_bits, PAGE, w)
    if key_split:
        xw = sb[lay["key_xcodes"]: lay["key_xcodes"] + 4 * PAGE * (w // 2)].view(np.uint32).reshape(PAGE, w // 2)
        out["kidx"] = unpack_codes_split(cw.transpose(1, 0, 2), xw, key_bits, d)
    else:
        kplanes = np.stack([unpack_bits(cw[p], d) for p in range(key_bits)], axis=1)  # [P, bits, d]
        out["kidx"] = planes_to_idx(kplanes)
    out["vnorm"] = sb[lay["value_norm"]: lay["value_norm"] + 4 * PAGE].view(np.float32).copy()
    vc = sb[lay["value_codes"]: lay["value_codes"] + 2 * value_bits * d].view(np.uint16).reshape(value_bits, d)
    vplanes = ((vc[None, :, :] >> np.arange(PAGE, dtype=np.uint16)[:, None, None]) & 1).astype(np.uint8)
    out["vidx"] = planes_to_idx(vplanes)  # [P, d]
    return out


def ring_capacity(W: int, P: int = PAGE) -> int:
    """Window ring slots per (sequence, kv head): W + P."""
    return W + P


def ring_slot(pos: int, W: int, P: int = PAGE) -> int:
    """Token position pos of a window token lives at ring slot pos mod (W + P)."""
    return pos % (W + P)


def decode_append_step(T: int, W: int, P: int = PAGE) -> tuple[int, bool]:
    """State change of one decode-step append to a sequence of length T.

    The new token (position T) goes to ring slot T mod (W + P).  If the window
    then holds W + P tokens, its oldest P tokens (positions n_c .. n_c + P - 1)
    are quantized into compressed page n_c / P.  Returns (n_c after the step,
    whether a page was flushed).
    """
    nc0 = n_compressed(T, W, P)
    nc1 = n_compressed(T + 1, W, P)
    return nc1, nc1 != nc0
