"""Parity helpers: the oracle's expected records and the comparison rules.

Tolerances:
* packed codes and QJL signs bit-exact, except coordinates within 1e-5 of a
  decision boundary (z units for codes; (S r)_j for the sign of a unit-vector
  residual), which must stay under 1e-4 of all codes and are counted; a code
  flip there changes r, gamma and the signs of that vector, so those are
  exempted for that vector too;
* norms n, m and gamma within 1e-6 relative; byte key norms (u8 log-norm)
  bit-exact except within 1e-4 code units of a decision point (the GPU takes
  log2 in float32: its error there is below 5e-5 code units), counted with
  the codes;
* attention scores within 1e-3 and outputs within 2e-3 absolute (fp32).
"""

from __future__ import annotations

import math

import numpy as np

from oracle import attention as OA
from oracle import codebook as OCB
from oracle import codec as OC
from oracle import paging as OP
from oracle import transforms as OT

BOUNDARY = 1e-5
NORM_RTOL = 1e-6
SCORE_ATOL = 1e-3
OUT_ATOL = 2e-3
EXEMPT_FRACTION = 1e-4
NORM_CODE_BAND = 1e-4


class OracleLayer:
    def __init__(self, d, hkv, hq, kb, vb, kind, window=0, qjl=True, seed=0, layer=0, key_split=0,
                 key_norm_range=None, qjl_structured=0):
        """qjl: key correction (False/0 none, True/1 QJL, 2 EDEN scale, 3 length renormalization).
        key_split: mixed-channel key rate; key_norm_range: (lo, hi) of the byte key norms."""
        self.d, self.hkv, self.hq, self.kb, self.vb, self.kind = d, hkv, hq, kb, vb, kind
        self.window, self.qjl = window, int(qjl)
        self.key_split, self.norm_range = int(key_split), key_norm_range
        self.kcb = OCB.lloyd_max(d, kb)
        self.kcb_hi = OCB.lloyd_max(d, kb + 1) if key_split else None
        self.vcb = OCB.lloyd_max(d, vb)
        self.k_rot = [OT.build_transform(kind, d, seed, layer, h, 0) for h in range(hkv)]
        self.v_rot = [OT.build_transform(kind, d, seed, layer, h, 1) for h in range(hkv)]
        if self.qjl == 1 and qjl_structured:  # S = H diag(sigma_S), +-1 entries
            self.S = [OT.structured_qjl_matrix(OT.build_transform(kind, d, seed, layer, h, OT.ROLE_QJL_SIGNS), d)
                      for h in range(hkv)]
        elif self.qjl == 1:
            self.S = [OT.build_transform(kind, d, seed, layer, h, 2) for h in range(hkv)]
        else:
            self.S = None

    def keys(self, x, head):
        """Key records; with byte norms also norm_code, its margin and norm_dec (the decoded norm)."""
        x = OC.pad_head(x, self.d)  # heads shorter than d: zero-padded to the transform size
        if self.qjl == 1:
            rec = OC.quantize_prod(x, self.kind, self.k_rot[head], self.kcb, self.S[head])
        elif self.qjl >= 2:
            rec = OC.quantize_scaled(x, self.kind, self.k_rot[head], self.kcb, self.qjl, cb_hi=self.kcb_hi)
        else:
            rec = OC.quantize_mse(x, self.kind, self.k_rot[head], self.kcb, cb_hi=self.kcb_hi)
        if self.norm_range is not None:
            code, margin = OC.norm_u8_encode(rec["norm_f64"], *self.norm_range)
            rec.update({"norm_code": code, "norm_code_margin": margin,
                        "norm_dec": OC.norm_u8_decode(code, *self.norm_range)})
        return rec

    def values(self, x, head):
        return OC.quantize_mse(OC.pad_head(x, self.d), self.kind, self.v_rot[head], self.vcb)

    def attention_params(self):
        return {"kind": self.kind, "k_rot": self.k_rot, "v_rot": self.v_rot, "qjl_s": self.S,
                "k_cb": self.kcb, "k_cb_hi": self.kcb_hi, "v_cb": self.vcb, "key_qjl": self.qjl}


def exempt_mask(rec, is_key):
    """Per-vector exemption: any coordinate within BOUNDARY of a decision."""
    ex = rec["margin"] < BOUNDARY
    if is_key and "sign_margin" in rec:
        ex = ex | (rec["sign_margin"] < BOUNDARY)
    return ex


def compare_records(ora, g_idx, g_norm, g_signs=None, g_rnorm=None, is_key=True, stats=None, exact=False,
                    g_norm_code=None):
    """Compare GPU records (code indices [N, d], norms [N], signs [N, d] bool,
    rnorms [N]) with the oracle's; returns counts and asserts the rules.
    exact=True (crafted inputs whose decisions are exactly computable, e.g.
    a zero vector lying on the z = 0 boundary) demands equality everywhere.
    g_norm_code: byte key norms, compared with the oracle's codes in place of g_norm."""
    idx = ora["idx"]
    if g_norm_code is not None:
        band = ora["norm_code_margin"] < NORM_CODE_BAND
        dc = np.abs(g_norm_code.astype(np.int64) - ora["norm_code"].astype(np.int64))
        assert not ((dc != 0) & ~band).any(), f"{int(((dc != 0) & ~band).sum())} byte norm mismatches"
        assert dc.max(initial=0) <= 1
        if stats is not None:
            stats["exempt"] = stats.get("exempt", 0) + int(band.sum())
            stats["codes"] = stats.get("codes", 0) + band.size
        g_norm = None  # the float norm is not stored
    if exact:
        assert np.array_equal(g_idx, idx)
        if g_norm is not None:
            np.testing.assert_allclose(g_norm.astype(np.float64), ora["norm"].astype(np.float64), rtol=NORM_RTOL,
                                       atol=0)
        if is_key and g_signs is not None:
            assert np.array_equal(g_signs, ora["signs"])
            np.testing.assert_allclose(g_rnorm.astype(np.float64), ora["rnorm"].astype(np.float64),
                                       rtol=NORM_RTOL, atol=0)
        return {"exempt": 0, "flipped": 0, "total": idx.size}
    code_ex = ora["margin"] < BOUNDARY
    diff = g_idx != idx
    bad = diff & ~code_ex
    assert not bad.any(), f"{bad.sum()} code mismatches outside the boundary band"
    vec_flip = diff.any(axis=1)
    if g_norm is not None:
        np.testing.assert_allclose(g_norm.astype(np.float64), ora["norm"].astype(np.float64), rtol=NORM_RTOL,
                                   atol=1e-30)
    n_exempt_codes = int(code_ex.sum())
    if is_key and g_signs is None and g_rnorm is not None:  # EDEN / length-renormalized keys: the scale
        ok = ~vec_flip
        np.testing.assert_allclose(g_rnorm[ok].astype(np.float64), ora["rnorm"][ok].astype(np.float64),
                                   rtol=NORM_RTOL, atol=1e-30)
    if is_key and g_signs is not None:
        sign_ex = (ora["sign_margin"] < BOUNDARY) | vec_flip[:, None]
        sbad = (g_signs != ora["signs"]) & ~sign_ex
        assert not sbad.any(), f"{sbad.sum()} sign mismatches outside the exemption"
        ok = ~vec_flip
        np.testing.assert_allclose(g_rnorm[ok].astype(np.float64), ora["rnorm"][ok].astype(np.float64),
                                   rtol=NORM_RTOL, atol=1e-30)
        n_exempt_codes += int((ora["sign_margin"] < BOUNDARY).sum())
    total = idx.size * (2 if (is_key and g_signs is not None) else 1)
    if stats is not None:
        stats["exempt"] = stats.get("exempt", 0) + n_exempt_codes
        stats["codes"] = stats.get("codes", 0) + total
        stats["flipped"] = stats.get("flipped", 0) + int(diff.sum())
    if stats is None:  # callers that pass stats check the fraction over the whole call
        assert n_exempt_codes <= max(3, EXEMPT_FRACTION * total), (n_exempt_codes, total)
    return {"exempt": n_exempt_codes, "flipped": int(diff.sum()), "total": total}


def adopt_exempt(rec, g_idx, g_signs=None, g_rnorm=None, g_norm_code=None, norm_range=None):
    """A copy of the oracle record that takes the GPU's decisions exactly where
    the parity rules accept either one: codes of coordinates within BOUNDARY of
    a boundary, QJL signs within BOUNDARY of zero, and the signs and residual
    norm of a vector whose code changed.  Everything else stays the oracle's,
    so a decode computed from the copy is compared without exemptions."""
    out = dict(rec)
    if g_norm_code is not None and "norm_code" in rec:
        band = rec["norm_code_margin"] < NORM_CODE_BAND
        code = np.where(band, g_norm_code, rec["norm_code"]).astype(np.uint8)
        out["norm_code"], out["norm_dec"] = code, OC.norm_u8_decode(code, *norm_range)
    ex = rec["margin"] < BOUNDARY
    idx = rec["idx"].copy()
    idx[ex] = g_idx[ex]
    out["idx"] = idx
    if g_signs is None and g_rnorm is not None and "rnorm" in rec:  # scale of EDEN / length-renormalized keys
        flip = (idx != rec["idx"]).any(axis=1)
        rn = rec["rnorm"].copy()
        rn[flip] = g_rnorm[flip]
        out["rnorm"] = rn
    if g_signs is not None and "signs" in rec:
        flip = (idx != rec["idx"]).any(axis=1)
        sex = (rec["sign_margin"] < BOUNDARY) | flip[:, None]
        sg = rec["signs"].copy()
        sg[sex] = g_signs[sex]
        out["signs"] = sg
        rn = rec["rnorm"].copy()
        rn[flip] = g_rnorm[flip]
        out["rnorm"] = rn
    return out


def unpack_flat_codes(words, bits, d, split=False):
    if split:  # bits full planes, then the top plane of the first d/64 words
        w = words.reshape(-1, bits * d // 32 + d // 64)
        return OC.unpack_codes_split(w[:, : bits * d // 32].reshape(-1, bits, d // 32), w[:, bits * d // 32:], bits, d)
    return OC.unpack_codes(words.reshape(-1, bits, d // 32), bits, d)


def unpack_flat_bits(words, d):
    return OC.unpack_bits(words.reshape(-1, d // 32), d).astype(bool)


def decode_reference(ol: OracleLayer, q, comp, win_k, win_v, scale):
    """Decode of one sequence; q (and window tokens) of head_dim <= d
    coordinates are zero-padded to d, the output keeps head_dim."""
    dh = q.shape[-1]
    pw = (lambda w: None if w is None else OC.pad_head(w, ol.d).astype(w.dtype))
    r = OA.decode_one(OC.pad_head(q, ol.d), comp, pw(win_k), pw(win_v), ol.attention_params(), scale)
    if dh != ol.d:
        r = dict(r, out=r["out"][..., :dh])
    return r


def stack_comp(recs_k, recs_v):
    """Per-kv-head oracle records -> the comp dict of oracle.attention."""
    comp = {"knorm": np.stack([r["norm_dec"] if "norm_dec" in r else r["norm"] for r in recs_k]),
            "kidx": np.stack([r["idx"] for r in recs_k]),
            "vnorm": np.stack([r["norm"] for r in recs_v]), "vidx": np.stack([r["idx"] for r in recs_v])}
    if "rnorm" in recs_k[0]:
        comp["krnorm"] = np.stack([r["rnorm"] for r in recs_k])
        comp["ksigns"] = (np.stack([r["signs"] for r in recs_k]) if "signs" in recs_k[0]
                          else np.ones(comp["kidx"].shape, dtype=bool))
    else:
        comp["krnorm"] = np.zeros_like(comp["knorm"])
        comp["ksigns"] = np.ones(comp["kidx"].shape, dtype=bool)
    return comp


def read_pool(pool_bytes: np.ndarray, ol: OracleLayer, page: int, head: int) -> dict:
    lay = OP.subblock_layout(ol.d, ol.kb, ol.qjl, ol.vb, key_split=ol.key_split,
                             key_norm_u8=int(ol.norm_range is not None))
    return OP.read_page(pool_bytes, lay, ol.hkv, page, head, ol.d, ol.kb, ol.qjl, ol.vb, key_split=ol.key_split,
                        norm_range=ol.norm_range)


def read_pages(pool_bytes: np.ndarray, ol: OracleLayer, pages, head: int) -> dict:
    """The records of the (page, head) sub-blocks of `pages`, in order, as arrays over all their
    tokens: the same decoding as oracle.paging.read_page, batched over pages (uniform-rate keys
    with float32 norms).  Returns kidx [n, d], knorm, krnorm, ksigns (QJL), vidx, vnorm."""
    lay = OP.subblock_layout(ol.d, ol.kb, ol.qjl, ol.vb)
    P, w, d = OP.PAGE, ol.d // 32, ol.d
    pages = np.asarray(pages, dtype=np.int64)
    sb = pool_bytes.reshape(-1, ol.hkv, lay["bytes"])[pages, head]          # [np, bytes]
    f32 = lambda off, n: np.ascontiguousarray(sb[:, off: off + 4 * n]).view(np.float32).reshape(-1)
    u32 = lambda off, n: np.ascontiguousarray(sb[:, off: off + 4 * n]).view(np.uint32)
    out = {"knorm": f32(lay["key_norm"], P)}
    if ol.qjl:
        out["krnorm"] = f32(lay["key_rnorm"], P)
    if ol.qjl == 1:
        out["ksigns"] = OC.unpack_bits(u32(lay["key_signs"], P * w).reshape(-1, P, w), d).reshape(-1, d).astype(bool)
    cw = u32(lay["key_codes"], ol.kb * P * w).reshape(-1, ol.kb, P, w).transpose(0, 2, 1, 3)   # [np, P, kb, w]
    out["kidx"] = OC.unpack_codes(cw.reshape(-1, ol.kb, w), ol.kb, d)
    out["vnorm"] = f32(lay["value_norm"], P)
    vc = np.ascontiguousarray(sb[:, lay["value_codes"]: lay["value_codes"] + 2 * ol.vb * d]).view(np.uint16)
    vc = vc.reshape(-1, ol.vb, d)
    vplanes = ((vc[:, None, :, :] >> np.arange(P, dtype=np.uint16)[None, :, None, None]) & 1).astype(np.uint8)
    out["vidx"] = OC.planes_to_idx(vplanes.reshape(-1, ol.vb, d))
    return out
