"""Decode attention scored directly in the compressed domain.

[Design study] §Transform placement: keys are quantized after RoPE and the
query is moved into the same rotated basis, q^T k = (T q)^T (T k); scores are
accumulated against packed key codes without reconstructing the history, and
value pages are streamed after the softmax.  §CPU and WASM kernel design
("Decode-time key scan", "Decode-time value scan", "Accumulator width"): the
query is transformed once per layer and head, value accumulation happens in
the transform domain with the inverse transform applied once to the head
output, and scores and outputs accumulate in FP32 (here float64).

Score of a compressed token i for query head h (KV head g = h // G):
  q' = Pi_g q,  q'' = S_g q',
  l_i = scale * n_i * ( <q', C[idx_i]> / sqrt(d)
                        + sqrt(pi/2)/d * gamma_i * <q'', 2 s_i - 1> )
([Reconstruction] §6 "The Asymmetric Unbiased Estimator": the inner product
estimate is <q', y_hat> + sqrt(pi/2)/d ||r|| <S q', sign(S r)>; C is
RMS-scaled so y_hat = C[idx] / sqrt(d)).  Window token (float16, unrotated):
l_i = scale * <q, k_i>.  The softmax scale is a caller argument (1/sqrt(d)
is the usual value; the pages do not state one).

Output:  o = Pi_v^T ( sum_{compressed} p_i m_i C_v[vidx_i] / sqrt(d) )
             + sum_{window} p_i v_i,     p = softmax(l) over all T tokens.
GQA: query head h reads KV head h // (Hq / Hkv); every cached token is
visible to the decode query.
"""

from __future__ import annotations

import math

import numpy as np

from . import transforms as T
from .codec import centroid_values, qjl_constant


def decode_one(q: np.ndarray, comp: dict | None, win_k: np.ndarray | None, win_v: np.ndarray | None,
               params: dict, scale: float) -> dict:
    """One sequence.

    q      : [Hq, d] query (float64 exact copy of the input).
    comp   : compressed tokens of this sequence, per KV head lists of arrays:
             knorm [Hkv, Tc], krnorm [Hkv, Tc], kidx [Hkv, Tc, d],
             ksigns [Hkv, Tc, d] (bool), vnorm [Hkv, Tc], vidx [Hkv, Tc, d].
    win_k, win_v : [Hkv, Tw, d] float16 window tokens (oldest first), or None.
    params : kind, k_rot[Hkv], v_rot[Hkv], qjl_s[Hkv] (stored float32 arrays),
             k_cb, v_cb (Codebook), key_qjl: key correction (0 none, 1 QJL,
             2 EDEN scale, 3 TurboVec length-renormalized correction; krnorm holds gamma or s);
             optional k_cb_hi: mixed-channel key rate (coordinates < d/2 read
             this book).  knorm holds decoded norms (byte norms decoded).
    Returns out [Hq, d], lse [Hq], scores [Hq, T] (compressed first, then window).
    """
    Hq, d = q.shape
    Hkv = len(params["k_rot"])
    G = Hq // Hkv
    kind = params["kind"]
    kap = qjl_constant(d)
    Cv = np.asarray(params["v_cb"].centroids, np.float32).astype(np.float64)
    Tc = 0 if comp is None else comp["knorm"].shape[1]
    Tw = 0 if win_k is None else win_k.shape[1]
    out = np.zeros((Hq, d))
    lse = np.zeros(Hq)
    scores = np.zeros((Hq, Tc + Tw))
    for h in range(Hq):
        g = h // G
        qh = np.asarray(q[h], np.float64)
        parts = []
        if Tc:
            q1 = T.rotate(kind, params["k_rot"][g], qh[None, :])[0]
            l_c = centroid_values(comp["kidx"][g], params["k_cb"], params.get("k_cb_hi")) @ q1 / math.sqrt(d)
            corr = int(params["key_qjl"])
            if corr == 1:  # QJL residual term
                q2 = np.asarray(params["qjl_s"][g], np.float32).astype(np.float64) @ q1
                pm = np.where(comp["ksigns"][g], 1.0, -1.0)
                l_c = l_c + kap * comp["krnorm"][g].astype(np.float64) * (pm @ q2)
            elif corr >= 2:  # EDEN or length-renormalized keys: the per-key scale
                l_c = l_c * comp["krnorm"][g].astype(np.float64)
            l_c = scale * comp["knorm"][g].astype(np.float64) * l_c
            parts.append(l_c)
        if Tw:
            parts.append(scale * (win_k[g].astype(np.float64) @ qh))
        l = np.concatenate(parts) if parts else np.zeros(0)
        scores[h] = l
        if l.size == 0:
            continue
        mx = np.max(l)
        e = np.exp(l - mx)
        den = np.sum(e)
        p = e / den
        lse[h] = mx + math.log(den)
        o = np.zeros(d)
        if Tc:
            acc_rot = (p[:Tc] * comp["vnorm"][g].astype(np.float64)) @ (Cv[comp["vidx"][g]] / math.sqrt(d))
            o += T.rotate_inverse(kind, params["v_rot"][g], acc_rot[None, :])[0]
        if Tw:
            o += p[Tc:] @ win_v[g].astype(np.float64)
        out[h] = o
    return {"out": out, "lse": lse, "scores": scores}


def exact_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> dict:
    """Textbook softmax attention for one sequence: q [Hq, d], K, V [Hkv, T, d]."""
    Hq, d = q.shape
    Hkv = K.shape[0]
    G = Hq // Hkv
    out = np.zeros((Hq, d))
    lse = np.zeros(Hq)
    scores = np.zeros((Hq, K.shape[1]))
    for h in range(Hq):
        g = h // G
        l = scale * (np.asarray(K[g], np.float64) @ np.asarray(q[h], np.float64))
        mx = l.max()
        e = np.exp(l - mx)
        out[h] = (e / e.sum()) @ np.asarray(V[g], np.float64)
        lse[h] = mx + math.log(e.sum())
        scores[h] = l
    return {"out": out, "lse": lse, "scores": scores}
