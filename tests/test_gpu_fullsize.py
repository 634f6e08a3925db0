"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (automatic split count), checked on sampled sequences the oracle
recomputes on its own.  For each sampled sequence every page record of every
kv head is compared with the oracle's (codes and signs bit-exact outside the
boundary band, norms to 1e-6), and the decode is compared on every score, the
log-sum-exp and the output of all query heads against the oracle's decode of
its own records with the GPU's choices adopted exactly where the rules accept
either decision (so no token is skipped).  The same cache then serves a
64-token prefill-attention chunk (the bench's), its first and last queries
checked against the oracle's decode over their visible positions.  Workloads: Qwen-like (batch 8,
32768 tokens, window 128, FWHT, keys 2b + QJL, values 2b), Llama-like (batch
32, 8192 tokens, no window, dense Pi, outlier channels, keys 3b + QJL, values
4b) and long context (one sequence of 131072 tokens, 8192 pages split over the
grid).  Sequences are independent in decode, so the unsampled ones are filled
on the device by another generator.
"""

import math

import numpy as np
import pytest

import synthetic_kv as SK
import parity as PY

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CASES = [("qwen", (0, 5)), ("llama", (0, 17)), ("long", (0,))]


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from kv_cache_vector_head_gb300 import build

    build.build()
    import kv_cache_vector_head_gb300 as tq

    return tq


@pytest.mark.parametrize("name,sampled", CASES)
def test_fullsize_decode_sampled_sequences(tq, name, sampled):
    w = SK.workload(name)
    SAMPLED = sampled
    B, T, W = w.batch, w.ctx, w.window
    L = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=W)
    O = PY.OracleLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=W)
    pc = tq.PagedCache(L, B, T)
    K_all, V_all, q_all = SK.keys_values_torch(w)
    kv = {}
    for b in SAMPLED:
        s = SK.keys_values(w, seqs=[b])
        K_all[b] = SK.to_torch(s["K"][0], w.dtype).cuda()
        V_all[b] = SK.to_torch(s["V"][0], w.dtype).cuda()
        q_all[b] = SK.to_torch(s["q"][0], w.dtype).cuda()
        kv[b] = s
    pc.prefill(K_all, V_all)
    del K_all, V_all
    ws = torch.empty(tq.decode_workspace_size(L.params, B, T), dtype=torch.uint8, device="cuda")
    out = torch.zeros(B, w.n_q_heads, w.d, device="cuda")
    lse = torch.zeros(B, w.n_q_heads, device="cuda")
    scores = torch.zeros(B, w.n_q_heads, T, device="cuda")
    scale = 1.0 / math.sqrt(w.d)
    tq.decode_attention(L.params, pc.cache, q_all, scale, out, lse, scores, ws, T)
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    nc = 16 * ((T - W) // 16)
    assert pc.n_compressed.cpu().tolist() == [nc] * B and pc.seq_len.cpu().tolist() == [T] * B
    pool = pc.pool.cpu().numpy()
    bt = pc.block_table.cpu().numpy()
    stats = {}
    adopted = {}
    for b in SAMPLED:
        s = kv[b]
        recs_k = [O.keys(s["K"][0, :nc, h], h) for h in range(w.n_kv_heads)]
        recs_v = [O.values(s["V"][0, :nc, h], h) for h in range(w.n_kv_heads)]
        # every page record of the sequence, then the oracle records with the GPU's accepted choices
        ad_k, ad_v = [], []
        for h in range(w.n_kv_heads):
            g = PY.read_pages(pool, O, bt[b, : nc // 16], h)
            PY.compare_records(recs_k[h], g["kidx"], g["knorm"], g["ksigns"], g["krnorm"], True, stats)
            PY.compare_records(recs_v[h], g["vidx"], g["vnorm"], is_key=False, stats=stats)
            ad_k.append(PY.adopt_exempt(recs_k[h], g["kidx"], g["ksigns"], g["krnorm"]))
            ad_v.append(PY.adopt_exempt(recs_v[h], g["vidx"]))
        assert stats["exempt"] <= max(3, PY.EXEMPT_FRACTION * stats["codes"])
        win_k = s["K"][0, nc:T].transpose(1, 0, 2).astype(np.float16) if T > nc else None
        win_v = s["V"][0, nc:T].transpose(1, 0, 2).astype(np.float16) if T > nc else None
        ref = PY.decode_reference(O, s["q"][0], PY.stack_comp(ad_k, ad_v), win_k, win_v, scale)
        err = np.abs(scores[b].cpu().numpy() - ref["scores"])
        assert err.max() < PY.SCORE_ATOL, err.max()
        assert np.abs(out[b].cpu().numpy() - ref["out"]).max() < PY.OUT_ATOL
        assert np.abs(lse[b].cpu().numpy() - ref["lse"]).max() < PY.SCORE_ATOL
        adopted[b] = (ad_k, ad_v)

    # prefill attention of the last 64 tokens (the bench's chunk) on the same cache: sampled
    # queries against the oracle's decode over positions 0 .. p of the adopted records
    nq = 64
    rng = np.random.default_rng(4321)
    qp = rng.standard_normal((B, nq, w.n_q_heads, w.dh)).astype(np.float32)
    qpt = SK.to_torch(qp, w.dtype).cuda()
    qp = qpt.float().cpu().numpy().astype(np.float64)
    pws = torch.empty(tq.prefill_workspace_size(L.params, B, nq, T), dtype=torch.uint8, device="cuda")
    pout = torch.zeros(B, nq, w.n_q_heads, w.dh, device="cuda")
    plse = torch.zeros(B, nq, w.n_q_heads, device="cuda")
    tq.prefill_attention(L.params, pc.cache, nq, qpt, scale, pout, plse, pws, T)
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    pout, plse = pout.cpu().numpy(), plse.cpu().numpy()
    for b in SAMPLED:
        s = kv[b]
        ad_k, ad_v = adopted[b]
        for i in (0, nq - 1):
            Ti = T - nq + i + 1
            nci = min(nc, Ti)
            comp = PY.stack_comp([_trunc(r, nc, nci) for r in ad_k], [_trunc(r, nc, nci) for r in ad_v])
            wk = s["K"][0, nci:Ti].transpose(1, 0, 2).astype(np.float16) if Ti > nci else None
            wv = s["V"][0, nci:Ti].transpose(1, 0, 2).astype(np.float16) if Ti > nci else None
            r = PY.decode_reference(O, qp[b, i], comp, wk, wv, scale)
            assert np.abs(pout[b, i] - r["out"]).max() < PY.OUT_ATOL, (b, i)
            assert np.abs(plse[b, i] - r["lse"]).max() < PY.SCORE_ATOL, (b, i)


def _trunc(rec, n_all, n):
    """The first n token records of an oracle record dict holding n_all tokens."""
    return {k: (v[:n] if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == n_all else v)
            for k, v in rec.items()}
