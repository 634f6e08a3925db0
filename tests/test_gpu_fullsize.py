"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (automatic split count), checked on sampled sequences the oracle
recomputes on its own: every non-exempt score, the log-sum-exp and the output
of all query heads of the sampled sequences, plus the page records of sampled
pages.  Workloads: Qwen-like (batch 8, 32768 tokens, window 128, FWHT, keys
2b + QJL, values 2b), Llama-like (batch 32, 8192 tokens, no window, dense Pi,
outlier channels, keys 3b + QJL, values 4b) and long context (one sequence of
131072 tokens, 8192 pages split over the grid).  Sequences are independent in
decode, so the unsampled ones are filled on the device by another generator.
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
    for b in SAMPLED:
        s = kv[b]
        recs_k = [O.keys(s["K"][0, :nc, h], h) for h in range(w.n_kv_heads)]
        recs_v = [O.values(s["V"][0, :nc, h], h) for h in range(w.n_kv_heads)]
        # sampled page records: first, middle and last compressed page of each head
        for h in range(w.n_kv_heads):
            for p in (0, nc // 32, nc // 16 - 1):
                pg = PY.read_pool(pool, O, int(bt[b, p]), h)
                sl = slice(16 * p, 16 * p + 16)
                sub_k = {k: v[sl] for k, v in recs_k[h].items() if isinstance(v, np.ndarray) and v.shape[:1] == (nc,)}
                sub_v = {k: v[sl] for k, v in recs_v[h].items() if isinstance(v, np.ndarray) and v.shape[:1] == (nc,)}
                PY.compare_records(sub_k, pg["kidx"], pg["knorm"], pg["ksigns"], pg["krnorm"], True, stats)
                PY.compare_records(sub_v, pg["vidx"], pg["vnorm"], is_key=False, stats=stats)
        assert stats["exempt"] <= max(3, PY.EXEMPT_FRACTION * stats["codes"])
        win_k = s["K"][0, nc:T].transpose(1, 0, 2).astype(np.float16) if T > nc else None
        win_v = s["V"][0, nc:T].transpose(1, 0, 2).astype(np.float16) if T > nc else None
        ref = PY.decode_reference(O, s["q"][0], PY.stack_comp(recs_k, recs_v), win_k, win_v, scale)
        g_sc = scores[b].cpu().numpy()
        G = w.n_q_heads // w.n_kv_heads
        n_ex = 0
        for g in range(w.n_kv_heads):
            # tokens whose key record (of this kv head) has a near-boundary coordinate are counted, not compared
            ex = np.zeros(T, dtype=bool)
            ex[:nc] = PY.exempt_mask(recs_k[g], True).any(axis=1)
            n_ex += int(ex.sum())
            err = np.abs(g_sc[g * G:(g + 1) * G] - ref["scores"][g * G:(g + 1) * G])[:, ~ex]
            assert err.max() < PY.SCORE_ATOL, err.max()
        assert n_ex <= 0.05 * T * w.n_kv_heads
        assert np.abs(out[b].cpu().numpy() - ref["out"]).max() < PY.OUT_ATOL
        assert np.abs(lse[b].cpu().numpy() - ref["lse"]).max() < PY.SCORE_ATOL
