"""GPU-vs-oracle parity of the CUDA path, through the C ABI.

Every case draws seeded synthetic inputs with the workload recipes of
synthetic_kv (reduced batch / context so the oracle finishes in seconds),
runs libtq on cuda:0 and compares element by element with the oracle's own
quantization and attention, under the tolerances in tests/parity.py.
"""

import math

import numpy as np
import pytest

import synthetic_kv as SK
import parity as PY

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from kv_cache_vector_head_gb300 import build

    build.build()
    import kv_cache_vector_head_gb300 as tq

    return tq


def _layer(tq, w, layer=0):
    L = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=w.window,
                   key_qjl=w.key_qjl, seed=w.seed, layer=layer, head_dim=w.dh, key_split=w.key_split,
                   key_norm_range=w.key_norm_range, qjl_structured=w.qjl_structured)
    O = PY.OracleLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=w.window,
                       qjl=w.key_qjl, seed=w.seed, layer=layer, key_split=w.key_split,
                       key_norm_range=w.key_norm_range, qjl_structured=w.qjl_structured)
    return L, O


CASES = [
    ("tiny", dict(ctx=200)),
    ("qwen", dict(batch=1, ctx=61)),
    ("llama", dict(batch=1, ctx=53)),
    ("long", dict(ctx=37)),
    ("bulk", dict(ctx=70)),
    ("tiny", dict(ctx=50, kind=SK.FWHT, key_bits=1, value_bits=1)),
    ("qwen", dict(batch=1, ctx=40, kind=SK.DENSE, key_bits=4, value_bits=3, key_qjl=False)),
    # d = 128 bf16: the tensor-core bulk path (several tiles per warp, ragged tail)
    ("bulk", dict(ctx=300, kind=SK.FWHT)),
    ("bulk", dict(ctx=4100)),
    ("llama", dict(batch=2, ctx=45, kind=SK.FWHT, key_bits=2, value_bits=1)),
    ("bulk", dict(ctx=400, key_bits=4, value_bits=2)),
    ("bulk", dict(ctx=5000, kind=SK.FWHT, key_bits=4, value_bits=3)),
    # FWHT with the rotation on tcgen05: more 128-token tiles per head than the grid's groups
    ("bulk", dict(ctx=6000, kind=SK.FWHT)),
    ("bulk", dict(ctx=20, kind=SK.FWHT, key_bits=1, key_qjl=False, value_bits=4)),
    ("bulk", dict(ctx=21, key_bits=2, key_qjl=False, value_bits=1)),
    # head sizes that are not powers of two, zero-padded to the transform size
    ("bulk", dict(ctx=300, kind=SK.FWHT, head_dim=80)),
    ("bulk", dict(ctx=200, head_dim=96, key_bits=2, value_bits=3)),
    ("tiny", dict(ctx=60, head_dim=120)),
    ("long", dict(ctx=33, head_dim=160)),
    # EDEN-unbiased (2) and length-renormalized (3) keys: a scale in place of the QJL sketch,
    # through the warp tiles (d = 128 bf16, FWHT and dense) and the CUDA-core tiles
    ("bulk", dict(ctx=300, kind=SK.FWHT, key_qjl=2)),
    ("bulk", dict(ctx=400, key_bits=4, key_qjl=3)),
    ("bulk", dict(ctx=130, kind=SK.FWHT, key_bits=1, key_qjl=2)),
    ("bulk", dict(ctx=90, key_bits=3, key_qjl=2, head_dim=96)),
    ("tiny", dict(ctx=70, key_qjl=3)),
    ("long", dict(ctx=30, key_qjl=2)),
    # mixed-channel keys (coordinates < d/2 one bit wider) with every correction but the sketch;
    # byte norms leave the flat output's float norms as they are
    ("mixed", dict(batch=1, ctx=40)),
    ("bulk", dict(ctx=300, kind=SK.FWHT, key_bits=3, key_qjl=0, key_split=1, value_bits=3)),
    ("qwen", dict(batch=1, ctx=40, key_bits=2, key_qjl=2, key_split=1)),
    ("tiny", dict(ctx=60, key_bits=1, key_qjl=3, key_split=1, key_norm_range=(-4.0, 12.0))),
    ("bulk", dict(ctx=90, key_bits=3, key_qjl=0, key_split=1, head_dim=96)),
    # the structured sketch S = H diag(sigma_S), FWHT and dense rotations
    ("qwen", dict(batch=1, ctx=40, qjl_structured=1)),
    ("bulk", dict(ctx=300, kind=SK.FWHT, qjl_structured=1)),
    ("bulk", dict(ctx=4100, kind=SK.DENSE, qjl_structured=1, key_bits=2)),
    ("tiny", dict(ctx=60, qjl_structured=1, key_bits=1)),
    ("long", dict(ctx=30, qjl_structured=1, head_dim=160)),
]


@pytest.mark.parametrize("name,over", CASES)
def test_quantize_flat_parity(tq, name, over):
    w = SK.workload(name, **over)
    kv = SK.keys_values(w)
    L, O = _layer(tq, w)
    dt = w.dtype
    K = kv["K"].reshape(-1, w.dh)
    V = kv["V"].reshape(-1, w.dh)
    n_vec = K.shape[0] - 1  # ragged: the last token is missing its last head
    kt = SK.to_torch(K, dt).cuda()
    vt = SK.to_torch(V, dt).cuda()
    E = w.d // 32
    kwords = w.key_bits * E + (E // 2 if w.key_split else 0)
    codes = torch.zeros(n_vec, kwords, dtype=torch.int32, device="cuda")
    signs = torch.zeros(n_vec, E, dtype=torch.int32, device="cuda") if w.key_qjl == 1 else None
    norms = torch.zeros(n_vec, device="cuda")
    rn = torch.zeros(n_vec, device="cuda") if w.key_qjl else None  # gamma or the key scale
    tq.quantize_keys(L.params, kt, n_vec, codes, signs, norms, rn)
    vcodes = torch.zeros(n_vec, w.value_bits * E, dtype=torch.int32, device="cuda")
    vnorms = torch.zeros(n_vec, device="cuda")
    tq.quantize_values(L.params, vt, n_vec, vcodes, vnorms)
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    heads = np.arange(n_vec) % w.n_kv_heads
    stats = {}
    for h in range(w.n_kv_heads):
        sel = heads == h
        ok = O.keys(K[:n_vec][sel], h)
        g_idx = PY.unpack_flat_codes(codes.cpu().numpy().view(np.uint32)[sel], w.key_bits, w.d, w.key_split)
        g_s = PY.unpack_flat_bits(signs.cpu().numpy().view(np.uint32)[sel], w.d) if w.key_qjl == 1 else None
        g_r = rn.cpu().numpy()[sel] if w.key_qjl else None
        PY.compare_records(ok, g_idx, norms.cpu().numpy()[sel], g_s, g_r, True, stats)
        ov = O.values(V[:n_vec][sel], h)
        g_vidx = PY.unpack_flat_codes(vcodes.cpu().numpy().view(np.uint32)[sel], w.value_bits, w.d)
        PY.compare_records(ov, g_vidx, vnorms.cpu().numpy()[sel], is_key=False, stats=stats)
    assert stats["exempt"] <= max(3, PY.EXEMPT_FRACTION * stats["codes"])


def test_quantize_zero_and_tiny_vectors(tq):
    w = SK.workload("qwen", batch=1, ctx=4)
    L, O = _layer(tq, w)
    x = np.zeros((4 * w.n_kv_heads, w.d))
    x[1, 5] = 5e-8        # below the 1e-7 guard -> zero record
    x[2, :] = 1e-3        # small but regular
    x[3, 7] = 1.0         # basis vector
    xt = torch.from_numpy(x.astype(np.float32)).cuda()
    E = w.d // 32
    n = x.shape[0]
    codes = torch.zeros(n, w.key_bits * E, dtype=torch.int32, device="cuda")
    signs = torch.zeros(n, E, dtype=torch.int32, device="cuda")
    norms = torch.zeros(n, device="cuda")
    rn = torch.zeros(n, device="cuda")
    tq.quantize_keys(L.params, xt, n, codes, signs, norms, rn)
    torch.cuda.synchronize()
    heads = np.arange(n) % w.n_kv_heads
    for h in range(w.n_kv_heads):
        sel = heads == h
        ok = O.keys(x[sel], h)
        g_idx = PY.unpack_flat_codes(codes.cpu().numpy().view(np.uint32)[sel], w.key_bits, w.d)
        g_s = PY.unpack_flat_bits(signs.cpu().numpy().view(np.uint32)[sel], w.d)
        PY.compare_records(ok, g_idx, norms.cpu().numpy()[sel], g_s, rn.cpu().numpy()[sel], True, exact=True)
    zero_rows = [0, 1]
    for r in zero_rows:
        assert norms[r].item() == 0.0 and rn[r].item() == 0.0
        assert np.all(signs[r].cpu().numpy().view(np.uint32) == 0xFFFFFFFF)


@pytest.mark.parametrize("kind", [SK.FWHT, SK.DENSE])
def test_quantize_zero_and_tiny_vectors_bf16(tq, kind):
    """The same crafted rows through the d = 128 bf16 path (rows rounded to
    bf16 first, so both sides see the same inputs).  A constant row puts many
    FWHT coordinates exactly on the z = 0 boundary, where the fp64 oracle
    lands at +-1e-17: those are compared under the boundary exemption, the
    zero rows exactly."""
    w = SK.workload("bulk", ctx=4, kind=kind)
    L, O = _layer(tq, w)
    x = np.zeros((4 * w.n_kv_heads + 3, w.d))
    x[1, 5] = 5e-8
    x[2, :] = 1e-3
    x[3, 7] = 1.0
    x[4 * w.n_kv_heads + 1, :] = -2.0
    xt = SK.to_torch(x, "bf16").cuda()
    x = xt.float().cpu().numpy().astype(np.float64)
    E = w.d // 32
    n = x.shape[0]
    codes = torch.zeros(n, w.key_bits * E, dtype=torch.int32, device="cuda")
    signs = torch.zeros(n, E, dtype=torch.int32, device="cuda")
    norms = torch.zeros(n, device="cuda")
    rn = torch.zeros(n, device="cuda")
    tq.quantize_keys(L.params, xt, n, codes, signs, norms, rn)
    vcodes = torch.zeros(n, w.value_bits * E, dtype=torch.int32, device="cuda")
    vnorms = torch.zeros(n, device="cuda")
    tq.quantize_values(L.params, xt, n, vcodes, vnorms)
    torch.cuda.synchronize()
    heads = np.arange(n) % w.n_kv_heads
    stats = {}
    for h in range(w.n_kv_heads):
        sel = heads == h
        ok = O.keys(x[sel], h)
        g_idx = PY.unpack_flat_codes(codes.cpu().numpy().view(np.uint32)[sel], w.key_bits, w.d)
        g_s = PY.unpack_flat_bits(signs.cpu().numpy().view(np.uint32)[sel], w.d)
        PY.compare_records(ok, g_idx, norms.cpu().numpy()[sel], g_s, rn.cpu().numpy()[sel], True, stats)
        ov = O.values(x[sel], h)
        g_v = PY.unpack_flat_codes(vcodes.cpu().numpy().view(np.uint32)[sel], w.value_bits, w.d)
        PY.compare_records(ov, g_v, vnorms.cpu().numpy()[sel], is_key=False, stats=stats)
        zr = np.where(np.all(x[sel] == 0, axis=1) | (np.linalg.norm(x[sel], axis=1) < 1e-7))[0]
        assert np.array_equal(g_idx[zr], ok["idx"][zr]) and np.array_equal(g_v[zr], ov["idx"][zr])
    for r in (0, 1):
        assert norms[r].item() == 0.0 and rn[r].item() == 0.0 and vnorms[r].item() == 0.0
        assert np.all(signs[r].cpu().numpy().view(np.uint32) == 0xFFFFFFFF)


def _paged_roundtrip(tq, w, T0, steps, seed_layer=0):
    """Prefill T0 tokens, run `steps` decode-step appends; return everything."""
    kv = SK.keys_values(w, layer=seed_layer, ctx=T0 + steps)
    L, O = _layer(tq, w, layer=seed_layer)
    B, H, d = w.batch, w.n_kv_heads, w.d
    pc = tq.PagedCache(L, B, T0 + steps)
    kt = SK.to_torch(kv["K"], w.dtype).cuda()
    vt = SK.to_torch(kv["V"], w.dtype).cuda()
    pc.prefill(kt[:, :T0], vt[:, :T0])
    for t in range(T0, T0 + steps):
        pc.append(kt[:, t].contiguous(), vt[:, t].contiguous())
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    return kv, L, O, pc


def _oracle_cache(w, O, kv, T, nc0):
    """Oracle records per (b, head) of compressed tokens [0, n_c(T)) and the window.
    Tokens < nc0 were quantized from the input; later pages from float16."""
    nc = 16 * (max(0, T - w.window) // 16) if w.window > 0 else T
    out = []
    for b in range(w.batch):
        recs_k, recs_v = [], []
        for h in range(w.n_kv_heads):
            K = kv["K"][b, :nc, h].copy()
            V = kv["V"][b, :nc, h].copy()
            K[nc0:] = K[nc0:].astype(np.float16).astype(np.float64)
            V[nc0:] = V[nc0:].astype(np.float16).astype(np.float64)
            recs_k.append(O.keys(K, h))
            recs_v.append(O.values(V, h))
        win_k = kv["K"][b, nc:T].transpose(1, 0, 2).astype(np.float16)
        win_v = kv["V"][b, nc:T].transpose(1, 0, 2).astype(np.float16)
        out.append((recs_k, recs_v, win_k, win_v, nc))
    return out


PAGED = [
    ("qwen", dict(batch=2, window=20), 75, 40),   # window with flushes
    ("tiny", dict(), 37, 30),                      # no window: partial pages, fp32 inputs
    ("llama", dict(batch=2), 33, 18),
    ("qwen", dict(batch=1, window=128), 150, 20),
    # no window, d = 128 bf16: decode-step appends through the tensor-core warp tiles
    ("llama", dict(batch=37, kind=SK.FWHT), 29, 21),
    ("bulk", dict(batch=20, key_qjl=False, key_bits=2, value_bits=2), 15, 20),
    # head sizes that are not powers of two
    ("llama", dict(batch=5, head_dim=96), 29, 21),
    ("qwen", dict(batch=2, window=20, head_dim=160), 45, 30),
    # EDEN-unbiased and length-renormalized keys
    ("llama", dict(batch=6, kind=SK.FWHT, key_qjl=2), 29, 21),
    ("qwen", dict(batch=2, window=20, key_qjl=3), 75, 30),
    ("bulk", dict(batch=9, key_qjl=3, key_bits=3), 40, 9),
    ("tiny", dict(key_qjl=2), 37, 12),
    # the recommended key mode (3.5 bits per channel, byte norms) with a window, and variants
    ("mixed", dict(batch=2, window=20), 75, 30),
    ("llama", dict(batch=5, kind=SK.FWHT, key_bits=3, key_qjl=0, value_bits=3, key_split=1,
                   key_norm_range=(-2.0, 10.0)), 29, 21),
    ("tiny", dict(key_bits=2, key_qjl=2, key_split=1, key_norm_range=(-4.0, 12.0)), 37, 12),
    ("bulk", dict(batch=7, key_bits=1, key_qjl=3, key_split=1), 21, 12),
    # byte norms alone, with the sketch; a narrow range that clamps the outlier keys' norms
    ("llama", dict(batch=3, key_norm_range=(3.0, 5.0)), 33, 10),
    ("qwen", dict(batch=1, window=20, key_norm_range=(2.0, 6.0)), 50, 20),
    # d = 256 without a window: prefill ends in a partly filled page (64-token tiles, bitwise value planes)
    ("long", dict(batch=3), 37, 12),
    ("long", dict(batch=2, key_qjl=0, key_bits=3, value_bits=1), 70, 9),
    # d = 256 with float32 and float16 inputs (the prefill kernels' element loads, the one-vector append)
    ("long", dict(batch=2, dtype="f32"), 37, 6),
    ("qwen", dict(batch=1, window=20, dtype="f16"), 45, 20),
    # the structured sketch
    ("qwen", dict(batch=2, window=20, qjl_structured=1), 75, 30),
    ("llama", dict(batch=5, kind=SK.FWHT, qjl_structured=1), 29, 21),
    ("tiny", dict(qjl_structured=1, key_norm_range=(-4.0, 12.0)), 37, 12),
]


@pytest.mark.parametrize("name,over,T0,steps", PAGED)
def test_paged_append_and_decode_parity(tq, name, over, T0, steps):
    w = SK.workload(name, **over)
    kv, L, O, pc = _paged_roundtrip(tq, w, T0, steps)
    T = T0 + steps
    nc0 = 16 * (max(0, T0 - w.window) // 16)
    exp_nc = 16 * (max(0, T - w.window) // 16) if w.window > 0 else T
    assert pc.seq_len.cpu().tolist() == [T] * w.batch
    assert pc.n_compressed.cpu().tolist() == [exp_nc] * w.batch
    ref = _oracle_cache(w, O, kv, T, nc0 if w.window > 0 else T)
    pool = pc.pool.cpu().numpy()
    bt = pc.block_table.cpu().numpy()
    stats = {}
    q = kv["q"]
    qt = SK.to_torch(q, w.dtype).cuda()
    scale = 1.0 / math.sqrt(w.dh)
    ws = torch.empty(tq.decode_workspace_size(L.params, w.batch, T), dtype=torch.uint8, device="cuda")
    out = torch.zeros(w.batch, w.n_q_heads, w.dh, device="cuda")
    lse = torch.zeros(w.batch, w.n_q_heads, device="cuda")
    scores = torch.full((w.batch, w.n_q_heads, T), float("nan"), device="cuda")
    tq.decode_attention(L.params, pc.cache, qt, scale, out, lse, scores, ws, T)
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    for b in range(w.batch):
        recs_k, recs_v, win_k, win_v, nc = ref[b]
        npg = (nc + 15) // 16
        for h in range(w.n_kv_heads):
            pages = [PY.read_pool(pool, O, int(bt[b, p]), h) for p in range(npg)]
            cat = {k: np.concatenate([pg[k] for pg in pages])[:nc] for k in pages[0]} if npg else None
            if nc:
                PY.compare_records(recs_k[h], cat["kidx"], cat["knorm"], cat.get("ksigns"), cat.get("krnorm"),
                                   True, stats, g_norm_code=cat.get("knorm_code"))
                PY.compare_records(recs_v[h], cat["vidx"], cat["vnorm"], is_key=False, stats=stats)
                # the reference decode takes the GPU's choice where either is correct
                recs_k[h] = PY.adopt_exempt(recs_k[h], cat["kidx"], cat.get("ksigns"), cat.get("krnorm"),
                                            cat.get("knorm_code"), w.key_norm_range)
                recs_v[h] = PY.adopt_exempt(recs_v[h], cat["vidx"])
            if w.window > 0 and T - nc > 0:
                ring = pc.win_k[b, h].cpu().numpy()
                slots = [p % pc.ring for p in range(nc, T)]
                assert np.array_equal(ring[slots][:, :w.dh], win_k[h])
                assert np.array_equal(pc.win_v[b, h].cpu().numpy()[slots][:, :w.dh], win_v[h])
                assert not ring[slots][:, w.dh:].any()  # the padding of the window rows stays zero
        comp = PY.stack_comp(recs_k, recs_v) if nc else None
        r = PY.decode_reference(O, q[b], comp, win_k if T > nc else None, win_v if T > nc else None, scale)
        g_sc = scores[b].cpu().numpy()
        sc_err = np.abs(g_sc - r["scores"])
        assert np.isfinite(g_sc).all()
        assert sc_err.max() < PY.SCORE_ATOL, sc_err.max()
        assert np.abs(out[b].cpu().numpy() - r["out"]).max() < PY.OUT_ATOL
        assert np.abs(lse[b].cpu().numpy() - r["lse"]).max() < PY.SCORE_ATOL
    if stats:  # the cap holds for the codes of the whole call
        assert stats["exempt"] <= max(3, PY.EXEMPT_FRACTION * stats["codes"])


@pytest.mark.parametrize("name", ["long", "tiny"])
def test_step_append_extreme_norms(tq, name):
    """Decode-step appends without a window (one vector a CTA) at norms far from 1: a float sum of squares
    outside [1e-30, 1e37] (scales 1e-21, 1e20) takes the double sum, one inside it (1e17, 1e-6) the float
    sum; zero and sub-threshold vectors give zero records, compared exactly.  Records only: the logits of a
    1e20-scale key overflow float32."""
    scales = [1.0, 1e-21, 1e20, 1e17, 1e-6, 0.0, None]
    w = SK.workload(name, batch=len(scales), window=0)
    T0, T = 16, 20
    kv = SK.keys_values(w, ctx=T)
    K, V = kv["K"].copy(), kv["V"].copy()
    for b, sc in enumerate(scales):
        for X in (K, V):
            if sc is None:  # one coordinate, norm 5e-8: below the zero-norm guard
                X[b, T0:] = 0.0
                X[b, T0:, :, 5] = 5e-8
            else:
                X[b, T0:] *= sc
    kt = SK.to_torch(K, w.dtype).cuda()
    vt = SK.to_torch(V, w.dtype).cuda()
    K = kt.double().cpu().numpy()  # both sides see the stored dtype's values
    V = vt.double().cpu().numpy()
    L, O = _layer(tq, w)
    pc = tq.PagedCache(L, w.batch, T)
    pc.prefill(kt[:, :T0], vt[:, :T0])
    for t in range(T0, T):
        pc.append(kt[:, t].contiguous(), vt[:, t].contiguous())
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    assert pc.n_compressed.cpu().tolist() == [T] * w.batch
    pool = pc.pool.cpu().numpy()
    bt = pc.block_table.cpu().numpy()
    npg = (T + 15) // 16
    stats = {}
    for b, sc in enumerate(scales):
        zero = sc is None or sc < 1e-20
        for h in range(w.n_kv_heads):
            pages = [PY.read_pool(pool, O, int(bt[b, p]), h) for p in range(npg)]
            cat = {k: np.concatenate([pg[k] for pg in pages])[:T] for k in pages[0]}
            for lo, hi in ((0, T0), (T0, T)):
                g = {k: v[lo:hi] for k, v in cat.items()}
                exact = zero and lo == T0
                PY.compare_records(O.keys(K[b, lo:hi, h], h), g["kidx"], g["knorm"], g.get("ksigns"),
                                   g.get("krnorm"), True, None if exact else stats, exact=exact)
                PY.compare_records(O.values(V[b, lo:hi, h], h), g["vidx"], g["vnorm"], is_key=False,
                                   stats=None if exact else stats, exact=exact)
                if exact:
                    assert not g["knorm"].any() and not g["vnorm"].any()
                if sc is not None and sc > 1e10 and lo == T0:
                    assert np.isfinite(g["knorm"]).all() and g["knorm"].min() > 1e15
    assert stats["exempt"] <= max(3, PY.EXEMPT_FRACTION * stats["codes"])


def test_decode_split_invariance_and_determinism(tq):
    w = SK.workload("qwen", batch=2, window=16)
    kv, L, O, pc = _paged_roundtrip(tq, w, 300, 5)
    T = 305
    qt = SK.to_torch(kv["q"], w.dtype).cuda()
    outs = []
    for ns in (1, 3, 0, 0):
        ws = torch.empty(tq.decode_workspace_size(L.params, w.batch, T, ns), dtype=torch.uint8, device="cuda")
        out = torch.zeros(w.batch, w.n_q_heads, w.d, device="cuda")
        tq.decode_attention(L.params, pc.cache, qt, 1 / math.sqrt(w.d), out, None, None, ws, T, ns)
        outs.append(out.cpu().numpy())
    assert np.abs(outs[0] - outs[1]).max() < 1e-5
    assert np.abs(outs[0] - outs[2]).max() < 1e-5
    assert np.array_equal(outs[2], outs[3])  # same launch configuration: bit-identical


def test_empty_sequence_and_device_error(tq):
    w = SK.workload("tiny")
    L, O = _layer(tq, w)
    pc = tq.PagedCache(L, 2, 64)
    q = torch.randn(2, w.n_q_heads, w.d, device="cuda")
    ws = torch.empty(tq.decode_workspace_size(L.params, 2, 64), dtype=torch.uint8, device="cuda")
    out = torch.full((2, w.n_q_heads, w.d), 7.0, device="cuda")
    lse = torch.zeros(2, w.n_q_heads, device="cuda")
    tq.decode_attention(L.params, pc.cache, q, 0.1, out, lse, None, ws, 64)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isinf(lse))
    assert tq.check_device_error() == 0
    # a sequence longer than max_ctx is flagged on the device, not trapped
    pc.seq_len.fill_(100)
    pc.n_compressed.fill_(100)
    tq.decode_attention(L.params, pc.cache, q, 0.1, out, lse, None, ws, 64)
    bits = tq.check_device_error()
    assert bits & 0x2
    # a block-table entry outside the pool is flagged
    pc.seq_len.fill_(32)
    pc.n_compressed.fill_(32)
    pc.block_table[0, 1] = 10 ** 6
    tq.decode_attention(L.params, pc.cache, q, 0.1, out, lse, None, ws, 64)
    bits = tq.check_device_error()
    assert bits & 0x1
    assert tq.check_device_error() == 0  # cleared


@pytest.mark.parametrize("layout", ["scattered", "pages"])
@pytest.mark.parametrize("name,over", [("llama", {}), ("long", {}), ("long", dict(qjl_structured=1)),
                                       ("qwen", dict(key_qjl=2, head_dim=160))])
def test_direct_slot_append_with_skips(tq, name, over, layout):
    """Direct slots with one skipped token: scattered over pages 0..7 (at d = 256 every 16-token value
    group then takes the bitwise path), or in slot order from page 3 on (the first 16 tokens fill
    page 3 whole, the next group holds the skipped token, the last fills half of page 5)."""
    w = SK.workload(name, batch=1, ctx=40, **over)
    kv = SK.keys_values(w, ctx=40)
    L, O = _layer(tq, w)
    pc = tq.PagedCache(L, 1, 64, pool_pages=8)
    kt = SK.to_torch(kv["K"][0], w.dtype).cuda()
    vt = SK.to_torch(kv["V"][0], w.dtype).cuda()
    if layout == "scattered":  # slots across pages 0..7; token 3 skipped (-1)
        rng = np.random.default_rng(0)
        slots = rng.permutation(8 * 16)[:40].astype(np.int64)
        slots[3] = -1
    else:
        slots = 48 + np.arange(40, dtype=np.int64)
        slots[20] = -1
    st = torch.from_numpy(slots).cuda()
    tq.append_page(L.params, pc.cache, kt, vt, 40, st)
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    pool = pc.pool.cpu().numpy()
    for h in range(w.n_kv_heads):
        ok = O.keys(kv["K"][0, :, h], h)
        ov = O.values(kv["V"][0, :, h], h)
        for t, s in enumerate(slots):
            if s < 0:
                continue
            pg = PY.read_pool(pool, O, int(s // 16), h)
            sl = int(s % 16)
            sub = {k: v[t: t + 1] for k, v in ok.items() if isinstance(v, np.ndarray) and v.shape[:1] == (40,)}
            gs = pg["ksigns"][sl: sl + 1] if "ksigns" in pg else None
            gr = pg["krnorm"][sl: sl + 1] if "krnorm" in pg else None
            PY.compare_records(sub, pg["kidx"][sl: sl + 1], pg["knorm"][sl: sl + 1], gs, gr, True)
            subv = {k: v[t: t + 1] for k, v in ov.items() if isinstance(v, np.ndarray) and v.shape[:1] == (40,)}
            PY.compare_records(subv, pg["vidx"][sl: sl + 1], pg["vnorm"][sl: sl + 1], is_key=False)


def _trunc(rec, n_all, n):
    """The first n token records of an oracle record dict holding n_all tokens."""
    return {k: (v[:n] if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == n_all else v)
            for k, v in rec.items()}


PREFILL = [
    # window with flushes; the chunk straddles the compressed frontier
    ("qwen", dict(batch=2, window=20), 75, 30, 40),
    # no window: partial pages; EDEN keys; structured sketch; mixed keys with byte norms
    ("llama", dict(batch=3), 33, 18, 20),
    ("tiny", dict(key_qjl=2), 37, 12, 49),
    ("llama", dict(batch=2, kind=SK.FWHT, qjl_structured=1), 40, 9, 16),
    ("mixed", dict(batch=1, window=20), 61, 20, 33),
    # query tiles: a ragged last unit (42 rows), one query, 4-bit values with a window, several splits
    ("qwen", dict(batch=2, window=20), 75, 30, 7),
    ("qwen", dict(batch=1), 50, 3, 1),
    ("llama", dict(batch=2, window=20), 60, 25, 37),
    ("qwen", dict(batch=1, window=20), 1500, 6, 11),
    ("qwen", dict(batch=2, window=20, head_dim=160), 45, 30, 13),
]


@pytest.mark.parametrize("name,over,T0,steps,nq", PREFILL)
def test_prefill_attention_parity(tq, name, over, T0, steps, nq):
    """The last nq appended tokens attend causally to the cache: query i at position
    p = T - nq + i against the oracle's decode over positions 0..p."""
    w = SK.workload(name, **over)
    kv, L, O, pc = _paged_roundtrip(tq, w, T0, steps)
    T = T0 + steps
    nc0 = 16 * (max(0, T0 - w.window) // 16)
    ref = _oracle_cache(w, O, kv, T, nc0 if w.window > 0 else T)
    pool = pc.pool.cpu().numpy()
    bt = pc.block_table.cpu().numpy()
    rng = np.random.default_rng(1234)
    qt = SK.to_torch(rng.standard_normal((w.batch, nq, w.n_q_heads, w.dh)), w.dtype).cuda()
    q = qt.float().cpu().numpy().astype(np.float64)
    scale = 1.0 / math.sqrt(w.dh)
    ws = torch.empty(tq.prefill_workspace_size(L.params, w.batch, nq, T), dtype=torch.uint8, device="cuda")
    out = torch.zeros(w.batch, nq, w.n_q_heads, w.dh, device="cuda")
    lse = torch.zeros(w.batch, nq, w.n_q_heads, device="cuda")
    tq.prefill_attention(L.params, pc.cache, nq, qt, scale, out, lse, ws, T)
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    g_out, g_lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(w.batch):
        recs_k, recs_v, _, _, nc = ref[b]
        npg = (nc + 15) // 16
        for h in range(w.n_kv_heads):
            if nc:
                pages = [PY.read_pool(pool, O, int(bt[b, p]), h) for p in range(npg)]
                cat = {k: np.concatenate([pg[k] for pg in pages])[:nc] for k in pages[0]}
                recs_k[h] = PY.adopt_exempt(recs_k[h], cat["kidx"], cat.get("ksigns"), cat.get("krnorm"),
                                            cat.get("knorm_code"), w.key_norm_range)
                recs_v[h] = PY.adopt_exempt(recs_v[h], cat["vidx"])
        for i in range(nq):
            Ti = T - nq + i + 1
            nci = min(nc, Ti)
            comp = (PY.stack_comp([_trunc(r, nc, nci) for r in recs_k], [_trunc(r, nc, nci) for r in recs_v])
                    if nci else None)
            wk = kv["K"][b, nc:Ti].transpose(1, 0, 2).astype(np.float16) if Ti > nc else None
            wv = kv["V"][b, nc:Ti].transpose(1, 0, 2).astype(np.float16) if Ti > nc else None
            r = PY.decode_reference(O, q[b, i], comp, wk, wv, scale)
            assert np.abs(g_out[b, i] - r["out"]).max() < PY.OUT_ATOL, (b, i)
            assert np.abs(g_lse[b, i] - r["lse"]).max() < PY.SCORE_ATOL, (b, i)


def test_prefill_attention_short_sequence_is_flagged(tq):
    """A sequence shorter than the chunk is flagged on the device (TQ_DEVERR_SEQ_LEN), its
    queries see the tokens that exist, and the other sequence's result is unaffected."""
    w = SK.workload("qwen", batch=2, window=20)
    kv, L, O, pc = _paged_roundtrip(tq, w, 40, 4)
    T, nq = 44, 8
    rng = np.random.default_rng(7)
    qt = SK.to_torch(rng.standard_normal((w.batch, nq, w.n_q_heads, w.dh)), w.dtype).cuda()
    ws = torch.empty(tq.prefill_workspace_size(L.params, w.batch, nq, T), dtype=torch.uint8, device="cuda")
    out = torch.zeros(w.batch, nq, w.n_q_heads, w.dh, device="cuda")
    tq.prefill_attention(L.params, pc.cache, nq, qt, 0.0625, out, None, ws, T)
    torch.cuda.synchronize()
    assert tq.check_device_error() == 0
    ref = out.clone()
    pc.seq_len[1] = 5
    pc.n_compressed[1] = 0
    tq.prefill_attention(L.params, pc.cache, nq, qt, 0.0625, out, None, ws, T)
    bits = tq.check_device_error()
    assert bits & 0x2
    assert torch.isfinite(out).all()
    assert torch.equal(out[0], ref[0])
