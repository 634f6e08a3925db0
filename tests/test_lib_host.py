"""libtq on the host (no GPU needed): exports, host setup functions and
argument checks.

The library's codebook (Lloyd-Max with an integration-by-parts recurrence for
the cell masses) and transforms (its own SplitMix64, Box-Muller and
Householder QR) are written independently of the oracle; here they are
compared with the oracle's.
"""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import codebook as OCB
from oracle import transforms as OT

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from kv_cache_vector_head_gb300 import build

    build.build()
    from kv_cache_vector_head_gb300 import _lib

    return _lib


def test_exports_every_declared_symbol(L):
    hdr = open(os.path.join(ROOT, "include", "tq.h")).read()
    declared = set(re.findall(r"^\S[^\n(]*?\b(tq_\w+)\(", hdr, flags=re.M))
    assert {"tq_build_codebook", "tq_decode_attention", "tq_append_page"} <= declared
    lib = ctypes.CDLL(L.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(L.EXPORTED)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_matches_oracle(L, d, bits):
    c, t, mse = L.build_codebook(d, bits)
    ref = OCB.lloyd_max(d, bits)
    ulp = np.abs(c.view(np.int32) - ref.centroids.view(np.int32))
    assert ulp.max() <= 1
    np.testing.assert_allclose(c, ref.centroids, rtol=2e-7, atol=0)
    assert np.array_equal(t, ((c[:-1] + c[1:]) * np.float32(0.5)).astype(np.float32))
    assert abs(mse - ref.mse_unit) < 1e-10


@pytest.mark.parametrize("d", [32, 128, 256])
def test_transforms_match_oracle(L, d):
    for layer, head in [(0, 0), (3, 1), (31, 7)]:
        s = L.build_transform(L.TQ_FWHT, d, 0, layer, head, L.ROLE_KEY_ROT)
        assert np.array_equal(s, OT.build_transform(OT.FWHT, d, 0, layer, head, 0))
        S = L.build_transform(L.TQ_FWHT, d, 5, layer, head, L.ROLE_QJL)
        So = OT.build_transform(OT.FWHT, d, 5, layer, head, 2).ravel()
        assert np.abs(S.view(np.int32) - So.view(np.int32)).max() <= 1
        P = L.build_transform(L.TQ_DENSE, d, 0, layer, head, L.ROLE_VALUE_ROT)
        Po = OT.build_transform(OT.DENSE, d, 0, layer, head, 1).ravel()
        assert np.max(np.abs(P - Po)) <= 2e-7


def test_argument_checks_return_status_without_gpu(L):
    p = L.LayerParams()
    p.d, p.n_kv_heads, p.n_q_heads, p.page_size = 96, 2, 4, 16
    p.key_bits, p.value_bits, p.key_qjl, p.kind = 2, 2, 1, L.TQ_FWHT
    lib = L.lib()
    st = lib.tq_quantize_keys(ctypes.byref(p), None, 0, 10, None, None, None, None, None)
    assert st == L.TQ_ERR_UNSUPPORTED and b"d must be" in lib.tq_last_error()
    p.d = 128
    st = lib.tq_quantize_keys(ctypes.byref(p), None, 0, 10, None, None, None, None, None)
    assert st == L.TQ_ERR_INVALID_ARG  # null transforms
    p.page_size = 32
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0
    p.page_size = 16
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 16 * 92
    p.n_q_heads = 20
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0  # G = 10 > 8
    p.n_q_heads = 4
    p.key_bits = 5
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0
    p.key_bits = 3
    p.value_bits = 4
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 16 * 140
    # head sizes below d are zero-padded to d: a multiple of 8 in (d/2, d]
    for hd, ok in ((96, True), (80, True), (128, True), (0, True), (64, False), (70, False), (136, False)):
        p.head_dim = hd
        assert (lib.tq_subblock_bytes(ctypes.byref(p)) == 16 * 140) == ok, hd
    p.head_dim = 0
    # key corrections: scale-only records drop the sign plane (d / 8 bytes a token), 0..3 only
    p.key_qjl = L.KEY_EDEN
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 16 * (140 - 16)
    p.key_qjl = L.KEY_RENORM
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 16 * (140 - 16)
    p.key_qjl = L.KEY_MSE
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 16 * (140 - 16 - 4)
    p.key_qjl = 4
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0 and b"key_qjl" in lib.tq_last_error()
    p.key_qjl = 1
    assert lib.tq_build_codebook(2, 2, None, None, None) == L.TQ_ERR_INVALID_ARG
    assert lib.tq_build_transform(L.TQ_FWHT, 96, 0, 0, 0, 0, None) == L.TQ_ERR_INVALID_ARG
    out = np.zeros(96, np.float32)
    assert lib.tq_build_transform(L.TQ_FWHT, 96, 0, 0, 0, 0,
                                  out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))) == L.TQ_ERR_UNSUPPORTED


def test_subblock_layout_matches_oracle(L):
    from oracle import paging as PG

    for d, kb, qjl, vb in [(128, 2, 1, 2), (256, 2, 1, 2), (128, 3, 1, 4), (256, 4, 0, 1), (128, 3, 2, 4),
                           (256, 2, 3, 2)]:
        p = L.LayerParams()
        p.d, p.n_kv_heads, p.n_q_heads, p.page_size = d, 2, 4, 16
        p.key_bits, p.value_bits, p.key_qjl, p.kind = kb, vb, qjl, L.TQ_FWHT
        assert L.subblock_bytes(p) == PG.subblock_layout(d, kb, qjl, vb)["bytes"]


def test_mixed_rate_and_byte_norm_layout_and_checks(L):
    from oracle import paging as PG

    lib = L.lib()
    for d, kb, qjl, vb, split, u8 in [(128, 3, 0, 3, 1, 1), (256, 3, 2, 3, 1, 1), (128, 2, 3, 2, 1, 0),
                                      (128, 1, 0, 4, 1, 0), (256, 2, 1, 2, 0, 1), (128, 4, 0, 4, 0, 1)]:
        p = L.LayerParams()
        p.d, p.n_kv_heads, p.n_q_heads, p.page_size = d, 2, 4, 16
        p.key_bits, p.value_bits, p.key_qjl, p.kind = kb, vb, qjl, L.TQ_FWHT
        p.key_split, p.key_norm_u8, p.key_norm_log2_lo, p.key_norm_log2_hi = split, u8, -4.0, 12.0
        assert L.subblock_bytes(p) == PG.subblock_layout(d, kb, qjl, vb, key_split=split, key_norm_u8=u8)["bytes"]
    # the recommended key mode: 3.5 bits per channel + a byte norm = 57 bytes a key at d = 128
    assert PG.record_bytes(128, 3, 0, 3, key_split=1, key_norm_u8=1) == 57 + 4 + 48
    p = L.LayerParams()
    p.d, p.n_kv_heads, p.n_q_heads, p.page_size = 128, 2, 4, 16
    p.key_bits, p.value_bits, p.key_qjl, p.kind = 4, 2, 0, L.TQ_FWHT
    p.key_split = 1
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0 and b"key_bits <= 3" in lib.tq_last_error()
    p.key_bits, p.key_qjl = 3, 1
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0 and b"QJL" in lib.tq_last_error()
    p.key_qjl, p.key_split = 0, 2
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0
    p.key_split, p.key_norm_u8, p.key_norm_log2_lo, p.key_norm_log2_hi = 1, 1, 3.0, 3.0
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0 and b"key_norm_log2_lo" in lib.tq_last_error()
    p.key_norm_log2_hi = float("inf")
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0
    p.key_norm_log2_hi = 9.0
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 16 * (57 + 4 + 32)  # values 2 bits


@pytest.mark.parametrize("d", [128, 256])
def test_structured_sketch_signs_and_checks(L, d):
    for kind in (L.TQ_FWHT, L.TQ_DENSE):
        s = L.build_transform(kind, d, 7, 3, 1, L.ROLE_QJL_SIGNS)
        assert np.array_equal(s, OT.build_transform(kind, d, 7, 3, 1, OT.ROLE_QJL_SIGNS))
    p = L.LayerParams()
    p.d, p.n_kv_heads, p.n_q_heads, p.page_size = d, 2, 4, 16
    p.key_bits, p.value_bits, p.key_qjl, p.kind = 2, 2, 1, L.TQ_FWHT
    p.qjl_structured = 1
    lib = L.lib()
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 16 * (8 + 3 * d // 8 + 4 + 2 * d // 8)
    p.key_qjl = L.KEY_EDEN
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0 and b"qjl_structured" in lib.tq_last_error()
    p.key_qjl, p.qjl_structured = 1, 2
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0


def test_kivi_layout_and_checks(L):
    from oracle import kivi as OKV

    lib = L.lib()
    for d, kb, vb in [(128, 2, 2), (256, 4, 2), (128, 2, 4), (256, 4, 4)]:
        p = L.LayerParams()
        p.d, p.n_kv_heads, p.n_q_heads, p.page_size, p.window = d, 2, 4, 16, 16
        p.key_bits, p.value_bits, p.key_qjl, p.kivi = kb, vb, 0, 1
        assert L.subblock_bytes(p) == OKV.subblock_layout(d, kb, vb)["bytes"]
    p.key_bits = 3
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0 and b"kivi" in lib.tq_last_error()
    p.key_bits, p.window = 2, 0
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0 and b"window" in lib.tq_last_error()
    p.window, p.key_qjl = 16, 1
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0
    p.key_qjl, p.head_dim = 0, 96
    assert lib.tq_subblock_bytes(ctypes.byref(p)) == 0
    p.head_dim = 0
    # flat quantize does not apply to the KIVI arm (checked before any pointer)
    assert lib.tq_quantize_keys(ctypes.byref(p), None, 1, 16, None, None, None, None, None) == L.TQ_ERR_UNSUPPORTED


def test_prefill_workspace_and_checks(L):
    p = L.LayerParams()
    p.d, p.n_kv_heads, p.n_q_heads, p.page_size, p.window = 128, 2, 8, 16, 16
    p.key_bits, p.value_bits, p.key_qjl, p.kind = 2, 2, 1, L.TQ_FWHT
    lib = L.lib()
    # the prefill workspace holds a decode workspace for batch * n_query virtual sequences plus
    # three int32 counters a query, 256-byte aligned
    w = lib.tq_prefill_workspace_size(ctypes.byref(p), 3, 5, 100)
    d = lib.tq_decode_workspace_size(ctypes.byref(p), 15, 100, 0)
    assert w == d + ((3 * 15 * 4 + 255) // 256) * 256
    assert lib.tq_prefill_workspace_size(ctypes.byref(p), 3, 0, 100) == 0
    assert lib.tq_prefill_workspace_size(ctypes.byref(p), 1 << 13, 1 << 12, 100) == 0  # > 65535 queries
    # one decode launch takes at most 65535 rows (grid dimension) and 262140 (row, head) vectors
    assert lib.tq_prefill_workspace_size(ctypes.byref(p), 5, 13107, 100) > 0  # 65535 rows, G = 4
    assert lib.tq_prefill_workspace_size(ctypes.byref(p), 2, 32768, 100) == 0
    assert lib.tq_decode_workspace_size(ctypes.byref(p), 65535, 100, 0) > 0
    assert lib.tq_decode_workspace_size(ctypes.byref(p), 65536, 100, 0) == 0
    c = L.Cache()
    st = lib.tq_prefill_attention(ctypes.byref(p), ctypes.byref(c), 4, None, 1, ctypes.c_float(1.0), None, None,
                                  None, 0, 100, None)
    assert st == L.TQ_ERR_INVALID_ARG  # null transforms (checked before anything touches the GPU)


def test_norm_range_and_bit_accounting_helpers(L):
    import kv_cache_vector_head_gb300 as tq
    from oracle import codec as OC

    rng = np.random.default_rng(0)
    n = np.linalg.norm(rng.standard_normal((1000, 256)), axis=1) * np.exp(rng.standard_normal(1000))
    lo, hi = tq.norm_range_for(np.concatenate([n, [0.0]]))
    assert lo == int(lo) and hi == int(hi)
    assert 2.0 ** (lo + 1) <= n.min() and n.max() <= 2.0 ** (hi - 1)
    codes, _ = OC.norm_u8_encode(n, lo, hi)
    assert codes.min() > 1 and codes.max() < 255  # nothing clamped
    with pytest.raises(ValueError):
        tq.norm_range_for([0.0])
    # bit accounting from the library's own sub-block size (no GPU needed)
    p = L.LayerParams()
    p.d, p.n_kv_heads, p.n_q_heads, p.page_size, p.window = 256, 4, 24, 16, 128
    p.key_bits, p.value_bits, p.key_qjl, p.kind = 2, 2, 1, L.TQ_FWHT

    class _Layer:
        params, d = p, 256

    b = tq.bits_per_channel(_Layer)
    assert b["kv_total_bits_per_channel"] == 172 * 8 / 256  # 2b + QJL keys, 2b values, float norms
    assert abs(b["compression_vs_fp16"] - 32 / (172 * 8 / 256)) < 1e-12


def test_prefill_cache_checks_capacity_before_any_launch(L):
    """tq_prefill_cache applies the window rule in the library: with W = 0, 40 tokens need
    3 pages per sequence, more than a block table of 2 pages holds (refused on the host); a
    window of 16 leaves n_c = 16 (one page) and passes the check."""
    p = L.LayerParams()
    p.d, p.n_kv_heads, p.n_q_heads, p.page_size = 128, 2, 4, 16
    p.key_bits, p.value_bits, p.key_qjl, p.kind = 2, 2, 1, L.TQ_FWHT
    fake = 1 << 20  # 16-byte aligned stand-ins: nothing is launched on these paths
    p.k_rot = p.v_rot = p.qjl_s = fake
    c = L.Cache()
    c.page_pool, c.n_pages, c.block_table, c.max_pages_per_seq = fake, 8, fake, 2
    c.seq_len = c.n_compressed = fake
    c.batch = 1
    lib = L.lib()
    st = lib.tq_prefill_cache(ctypes.byref(p), ctypes.byref(c), fake, fake, L.TQ_BF16, 40, None)
    assert st == L.TQ_ERR_CAPACITY and b"max_pages_per_seq" in lib.tq_last_error()
    assert lib.tq_prefill_cache(ctypes.byref(p), ctypes.byref(c), fake, fake, L.TQ_BF16, -1, None) == L.TQ_ERR_INVALID_ARG
    p.window = 16
    st = lib.tq_prefill_cache(ctypes.byref(p), ctypes.byref(c), fake, fake, L.TQ_BF16, 40, None)
    assert st == L.TQ_ERR_INVALID_ARG and b"win_k" in lib.tq_last_error()  # window needs the ring buffers
