"""Pins of the oracle page layout and window policy.

* Bytes per (token, kv head) follow the storage formulas of
  [Reconstruction] §8 with float32 norms: 8 + (b_k + 1) d / 8 for a
  TurboQuant_prod key, 4 + b_v d / 8 for a TurboQuant_mse value.
* Pages round-trip exactly, including rewriting one slot of a page.
* The window policy: a brute-force per-token simulation (quantize the oldest
  P window tokens whenever the window reaches W + P) agrees with
  n_c(T) = P floor(max(0, T - W) / P).
"""

import numpy as np
import pytest

from oracle import codec as C
from oracle import paging as PG


@pytest.mark.parametrize("d,kb,vb,expect", [(128, 2, 2, 92), (256, 2, 2, 172), (128, 3, 4, 140)])
def test_record_bytes(d, kb, vb, expect):
    assert PG.record_bytes(d, kb, True, vb) == expect
    lay = PG.subblock_layout(d, kb, True, vb)
    assert lay["bytes"] == 16 * expect and lay["bytes"] % 16 == 0
    assert all(v % 16 == 0 for v in lay.values())


@pytest.mark.parametrize("d,kb,qjl,vb", [(128, 2, True, 2), (256, 3, True, 4), (64, 1, False, 1)])
def test_page_round_trip(d, kb, qjl, vb):
    rng = np.random.default_rng(d + kb)
    lay = PG.subblock_layout(d, kb, qjl, vb)
    H, npages = 3, 4
    pool = np.zeros(npages * H * lay["bytes"], dtype=np.uint8)
    truth = {}
    for it in range(2):  # second pass rewrites every slot
        for page in range(npages):
            for h in range(H):
                for slot in range(16):
                    rec = dict(knorm=rng.random(), krnorm=rng.random(),
                               kidx=rng.integers(0, 1 << kb, d), ks=rng.integers(0, 2, d).astype(bool),
                               vnorm=rng.random(), vidx=rng.integers(0, 1 << vb, d))
                    truth[(page, h, slot)] = rec
                    PG.write_page(pool, lay, H, page, h, slot, d, kb, qjl, vb,
                                  rec["knorm"], rec["krnorm"], C.pack_codes(rec["kidx"][None], kb)[0],
                                  C.pack_bits(rec["ks"][None].astype(np.uint8))[0], rec["vnorm"],
                                  C.code_planes(rec["vidx"][None], vb)[0])
    for page in range(npages):
        for h in range(H):
            got = PG.read_page(pool, lay, H, page, h, d, kb, qjl, vb)
            for slot in range(16):
                rec = truth[(page, h, slot)]
                assert got["knorm"][slot] == np.float32(rec["knorm"])
                assert np.array_equal(got["kidx"][slot], rec["kidx"])
                assert np.array_equal(got["vidx"][slot], rec["vidx"])
                assert got["vnorm"][slot] == np.float32(rec["vnorm"])
                if qjl:
                    assert got["krnorm"][slot] == np.float32(rec["krnorm"])
                    assert np.array_equal(got["ksigns"][slot], rec["ks"])


@pytest.mark.parametrize("W", [0, 5, 16, 128])
def test_window_policy_brute_force(W):
    P = 16
    window = []          # positions held in fp16
    compressed = 0
    for T in range(0, 700):
        assert compressed == PG.n_compressed(T, W)
        assert len(window) == T - compressed
        if T >= W:
            assert W <= len(window) < W + P
        slots = {PG.ring_slot(p, W) for p in window}
        assert len(slots) == len(window)  # ring never overwrites a live token
        nc1, flushed = PG.decode_append_step(T, W)
        window.append(T)
        if len(window) == W + P:
            window = window[P:]
            compressed += P
            assert flushed
        else:
            assert not flushed
        assert nc1 == compressed


@pytest.mark.parametrize("d,kb,qjl,vb", [(128, 3, 1, 4), (256, 2, 1, 2), (128, 2, 2, 3)])
def test_batched_page_reader_equals_read_page(d, kb, qjl, vb):
    """tests/parity.read_pages (every page of a sequence at once) decodes the same records as
    read_page page by page."""
    import parity as PY

    rng = np.random.default_rng(3)
    H, n_pages = 2, 5
    O = PY.OracleLayer(d, H, H, kb, vb, 1, qjl=qjl)
    lay = PG.subblock_layout(d, kb, qjl, vb)
    pool = rng.integers(0, 256, size=n_pages * H * lay["bytes"], dtype=np.uint8)
    pages = [3, 0, 4]
    for h in range(H):
        got = PY.read_pages(pool, O, pages, h)
        for i, pg in enumerate(pages):
            ref = PG.read_page(pool, lay, H, pg, h, d, kb, qjl, vb)
            sl = slice(16 * i, 16 * i + 16)
            assert np.array_equal(got["kidx"][sl], ref["kidx"]) and np.array_equal(got["vidx"][sl], ref["vidx"])
            assert np.array_equal(got["knorm"][sl].view(np.uint32), ref["knorm"].view(np.uint32))
            assert np.array_equal(got["vnorm"][sl].view(np.uint32), ref["vnorm"].view(np.uint32))
            if qjl:
                assert np.array_equal(got["krnorm"][sl].view(np.uint32), ref["krnorm"].view(np.uint32))
            if qjl == 1:
                assert np.array_equal(got["ksigns"][sl], ref["ksigns"])
