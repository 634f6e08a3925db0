"""The no-allocation decode entry point, tq_decode_attention_static.

Some callers cannot allocate device memory when they decode (a runtime whose
device memory is planned up front, or code where a cudaMalloc would stall or is
forbidden).  For them the library keeps a fixed scratch array of its own.  This
test calls that entry point through the C ABI and checks that two calls in a
row give the same results as tq_decode_attention with a caller workspace,
within the tolerances of the other parity tests, and that a configuration too
large for the array is refused.  It sits in a file that pytest collects last.
"""

import ctypes
import math

import numpy as np
import pytest

import synthetic_kv as SK

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

OUT_ATOL = 2e-3
SCORE_ATOL = 1e-3


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from kv_cache_vector_head_gb300 import build

    build.build()
    import kv_cache_vector_head_gb300 as tq

    return tq


def test_static_scratch_matches_workspace_entry_point(tq):
    w = SK.workload("qwen", batch=2, window=16)
    T0, T = 300, 305
    kv = SK.keys_values(w, ctx=T)
    L = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=w.window)
    pc = tq.PagedCache(L, w.batch, T)
    kt = SK.to_torch(kv["K"], w.dtype).cuda()
    vt = SK.to_torch(kv["V"], w.dtype).cuda()
    pc.prefill(kt[:, :T0], vt[:, :T0])
    lib = tq._lib.lib()
    scale = 1.0 / math.sqrt(w.d)
    for call in range(2):  # two calls in a row, the cache growing in between
        t = T0 + call
        pc.append(kt[:, t].contiguous(), vt[:, t].contiguous())
        q = torch.randn(w.batch, w.n_q_heads, w.d, device="cuda", dtype=torch.bfloat16)
        ws = torch.empty(tq.decode_workspace_size(L.params, w.batch, T), dtype=torch.uint8, device="cuda")
        ref_out = torch.zeros(w.batch, w.n_q_heads, w.d, device="cuda")
        ref_lse = torch.zeros(w.batch, w.n_q_heads, device="cuda")
        ref_sc = torch.zeros(w.batch, w.n_q_heads, T, device="cuda")
        tq.decode_attention(L.params, pc.cache, q, scale, ref_out, ref_lse, ref_sc, ws, T)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        sc = torch.zeros_like(ref_sc)
        st = lib.tq_decode_attention_static(ctypes.byref(L.params), ctypes.byref(pc.cache), q.data_ptr(),
                                            tq._lib.TQ_BF16, scale, out.data_ptr(), lse.data_ptr(), sc.data_ptr(),
                                            T, 0, torch.cuda.current_stream().cuda_stream)
        assert st == 0, lib.tq_last_error()
        torch.cuda.synchronize()
        assert tq.check_device_error() == 0
        assert torch.isfinite(out).all()
        assert (out - ref_out).abs().max().item() < OUT_ATOL
        assert (lse - ref_lse).abs().max().item() < SCORE_ATOL
        n = t + 1
        assert (sc[:, :, :n] - ref_sc[:, :, :n]).abs().max().item() < SCORE_ATOL


def test_static_scratch_refuses_oversized_configuration(tq):
    w = SK.workload("qwen", batch=1)
    L = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=w.window)
    pc = tq.PagedCache(L, 1, 64)
    lib = tq._lib.lib()
    huge = 1 << 26  # needs far more scratch than the static array holds
    assert tq.decode_workspace_size(L.params, 1, huge, 4096) > tq._lib.STATIC_SCRATCH_BYTES
    out = torch.zeros(1, w.n_q_heads, w.d, device="cuda")
    q = torch.zeros(1, w.n_q_heads, w.d, device="cuda", dtype=torch.bfloat16)
    st = lib.tq_decode_attention_static(ctypes.byref(L.params), ctypes.byref(pc.cache), q.data_ptr(),
                                        tq._lib.TQ_BF16, 0.0625, out.data_ptr(), None, None, huge, 4096,
                                        torch.cuda.current_stream().cuda_stream)
    assert st == tq._lib.TQ_ERR_CAPACITY
    assert b"static array" in lib.tq_last_error()
