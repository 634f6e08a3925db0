"""A bounded device wait that runs out is reported, and the context stays usable.

The decode kernels wait on TMA page copies with bounded mbarrier polls; when a
wait runs out the split stops issuing copies, waits (bounded) for the copies
still in flight and sets TQ_DEVERR_TIMEOUT in the device error word, which
tq_check_device_error returns.  To reach that branch without faulting the GPU,
this test uses libtq_testhooks.so, the same sources built with TQ_TEST_HOOKS:
a short wait limit (~16 ms) and tq_test_wait_fault(1), under which the first
chunk of every page split expects 16 bytes more than its copies deliver.  The
copies land, the barrier phase never completes, the wait runs out.  The test
checks that the call returns promptly with the timeout bit, then that the same
library decodes correctly again after tq_test_wait_fault(0).
"""

import ctypes
import math
import time

import numpy as np
import pytest

import synthetic_kv as SK

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_wait_that_runs_out_is_reported_and_the_context_survives():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from kv_cache_vector_head_gb300 import build

    build.build()
    hooks_path = build.build_test_hooks()
    import kv_cache_vector_head_gb300 as tq
    from kv_cache_vector_head_gb300 import _lib as L

    H = ctypes.CDLL(hooks_path)
    H.tq_test_wait_fault.argtypes = [ctypes.c_int]
    H.tq_test_wait_fault.restype = ctypes.c_int
    H.tq_decode_attention.argtypes = L.lib().tq_decode_attention.argtypes
    H.tq_decode_attention.restype = ctypes.c_int
    H.tq_check_device_error.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    H.tq_check_device_error.restype = ctypes.c_int

    w = SK.workload("tiny", batch=2, ctx=640)
    B, T = w.batch, w.ctx
    layer = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=0)
    pc = tq.PagedCache(layer, B, T)
    K, V, q = SK.keys_values_torch(w, ctx=T)
    pc.prefill(K, V)
    ws = torch.empty(tq.decode_workspace_size(layer.params, B, T), dtype=torch.uint8, device="cuda")
    ref = torch.zeros(B, w.n_q_heads, w.d, device="cuda")
    scale = 1.0 / math.sqrt(w.d)
    tq.decode_attention(layer.params, pc.cache, q, scale, ref, None, None, ws, T)
    assert tq.check_device_error() == 0
    stream = torch.cuda.current_stream().cuda_stream

    def hooked_decode(out):
        return H.tq_decode_attention(ctypes.byref(layer.params), ctypes.byref(pc.cache), q.data_ptr(), L.dtype_code(q),
                                     scale, out.data_ptr(), None, None, ws.data_ptr(), ws.numel(), T, 0, stream)

    bits = ctypes.c_uint32(0)
    assert H.tq_test_wait_fault(1) == L.TQ_OK
    out = torch.zeros_like(ref)
    t0 = time.monotonic()
    assert hooked_decode(out) == L.TQ_OK
    st = H.tq_check_device_error(stream, ctypes.byref(bits))
    elapsed = time.monotonic() - t0
    assert st == L.TQ_ERR_DEVICE_CHECK and bits.value & 0x8, (st, bits.value)  # TQ_DEVERR_TIMEOUT
    assert elapsed < 30.0, elapsed

    assert H.tq_test_wait_fault(0) == L.TQ_OK
    out.zero_()
    assert hooked_decode(out) == L.TQ_OK
    bits.value = 0
    assert H.tq_check_device_error(stream, ctypes.byref(bits)) == L.TQ_OK and bits.value == 0
    np.testing.assert_array_equal(out.cpu().numpy(), ref.cpu().numpy())
