"""ctypes binding of libtq (include/tq.h): argument marshalling only.

Every computation of the hot path runs in libtq's CUDA kernels.  If the shared
library is missing this module raises; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_double, c_float, c_int, c_int64, c_size_t, c_uint32, c_uint64, c_void_p

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtq.so")

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_NO_CONVERGENCE, TQ_ERR_CAPACITY, \
    TQ_ERR_DEVICE_CHECK = range(7)
TQ_DENSE, TQ_FWHT = 0, 1
TQ_F32, TQ_BF16, TQ_F16 = 0, 1, 2
ROLE_KEY_ROT, ROLE_VALUE_ROT, ROLE_QJL, ROLE_QJL_SIGNS = 0, 1, 2, 3
KEY_MSE, KEY_QJL, KEY_EDEN, KEY_RENORM = 0, 1, 2, 3  # tq_key_correction
PAGE_SIZE = 16

EXPORTED = [
    "tq_build_codebook", "tq_build_transform", "tq_quantize_keys", "tq_quantize_values", "tq_subblock_bytes",
    "tq_append_page", "tq_decode_workspace_size", "tq_decode_attention", "tq_check_device_error", "tq_last_error",
    "tq_decode_attention_static", "tq_prefill_workspace_size", "tq_prefill_attention", "tq_prefill_cache",
]
STATIC_SCRATCH_BYTES = 16 << 20


class TQError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"tq status {status}: {msg}")
        self.status = status


class LayerParams(ctypes.Structure):
    _fields_ = [
        ("d", c_int), ("n_kv_heads", c_int), ("n_q_heads", c_int), ("page_size", c_int), ("window", c_int),
        ("key_bits", c_int), ("key_qjl", c_int), ("value_bits", c_int), ("kind", c_int),
        ("k_rot", c_void_p), ("v_rot", c_void_p), ("qjl_s", c_void_p),
        ("k_centroids", c_float * 16), ("k_bounds", c_float * 16),
        ("v_centroids", c_float * 16), ("v_bounds", c_float * 16),
        ("head_dim", c_int),
        ("key_split", c_int), ("k_hi_centroids", c_float * 16), ("k_hi_bounds", c_float * 16),
        ("key_norm_u8", c_int), ("key_norm_log2_lo", c_float), ("key_norm_log2_hi", c_float),
        ("qjl_structured", c_int), ("kivi", c_int),
    ]


class Cache(ctypes.Structure):
    _fields_ = [
        ("page_pool", c_void_p), ("n_pages", c_int64), ("block_table", c_void_p), ("max_pages_per_seq", c_int),
        ("seq_len", c_void_p), ("n_compressed", c_void_p), ("win_k", c_void_p), ("win_v", c_void_p),
        ("batch", c_int),
    ]


_lib = None


def lib():
    """Load libtq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtq.so not built at {LIB_PATH}; run kv_cache_vector_head_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.tq_build_codebook.argtypes = [c_int, c_int, POINTER(c_float), POINTER(c_float), POINTER(c_double)]
        L.tq_build_transform.argtypes = [c_int, c_int, c_uint64, c_int, c_int, c_int, POINTER(c_float)]
        L.tq_quantize_keys.argtypes = [POINTER(LayerParams), c_void_p, c_int, c_int64, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p]
        L.tq_quantize_values.argtypes = [POINTER(LayerParams), c_void_p, c_int, c_int64, c_void_p, c_void_p, c_void_p]
        L.tq_subblock_bytes.argtypes = [POINTER(LayerParams)]
        L.tq_subblock_bytes.restype = c_size_t
        L.tq_append_page.argtypes = [POINTER(LayerParams), POINTER(Cache), c_void_p, c_void_p, c_int, c_int64,
                                     c_void_p, c_void_p]
        L.tq_prefill_cache.argtypes = [POINTER(LayerParams), POINTER(Cache), c_void_p, c_void_p, c_int, c_int, c_void_p]
        L.tq_decode_workspace_size.argtypes = [POINTER(LayerParams), c_int, c_int, c_int]
        L.tq_decode_workspace_size.restype = c_size_t
        L.tq_decode_attention.argtypes = [POINTER(LayerParams), POINTER(Cache), c_void_p, c_int, c_float, c_void_p,
                                          c_void_p, c_void_p, c_void_p, c_size_t, c_int, c_int, c_void_p]
        L.tq_decode_attention_static.argtypes = [POINTER(LayerParams), POINTER(Cache), c_void_p, c_int, c_float,
                                                 c_void_p, c_void_p, c_void_p, c_int, c_int, c_void_p]
        L.tq_prefill_workspace_size.argtypes = [POINTER(LayerParams), c_int, c_int, c_int]
        L.tq_prefill_workspace_size.restype = c_size_t
        L.tq_prefill_attention.argtypes = [POINTER(LayerParams), POINTER(Cache), c_int, c_void_p, c_int, c_float,
                                           c_void_p, c_void_p, c_void_p, c_size_t, c_int, c_void_p]
        L.tq_check_device_error.argtypes = [c_void_p, POINTER(c_uint32)]
        L.tq_last_error.restype = ctypes.c_char_p
        for name in EXPORTED:
            if name not in ("tq_subblock_bytes", "tq_decode_workspace_size", "tq_prefill_workspace_size",
                            "tq_last_error"):
                getattr(L, name).restype = c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != TQ_OK:
        raise TQError(status, lib().tq_last_error().decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def dtype_code(t) -> int:
    import torch

    return {torch.float32: TQ_F32, torch.bfloat16: TQ_BF16, torch.float16: TQ_F16}[t.dtype]


# ---------------------------------------------------------------------------- host setup

def build_codebook(d: int, bits: int):
    c = np.zeros(1 << bits, dtype=np.float32)
    t = np.zeros(max(1, (1 << bits) - 1), dtype=np.float32)
    mse = c_double(0.0)
    _check(lib().tq_build_codebook(d, bits, c.ctypes.data_as(POINTER(c_float)), t.ctypes.data_as(POINTER(c_float)),
                                   ctypes.byref(mse)))
    return c, t, mse.value


def build_transform(kind: int, d: int, seed: int, layer: int, head: int, role: int) -> np.ndarray:
    n = d if ((kind == TQ_FWHT and role != ROLE_QJL) or role == ROLE_QJL_SIGNS) else d * d
    out = np.zeros(n, dtype=np.float32)
    _check(lib().tq_build_transform(kind, d, seed, layer, head, role, out.ctypes.data_as(POINTER(c_float))))
    return out


def subblock_bytes(p: LayerParams) -> int:
    n = lib().tq_subblock_bytes(ctypes.byref(p))
    if n == 0:
        _check(TQ_ERR_INVALID_ARG)
    return n


# ---------------------------------------------------------------------------- hot path

def quantize_keys(p: LayerParams, k, n_vec: int, codes, signs, norms, rnorms, stream=None) -> None:
    _check(lib().tq_quantize_keys(ctypes.byref(p), _ptr(k), dtype_code(k), n_vec, _ptr(codes), _ptr(signs),
                                  _ptr(norms), _ptr(rnorms), _stream(stream)))


def quantize_values(p: LayerParams, v, n_vec: int, codes, norms, stream=None) -> None:
    _check(lib().tq_quantize_values(ctypes.byref(p), _ptr(v), dtype_code(v), n_vec, _ptr(codes), _ptr(norms),
                                    _stream(stream)))


def append_page(p: LayerParams, cache: Cache, k, v, n_tok: int, slot_mapping=None, stream=None) -> None:
    _check(lib().tq_append_page(ctypes.byref(p), ctypes.byref(cache), _ptr(k), _ptr(v), dtype_code(k), n_tok,
                                _ptr(slot_mapping), _stream(stream)))


def prefill_cache(p: LayerParams, cache: Cache, k, v, n_tok: int, stream=None) -> None:
    """Every sequence gets its first n_tok tokens (k, v [batch, n_tok, Hkv, head_dim]); the
    library splits them into pages and the float16 window and sets the counters."""
    _check(lib().tq_prefill_cache(ctypes.byref(p), ctypes.byref(cache), _ptr(k), _ptr(v), dtype_code(k), n_tok,
                                  _stream(stream)))


def decode_workspace_size(p: LayerParams, batch: int, max_ctx: int, n_splits: int = 0) -> int:
    n = lib().tq_decode_workspace_size(ctypes.byref(p), batch, max_ctx, n_splits)
    if n == 0:
        _check(TQ_ERR_INVALID_ARG)
    return n


def decode_attention(p: LayerParams, cache: Cache, q, scale: float, out, lse, scores, workspace, max_ctx: int,
                     n_splits: int = 0, stream=None) -> None:
    _check(lib().tq_decode_attention(ctypes.byref(p), ctypes.byref(cache), _ptr(q), dtype_code(q), scale, _ptr(out),
                                     _ptr(lse), _ptr(scores), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     max_ctx, n_splits, _stream(stream)))


def decode_attention_static(p: LayerParams, cache: Cache, q, scale: float, out, lse, scores, max_ctx: int,
                            n_splits: int = 0, stream=None) -> None:
    """tq_decode_attention with the library's own static scratch (no workspace)."""
    _check(lib().tq_decode_attention_static(ctypes.byref(p), ctypes.byref(cache), _ptr(q), dtype_code(q), scale,
                                            _ptr(out), _ptr(lse), _ptr(scores), max_ctx, n_splits, _stream(stream)))


def prefill_workspace_size(p: LayerParams, batch: int, n_query: int, max_ctx: int) -> int:
    n = lib().tq_prefill_workspace_size(ctypes.byref(p), batch, n_query, max_ctx)
    if n == 0:
        _check(TQ_ERR_INVALID_ARG)
    return n


def prefill_attention(p: LayerParams, cache: Cache, n_query: int, q, scale: float, out, lse, workspace, max_ctx: int,
                      stream=None) -> None:
    """The last n_query appended tokens of every sequence attend causally to the cache:
    q, out [batch, n_query, Hq, head_dim], lse [batch, n_query, Hq] (or None)."""
    _check(lib().tq_prefill_attention(ctypes.byref(p), ctypes.byref(cache), n_query, _ptr(q), dtype_code(q), scale,
                                      _ptr(out), _ptr(lse), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), max_ctx, _stream(stream)))


def check_device_error(stream=None) -> int:
    bits = c_uint32(0)
    st = lib().tq_check_device_error(_stream(stream), ctypes.byref(bits))
    if st not in (TQ_OK, TQ_ERR_DEVICE_CHECK):
        _check(st)
    return bits.value
