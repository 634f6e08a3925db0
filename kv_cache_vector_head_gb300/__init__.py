"""TurboQuant KV-cache hot path for NVIDIA GB300 (sm_103a).

Python side of the C ABI in ``include/tq.h``: ``_lib`` marshals arguments to
libtq.so; the classes below only allocate device memory (PyTorch) and fill
the ctypes structures.  Every step of quantization, paging and decode runs in
libtq's CUDA kernels; if libtq.so is missing, importing the binding's functions
raises.
"""

from __future__ import annotations

import math

import numpy as np

from . import _lib
from ._lib import (KEY_EDEN, KEY_MSE, KEY_QJL, KEY_RENORM, PAGE_SIZE, ROLE_KEY_ROT, ROLE_QJL, ROLE_QJL_SIGNS, ROLE_VALUE_ROT, TQ_BF16, TQ_DENSE, TQ_F16, TQ_F32, TQ_FWHT,
                   Cache, LayerParams, TQError, append_page, build_codebook, build_transform, check_device_error,
                   decode_attention, decode_workspace_size, prefill_attention, prefill_cache, prefill_workspace_size,
                   quantize_keys, quantize_values, subblock_bytes)

__all__ = [
    "TQLayer", "PagedCache", "LayerParams", "Cache", "TQError", "build_codebook", "build_transform",
    "quantize_keys", "quantize_values", "append_page", "decode_workspace_size", "decode_attention",
    "prefill_workspace_size", "prefill_attention", "prefill_cache", "norm_range_for", "bits_per_channel",
    "check_device_error", "subblock_bytes", "TQ_DENSE", "TQ_FWHT", "TQ_F32", "TQ_BF16", "TQ_F16", "PAGE_SIZE",
    "ROLE_KEY_ROT", "ROLE_VALUE_ROT", "ROLE_QJL", "ROLE_QJL_SIGNS", "KEY_MSE", "KEY_QJL", "KEY_EDEN", "KEY_RENORM",
]


def norm_range_for(norms, margin: float = 1.0) -> tuple[float, float]:
    """A byte-norm range (log2 lo, hi) covering sample key norms with `margin` octaves on each
    side: the per-layer calibration the u8 log-norm takes ([Design study] §Packed format).
    Zero norms are ignored; integer bounds keep the code grid reproducible."""
    n = np.asarray(norms, dtype=np.float64).ravel()
    n = n[n > 1e-7]
    if n.size == 0:
        raise ValueError("no nonzero norms to calibrate from")
    lo = math.floor(math.log2(n.min()) - margin)
    hi = math.ceil(math.log2(n.max()) + margin)
    return float(lo), float(max(hi, lo + 1))


def bits_per_channel(layer: "TQLayer") -> dict:
    """Bits per channel of the layer's compressed records ([Design study] §Packed format and
    complete bit accounting): the 16-token sub-block bytes of a (page, kv head) over
    16 tokens x d channels, for keys and values together, next to the float16 cache's 16."""
    total = subblock_bytes(layer.params) * 8 / (PAGE_SIZE * layer.d)
    return {"kv_bits_per_channel": total / 2, "kv_total_bits_per_channel": total,
            "compression_vs_fp16": 32.0 / total}


class TQLayer:
    """Codebooks, per-head transforms (device) and the tq_layer_params of one layer."""

    def __init__(self, d: int, n_kv_heads: int, n_q_heads: int, key_bits: int, value_bits: int, kind: int,
                 window: int = 0, key_qjl: int = KEY_QJL, seed: int = 0, layer: int = 0, device="cuda",
                 head_dim: int | None = None, key_split: bool = False,
                 key_norm_range: tuple[float, float] | None = None, qjl_structured: bool = False,
                 kivi: bool = False):
        """d: the transform and code dimension (128 or 256); head_dim (default d):
        the length of the vectors the caller passes, zero-padded to d inside
        the kernels (a multiple of 8 in (d/2, d]).  key_qjl: the key
        correction, KEY_QJL (TurboQuant_prod, default), KEY_MSE (code only),
        KEY_EDEN (unbiased scale) or KEY_RENORM (TurboVec's length-renormalized
        correction norm / <y, y_hat>, stored as the same scale as KEY_EDEN);
        True / False stand for KEY_QJL / KEY_MSE.  key_split: mixed-channel
        key rate, rotated coordinates < d/2 at key_bits + 1 bits (key_bits = 3
        gives 3.5 bits per channel; not with KEY_QJL).  key_norm_range =
        (lo, hi): key norms stored as one byte, log2-uniform over [2^lo, 2^hi].
        qjl_structured (with KEY_QJL): the sketch matrix is S = H diag(sigma_S),
        applied as a fast Walsh-Hadamard transform, instead of a dense Gaussian.
        kivi: the KIVI-like control arm (asymmetric min-max codes of key_bits /
        value_bits = 2 or 4 bits, keys per channel over a page, values per
        token; no rotation; key_qjl must be KEY_MSE and window >= 1)."""
        import torch

        self.d, self.n_kv_heads, self.n_q_heads = d, n_kv_heads, n_q_heads
        self.head_dim = d if head_dim is None else head_dim
        self.key_bits, self.value_bits, self.kind, self.window = key_bits, value_bits, kind, window
        self.key_qjl, self.seed, self.layer = int(key_qjl), seed, layer
        if self.key_qjl not in (KEY_MSE, KEY_QJL, KEY_EDEN, KEY_RENORM):
            raise ValueError(f"key_qjl must be one of KEY_MSE, KEY_QJL, KEY_EDEN, KEY_RENORM, got {key_qjl}")
        self.key_split, self.key_norm_range = bool(key_split), key_norm_range
        self.kivi = bool(kivi)
        self.k_cb = build_codebook(d, key_bits)
        self.k_cb_hi = build_codebook(d, key_bits + 1) if key_split else None
        self.v_cb = build_codebook(d, value_bits)
        if self.kivi:  # no transforms
            self.k_rot_host = self.v_rot_host = self.k_rot = self.v_rot = None
        else:
            kr = np.stack([build_transform(kind, d, seed, layer, h, ROLE_KEY_ROT) for h in range(n_kv_heads)])
            vr = np.stack([build_transform(kind, d, seed, layer, h, ROLE_VALUE_ROT) for h in range(n_kv_heads)])
            self.k_rot_host, self.v_rot_host = kr, vr
            self.k_rot = torch.from_numpy(kr).to(device)
            self.v_rot = torch.from_numpy(vr).to(device)
        self.qjl_structured = bool(qjl_structured)
        if self.key_qjl == KEY_QJL:
            role = ROLE_QJL_SIGNS if qjl_structured else ROLE_QJL
            s = np.stack([build_transform(kind, d, seed, layer, h, role) for h in range(n_kv_heads)])
            self.qjl_s_host = s
            self.qjl_s = torch.from_numpy(s).to(device)
        else:
            self.qjl_s_host, self.qjl_s = None, None
        p = LayerParams()
        p.d, p.n_kv_heads, p.n_q_heads, p.page_size, p.window = d, n_kv_heads, n_q_heads, PAGE_SIZE, window
        p.key_bits, p.key_qjl, p.value_bits, p.kind = key_bits, self.key_qjl, value_bits, kind
        p.head_dim = self.head_dim
        p.k_rot = self.k_rot.data_ptr() if self.k_rot is not None else None
        p.v_rot = self.v_rot.data_ptr() if self.v_rot is not None else None
        p.kivi = int(self.kivi)
        p.qjl_s = self.qjl_s.data_ptr() if self.qjl_s is not None else None
        for name, (c, t, _) in (("k", self.k_cb), ("v", self.v_cb)):
            getattr(p, f"{name}_centroids")[: len(c)] = [float(x) for x in c]
            getattr(p, f"{name}_bounds")[: len(t)] = [float(x) for x in t]
        if key_split:
            c, t, _ = self.k_cb_hi
            p.key_split = 1
            p.k_hi_centroids[: len(c)] = [float(x) for x in c]
            p.k_hi_bounds[: len(t)] = [float(x) for x in t]
        p.qjl_structured = int(self.qjl_structured)
        if key_norm_range is not None:
            p.key_norm_u8 = 1
            p.key_norm_log2_lo, p.key_norm_log2_hi = float(key_norm_range[0]), float(key_norm_range[1])
        self.params = p
        self.sub_bytes = subblock_bytes(p)


class PagedCache:
    """Device buffers of one layer's paged cache and its tq_cache descriptor.

    Pages are handed out contiguously: sequence b owns pages
    [b * max_pages_per_seq, (b + 1) * max_pages_per_seq).
    """

    def __init__(self, layer: TQLayer, batch: int, max_ctx: int, device="cuda", pool_pages: int | None = None):
        import torch

        self.layer, self.batch = layer, batch
        self.max_pages = max(1, math.ceil(max_ctx / PAGE_SIZE))
        n_pages = pool_pages if pool_pages is not None else batch * self.max_pages
        self.pool = torch.zeros(n_pages * layer.n_kv_heads * layer.sub_bytes, dtype=torch.uint8, device=device)
        bt = torch.arange(batch * self.max_pages, dtype=torch.int32, device=device).reshape(batch, self.max_pages)
        self.block_table = bt % n_pages
        self.seq_len = torch.zeros(batch, dtype=torch.int32, device=device)
        self.n_compressed = torch.zeros(batch, dtype=torch.int32, device=device)
        self.ring = layer.window + PAGE_SIZE if layer.window > 0 else 0
        if self.ring:
            shape = (batch, layer.n_kv_heads, self.ring, layer.d)
            self.win_k = torch.zeros(shape, dtype=torch.float16, device=device)
            self.win_v = torch.zeros(shape, dtype=torch.float16, device=device)
        else:
            self.win_k = self.win_v = None
        c = Cache()
        c.page_pool, c.n_pages = self.pool.data_ptr(), n_pages
        c.block_table, c.max_pages_per_seq = self.block_table.data_ptr(), self.max_pages
        c.seq_len, c.n_compressed = self.seq_len.data_ptr(), self.n_compressed.data_ptr()
        c.win_k = self.win_k.data_ptr() if self.win_k is not None else None
        c.win_v = self.win_v.data_ptr() if self.win_v is not None else None
        c.batch = batch
        self.cache = c
        self.n_pages = n_pages

    def slot_mapping(self, T: int):
        """Pool slots (page * 16 + slot) of token positions 0..T-1 of every sequence, [batch * T]."""
        import torch

        pos = torch.arange(T, device=self.block_table.device)
        pages = self.block_table[:, pos // PAGE_SIZE].to(torch.int64)
        return (pages * PAGE_SIZE + (pos % PAGE_SIZE)[None, :]).reshape(-1)

    def prefill(self, k, v, stream=None) -> None:
        """Fill every sequence with T tokens: k, v [batch, T, Hkv, head_dim].  The library
        (tq_prefill_cache) applies the window rule: the oldest whole pages are quantized
        straight into their pages, the last W .. W + 15 tokens go to the float16 window, and
        the counters are set, as live decoding would leave them."""
        prefill_cache(self.layer.params, self.cache, k.contiguous(), v.contiguous(), k.shape[1], stream)

    def append(self, k, v, stream=None) -> None:
        """One decode step: k, v [batch, Hkv, d]."""
        append_page(self.layer.params, self.cache, k, v, self.batch, None, stream)
