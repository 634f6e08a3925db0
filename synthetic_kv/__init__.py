"""Seeded synthetic K, V and q inputs for the TurboQuant KV-cache hot path.

This module only draws inputs.  It holds none of the method's arithmetic and
is the one piece that both the oracle-side tests and the GPU side consume.
The pages measure on trained models and needle tests, which are not
available here; these synthetic tensors stand in for them, with the shapes of
the workloads below.

Generator: SplitMix64 over counters (one stream per (tensor, layer, sequence)),
uniform (x >> 11) * 2^-53, Box-Muller normals; this module's own copy.

Workloads:
  tiny      1 seq, 1 layer, 2 KV / 4 q heads, d = 128, T = 1024; K, V, q fp32
            N(0,1); keys times exp(g_c), g_c ~ N(0,1) per (head, channel),
            before RoPE; RoPE theta = 1e4 (rotate-half pairs (j, j + d/2)) at
            positions 0..T-1 and q at position T; keys 2b MSE + QJL, values 2b,
            dense rotation, seed 0, no window.
  qwen      bf16 N(0,1) K, V, q; d = 256, 4 KV / 24 q heads, batch 8,
            T = 32768, keys 2b + QJL, values 2b, FWHT rotation, page 16,
            fp16 window 128.
  llama     bf16, d = 128, 8 KV / 32 q heads, batch 32, T = 8192, 32 layers;
            keys 3b + QJL, values 4b; K ~ N(0,1) with 4 outlier channels x20
            (drawn without replacement per (layer, head)) applied after RoPE;
            V, q ~ N(0,1); paged, page 16, dense rotation, no window.
  long      bf16 N(0,1), d = 256, 2 KV / 16 q heads, batch 1, T = 131072;
            keys 2b + QJL, values 2b, FWHT, no window.
  bulk      65536 tokens x 32 layers x 8 KV heads, d = 128, bf16 N(0,1) K and V
            times lognormal(sigma = 1) per (layer, head, channel) scales;
            keys 3b + QJL, values 4b; dense and FWHT.
  mixed     the qwen shape in the recommended first product mode of the
            design study: keys 3.5 bits per channel (rotated coordinates
            < d/2 at 4 bits, the rest at 3), no residual sketch, byte
            log-norms over [2^0, 2^8] (N(0,1) keys of d = 256 have norms near
            2^4); values 3b; FWHT; fp16 window 128.
  kivi      the qwen shape through the KIVI-like control arm of the design
            study: 2-bit keys per channel (page groups) and 2-bit values per
            token, float16 scale and zero, fp16 window 128; no rotation.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

_M64 = (1 << 64) - 1
_GOLD = 0x9E3779B97F4A7C15

DENSE = 0
FWHT = 1

TENSOR_K, TENSOR_V, TENSOR_Q, TENSOR_KSCALE, TENSOR_OUTLIER, TENSOR_VSCALE = 1, 2, 3, 4, 5, 6


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_kv_heads: int
    n_q_heads: int
    d: int
    ctx: int
    key_bits: int          # MSE bits of the key code (QJL adds one more bit)
    key_qjl: int           # key correction: 0 MSE only, 1 QJL, 2 EDEN scale, 3 length renormalization
    value_bits: int
    kind: int              # DENSE or FWHT
    window: int
    dtype: str             # "f32" or "bf16"
    layers: int = 1
    key_scale: str = "none"   # "pre_rope_exp", "outliers", "lognormal"
    value_scale: str = "none"
    rope: bool = True
    seed: int = 0
    head_dim: int = 0      # length of the generated vectors (0: d); heads shorter than d are zero-padded to d
    key_split: int = 0     # mixed-channel key rate: the first d/2 rotated coordinates one bit wider
    key_norm_range: tuple | None = None  # (lo, hi): byte key norms, log2-uniform over [2^lo, 2^hi]
    qjl_structured: int = 0  # QJL sketch S = H diag(sigma_S) in place of a dense Gaussian
    kivi: int = 0          # KIVI-like control arm (integer codes, key_bits / value_bits 2 or 4)

    @property
    def dh(self) -> int:
        return self.head_dim or self.d


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 4, 128, 1024, 2, True, 2, DENSE, 0, "f32", key_scale="pre_rope_exp"),
    "qwen": Workload("qwen", 8, 4, 24, 256, 32768, 2, True, 2, FWHT, 128, "bf16"),
    "llama": Workload("llama", 32, 8, 32, 128, 8192, 3, True, 4, DENSE, 0, "bf16", layers=32,
                      key_scale="outliers"),
    "long": Workload("long", 1, 2, 16, 256, 131072, 2, True, 2, FWHT, 0, "bf16"),
    "bulk": Workload("bulk", 1, 8, 8, 128, 65536, 3, True, 4, DENSE, 0, "bf16", layers=32,
                     key_scale="lognormal", value_scale="lognormal", rope=False),
    "mixed": Workload("mixed", 8, 4, 24, 256, 32768, 3, 0, 3, FWHT, 128, "bf16", key_split=1,
                      key_norm_range=(0.0, 8.0)),
    "kivi": Workload("kivi", 8, 4, 24, 256, 32768, 2, 0, 2, FWHT, 128, "bf16", kivi=1),
}


def workload(name: str, **over) -> Workload:
    return replace(WORKLOADS[name], **over)


# ----------------------------------------------------------------------------- generator

def _mix(z: int) -> int:
    z = (z + _GOLD) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_start(seed: int, *key: int) -> int:
    s = seed & _M64
    for k in key:
        s = _mix(s ^ (k & _M64))
    return s


def _outputs(state: int, first: int, n: int) -> np.ndarray:
    k = np.arange(first + 1, first + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(state) + k * np.uint64(_GOLD)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z ^= z >> np.uint64(31)
    return z


def normals(state: int, n: int, chunk: int = 1 << 22) -> np.ndarray:
    """n standard normals (float64) from one counter stream."""
    m = (n + 1) // 2
    out = np.empty(2 * m, dtype=np.float64)
    for c0 in range(0, m, chunk):
        c1 = min(m, c0 + chunk)
        z = _outputs(state, 2 * c0, 2 * (c1 - c0))
        u = (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        a = 2.0 * np.pi * u[1::2]
        out[2 * c0: 2 * c1: 2] = r * np.cos(a)
        out[2 * c0 + 1: 2 * c1: 2] = r * np.sin(a)
    return out[:n]


def uniform_ints(state: int, n: int, hi: int) -> np.ndarray:
    z = _outputs(state, 0, n)
    return (z % np.uint64(hi)).astype(np.int64)


# ----------------------------------------------------------------------------- tensors

def rope(x: np.ndarray, pos: np.ndarray, theta: float = 1e4) -> np.ndarray:
    """Rotate-half RoPE on the last axis; x [..., T, H, d], pos [T]."""
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = pos[:, None].astype(np.float64) * inv[None, :]          # [T, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the storage dtype (returned as float64 copies)."""
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        f = x.astype(np.float32)
        u = f.view(np.uint32).astype(np.uint64)
        u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
        return (u.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def keys_values(w: Workload, layer: int = 0, seqs=None, ctx: int | None = None) -> dict:
    """K, V [B', T, Hkv, d] and q [B', Hq, d] as float64 copies of the stored dtype.

    Sequences are generated independently (one stream per (tensor, layer,
    sequence)), so any subset of sequences can be drawn on its own.
    """
    T = w.ctx if ctx is None else ctx
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    H, Hq, d = w.n_kv_heads, w.n_q_heads, w.dh
    Ks, Vs, Qs = [], [], []
    for b in seqs:
        K = normals(stream_start(w.seed, TENSOR_K, layer, b), T * H * d).reshape(T, H, d)
        V = normals(stream_start(w.seed, TENSOR_V, layer, b), T * H * d).reshape(T, H, d)
        q = normals(stream_start(w.seed, TENSOR_Q, layer, b), Hq * d).reshape(1, Hq, d)
        if w.key_scale == "pre_rope_exp":
            g = normals(stream_start(w.seed, TENSOR_KSCALE, layer), H * d).reshape(H, d)
            K = K * np.exp(g)[None]
        if w.key_scale == "lognormal":
            g = normals(stream_start(w.seed, TENSOR_KSCALE, layer), H * d).reshape(H, d)
            K = K * np.exp(g)[None]
        if w.value_scale == "lognormal":
            g = normals(stream_start(w.seed, TENSOR_VSCALE, layer), H * d).reshape(H, d)
            V = V * np.exp(g)[None]
        if w.rope:
            K = rope(K, np.arange(T))
            q = rope(q, np.array([T]))
        if w.key_scale == "outliers":
            for h in range(H):
                st = stream_start(w.seed, TENSOR_OUTLIER, layer, h)
                perm = np.argsort(normals(st, d), kind="stable")[:4]
                K[:, h, perm] *= 20.0
        Ks.append(round_to(K, w.dtype))
        Vs.append(round_to(V, w.dtype))
        Qs.append(round_to(q[0], w.dtype))
    return {"K": np.stack(Ks), "V": np.stack(Vs), "q": np.stack(Qs)}


def to_torch(x: np.ndarray, dtype: str):
    """Convert float64 values (already representable) to a torch CPU tensor."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return {"f32": t, "bf16": t.to(torch.bfloat16), "f16": t.to(torch.float16)}[dtype]


def keys_values_torch(w: Workload, layer: int = 0, ctx: int | None = None, device="cuda", seed: int | None = None):
    """The same recipe drawn on the device with torch's seeded generator (for
    full-size benchmark caches, where the host generator is too slow).  The
    values differ from keys_values() (different generator), the distribution
    does not.  Returns K, V [B, T, Hkv, d] and q [B, Hq, d] in the workload dtype."""
    import torch

    T = w.ctx if ctx is None else ctx
    g = torch.Generator(device=device)
    g.manual_seed(stream_start(w.seed if seed is None else seed, 0xB0, layer) & ((1 << 63) - 1))
    B, H, Hq, d = w.batch, w.n_kv_heads, w.n_q_heads, w.dh
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.dtype]
    K = torch.randn(B, T, H, d, generator=g, device=device, dtype=torch.float32)
    V = torch.randn(B, T, H, d, generator=g, device=device, dtype=torch.float32)
    q = torch.randn(B, 1, Hq, d, generator=g, device=device, dtype=torch.float32)
    if w.key_scale in ("pre_rope_exp", "lognormal"):
        K *= torch.exp(torch.randn(H, d, generator=g, device=device))[None, None]
    if w.value_scale == "lognormal":
        V *= torch.exp(torch.randn(H, d, generator=g, device=device))[None, None]
    if w.rope:
        half = d // 2
        inv = 1e4 ** (-torch.arange(half, device=device, dtype=torch.float64) * 2.0 / d)

        def rot(x, pos):
            ang = (pos[:, None].double() * inv[None, :]).float()
            c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
            x1, x2 = x[..., :half], x[..., half:]
            return torch.cat([x1 * c - x2 * s, x1 * s + x2 * c], dim=-1)

        for b in range(B):
            K[b] = rot(K[b], torch.arange(T, device=device))
        q = rot(q, torch.tensor([T], device=device))
    if w.key_scale == "outliers":
        for h in range(H):
            idx = torch.randperm(d, generator=g, device=device)[:4]
            K[:, :, h, idx] *= 20.0
    return K.to(dt), V.to(dt), q[:, 0].to(dt)
