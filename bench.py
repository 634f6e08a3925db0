#!/usr/bin/env python
"""Benchmark of the TurboQuant KV-cache hot path on GB300.

Workload (Qwen-like full-attention layer): bf16 inputs, d = 256, 4 KV / 24 q
heads, batch 8, 32768-token context, keys 3 bits (2-bit Lloyd-Max code + 1-bit
QJL sketch), values 2 bits, FWHT rotation, 16-token pages, float16 window of
the last 128 tokens.  One step = the whole hot path of one decode step of one
layer: append one token per sequence (quantize K and V into the window ring,
flushing a page of 16 quantized tokens when due) and decode attention over the
compressed pages plus the window.  Steps rotate over several resident layer
caches so the working set (~770 MB) is far above the 129 MB L2.

Metric: algorithmic bytes of the step (compressed records of every cached
token, the float16 window, the new K/V, q and the output) per second, as GB/s
and as a fraction of the measured HBM bandwidth; plus bulk quantize
token-heads/s as a secondary line item.

  python bench.py [--gpus N --steps K --warmup W]          GPU path (libtq)
  python bench.py --impl reference [...]                   the CPU oracle
Under torchrun every rank runs its own replica (independent sequences, no
collective on the data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attention compressed-KV GB/s & % HBM roofline; quantize tokens·heads/s"


def key_mode(w) -> str:
    if w.kivi:
        return (f"KIVI-like control arm: keys {w.key_bits}b per channel over 16-token pages, "
                f"float16 scale and zero")
    if w.key_split:
        code = f"{w.key_bits + 0.5}b per channel (coordinates < d/2 at {w.key_bits + 1}b, the rest {w.key_bits}b)"
    else:
        code = f"{w.key_bits}b Lloyd-Max"
    corr = {0: "", 1: " + 1b QJL", 2: " + EDEN scale", 3: " + length renormalization"}[int(w.key_qjl)]
    total = f"{w.key_bits + 1}b " if int(w.key_qjl) == 1 and not w.key_split else ""
    norm = f", byte log-norms over [2^{w.key_norm_range[0]:g}, 2^{w.key_norm_range[1]:g}]" if w.key_norm_range else ""
    return f"keys {total}({code}{corr}{norm})"


def workload_name(w) -> str:
    kind = "FWHT" if w.kind == 1 else "dense Pi"
    return (f"{w.name}-like full-attention layer: {w.dtype}, d={w.d}, {w.n_kv_heads} KV / {w.n_q_heads} q heads, "
            f"batch {w.batch}, {w.ctx} ctx, {key_mode(w)}, "
            f"values {w.value_bits}b, {kind}, page 16, fp16 window {w.window}")


DEFAULT_LAYERS = {"qwen": 4, "llama": 4, "long": 8, "mixed": 4, "kivi": 4}  # resident layer caches: far above L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--workload", default="qwen", choices=["qwen", "llama", "long", "mixed", "kivi"],
                    help="decode configuration (default: the Qwen-like headline workload)")
    ap.add_argument("--layers", type=int, default=0, help="resident layer caches rotated over (0: per workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--quantize-only", action="store_true",
                    help="only the bulk quantize measurement (one JSON line), e.g. under a profiler")
    ap.add_argument("--prefill-attention-only", action="store_true",
                    help="only the prefill attention of 64-token chunks on the workload's cache (one JSON line)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="only the prefill of the workload's cache into pages (one JSON line)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers

def record_bytes(d, kb, qjl, vb, split=0, norm_u8=False):
    """Bytes of one key and one value record: norm (float32 or a byte), the correction's
    float32 slot, the code planes (half a bit more per channel with the mixed rate), the
    sign sketch (QJL)."""
    qjl = int(qjl)
    key = (1 if norm_u8 else 4) + (4 if qjl else 0) + kb * d // 8 + (d // 16 if split else 0) + (d // 8 if qjl == 1 else 0)
    return key, 4 + vb * d // 8


def launches_per_step(w) -> int:
    """Kernels one timed step launches: the append (d = 128 bf16 without a window: the key and value warp-tile
    kernels, else one step kernel) and the counters, then the decode call (query transform, page kernel and
    merge; the KIVI arm has no query transform)."""
    append = 2 if (w.window == 0 and w.d == 128 and w.dtype == "bf16" and not w.kivi) else 1
    return append + 1 + (2 if w.kivi else 3)


def workload_records(w):
    if w.kivi:  # key scale and zero per channel shared by a page's 16 tokens; value scale and zero per token
        return w.d // 4 + w.key_bits * w.d // 8, 4 + w.value_bits * w.d // 8
    return record_bytes(w.d, w.key_bits, w.key_qjl, w.value_bits, w.key_split, w.key_norm_range is not None)


def decode_bytes(T, W, B, Hkv, Hq, d, kb, vb, qjl=True, rec=None):
    """Algorithmic bytes one decode call reads and writes for sequences of length T:
    compressed records, the float16 window K and V, q (bf16) and the output (fp32)."""
    kr, vr = rec if rec is not None else record_bytes(d, kb, qjl, vb)
    nc = 16 * (max(0, T - W) // 16)
    return B * Hkv * (nc * (kr + vr) + (T - nc) * d * 2 * 2) + B * Hq * d * (2 + 4)


def step_bytes(T, W, B, Hkv, Hq, d, kb, vb, qjl=True, rec=None):
    """Algorithmic bytes of one step for sequences of length T (after the append)."""
    kr, vr = rec if rec is not None else record_bytes(d, kb, qjl, vb)
    nc = 16 * (max(0, T - W) // 16)
    nw = T - nc
    per_head = nc * (kr + vr) + nw * d * 2 * 2           # compressed records + fp16 window K,V
    append = B * Hkv * d * (2 * 2 + 2 * 2)                # new K,V in (bf16) + ring writes (fp16)
    return B * Hkv * per_head + append + B * Hq * d * (2 + 4)   # + q in (bf16) + out (fp32)


class Clocks:
    """nvidia-smi sampling around the timed region.  A reader thread stamps every
    sample with the host clock, so the samples that fall inside a marked window
    (plus a margin of one sampling period) can be picked out afterwards; if the
    window is shorter than the sampling period, the samples just before and just
    after it bracket it.  The GPU's row is matched by PCI bus id."""

    Q = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, bus_id=None):
        self.bus_id = (bus_id or "").lower()
        self.proc, self.samples, self.thread = None, [], None
        self.windows = {}

    def start(self):
        import threading

        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.PERIOD_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    rec = {"t": time.monotonic(), "bus": p[0].lower(), "sm": float(p[1]), "max": float(p[2]),
                           "reasons": [n for n, v in zip(self.NAMES, p[5:9]) if v.lower().startswith("active")]}
                except ValueError:
                    continue
                self.samples.append(rec)

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        t0 = time.monotonic()
        while not self.samples and time.monotonic() - t0 < 5.0:  # the first sample, so the window is bracketed
            time.sleep(0.01)

    def mark(self, name, which):
        w = self.windows.setdefault(name, [None, None])
        w[0 if which == "start" else 1] = time.monotonic()

    def stop(self):
        if self.proc is None:
            return
        t0 = time.monotonic()
        last = max((w[1] or 0.0) for w in self.windows.values()) if self.windows else t0
        while time.monotonic() - t0 < 2.0 and not any(r["t"] > last for r in self.samples):
            time.sleep(0.01)  # one sample after the last window
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    @staticmethod
    def bus_key(s):
        """'bus:device' in hex from nvidia-smi's 'domain:bus:device.function'."""
        p = s.lower().split(":")
        try:
            return f"{int(p[-2], 16):02x}:{int(p[-1].split('.')[0], 16):02x}"
        except (IndexError, ValueError):
            return s.lower()

    def summary(self, name):
        rows = self.samples
        buses = {self.bus_key(r["bus"]) for r in rows}
        if self.bus_id and self.bus_id in buses:
            rows = [r for r in rows if self.bus_key(r["bus"]) == self.bus_id]
        elif len(buses) > 1:
            return None
        if not rows or name not in self.windows or None in self.windows[name]:
            return None
        a, b = self.windows[name]
        pad = self.PERIOD_MS * 1e-3
        inside = [r for r in rows if a - pad <= r["t"] <= b + pad]
        how = "inside the window"
        if not inside:
            before = [r for r in rows if r["t"] < a]
            after = [r for r in rows if r["t"] > b]
            inside = before[-1:] + after[:1]
            how = "bracketing samples (window shorter than the sampling period)"
        if not inside:
            return None
        return {"sm_mhz": statistics.median(r["sm"] for r in inside), "sm_max_mhz": max(r["max"] for r in inside),
                "reasons": sorted({n for r in inside for n in r["reasons"]}), "samples": len(inside),
                "window_s": round(b - a, 4), "how": how}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def profiled_traffic():
    """DRAM bytes per decode call from the committed ncu summary, or None when
    the decode source changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "decode_qwen_ncu.md")
    src = os.path.join(ROOT, "kv_cache_vector_head_gb300", "csrc", "tq_decode.cu")
    try:
        fields = dict(ln.split(":", 1) for ln in open(path) if ln.startswith(("traffic_bytes_per_call:", "source_sha256:")))
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if fields.get("source_sha256", "").strip() != digest:
            return None
        return int(fields["traffic_bytes_per_call"].strip())
    except (OSError, ValueError, KeyError):
        return None


def max_over_ranks(x: float) -> float:
    """The largest value of x over all ranks (identity without torch.distributed)."""
    import torch

    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample_setup(name="qwen", seq=0, head=0):
    """One (sequence, KV head) unit of the workload (its G query heads), quantized
    by the oracle; a step is one append + decode over it."""
    import numpy as np

    import synthetic_kv as SK
    from oracle import codebook as OCB
    from oracle import codec as OC
    from oracle import transforms as OT

    w = SK.workload(name)
    kv = SK.keys_values(w, seqs=[seq])
    G = w.n_q_heads // w.n_kv_heads
    T, W, d = w.ctx, w.window, w.d
    nc = 16 * (max(0, T - W) // 16)
    kcb, vcb = OCB.lloyd_max(d, w.key_bits), OCB.lloyd_max(d, w.value_bits)
    kcb_hi = OCB.lloyd_max(d, w.key_bits + 1) if w.key_split else None
    corr = int(w.key_qjl)
    prm = {"kind": w.kind, "k_cb": kcb, "k_cb_hi": kcb_hi, "v_cb": vcb, "key_qjl": corr,
           "k_rot": [OT.build_transform(w.kind, d, 0, 0, head, 0)],
           "v_rot": [OT.build_transform(w.kind, d, 0, 0, head, 1)],
           "qjl_s": [OT.build_transform(w.kind, d, 0, 0, head, 2)] if corr == 1 else None}
    K, V = kv["K"][0, :, head].copy(), kv["V"][0, :, head].copy()
    q = kv["q"][0, head * G:(head + 1) * G].copy()
    del kv
    S = {"prm": prm, "kind": w.kind, "k_cb": kcb, "v_cb": vcb, "norm_range": w.key_norm_range}
    if w.kivi:  # the control arm: dequantized pages, attention over them and the window
        from oracle import kivi as OKV

        S["kivi"] = (OKV.dequantize_keys(OKV.quantize_keys(K[:nc], w.key_bits))[None],
                     OKV.dequantize_values(OKV.quantize_values(V[:nc], w.value_bits))[None])
        comp = None
    else:
        kr = oracle_keys(S, K[:nc])
        vr = OC.quantize_mse(V[:nc], w.kind, prm["v_rot"][0], vcb)
        comp = {"knorm": kr["norm"][None], "krnorm": kr["rnorm"][None], "kidx": kr["idx"][None],
                "ksigns": kr["signs"][None], "vnorm": vr["norm"][None], "vidx": vr["idx"][None]}
    win_k = K[nc:].astype(np.float16)[None]
    win_v = V[nc:].astype(np.float16)[None]
    kr_b, vr_b = workload_records(w)
    nbytes = nc * (kr_b + vr_b) + (T - nc) * d * 4 + d * (2 * 2 + 2 * 2) + G * d * 6
    S.update({"comp": comp, "win_k": win_k, "win_v": win_v, "q": q, "d": d, "bytes": nbytes,
              "new_k": K[-1:], "new_v": V[-1:], "T": T, "nc": nc, "G": G, "W": W})
    return S


def oracle_keys(S, K):
    """The oracle's key records in the workload's key mode, with the norms as stored
    (byte norms decoded) and neutral sketch fields where the mode has none."""
    import numpy as np

    from oracle import codec as OC

    prm = S["prm"]
    corr = prm["key_qjl"]
    if corr == 1:
        kr = OC.quantize_prod(K, S["kind"], prm["k_rot"][0], S["k_cb"], prm["qjl_s"][0])
    elif corr >= 2:
        kr = OC.quantize_scaled(K, S["kind"], prm["k_rot"][0], S["k_cb"], corr, cb_hi=prm["k_cb_hi"])
    else:
        kr = OC.quantize_mse(K, S["kind"], prm["k_rot"][0], S["k_cb"], cb_hi=prm["k_cb_hi"])
        kr["rnorm"] = np.zeros(K.shape[0], np.float32)
    kr.setdefault("signs", np.ones(kr["idx"].shape, dtype=bool))
    if S["norm_range"] is not None:
        kr["norm"] = OC.norm_u8_decode(OC.norm_u8_encode(kr["norm_f64"], *S["norm_range"])[0], *S["norm_range"])
    return kr


def oracle_step(S):
    from oracle import attention as OA
    from oracle import codec as OC

    import numpy as np

    if S["W"] > 0:
        # append: the new token enters the float16 window (no page flush due at this length)
        nk = S["new_k"].astype(np.float16)[None]
        nv = S["new_v"].astype(np.float16)[None]
        wk = np.concatenate([S["win_k"][:, 1:], nk], axis=1)
        wv = np.concatenate([S["win_v"][:, 1:], nv], axis=1)
        comp = S["comp"]
        if "kivi" in S:
            from oracle import kivi as OKV

            return OKV.decode_one(S["q"], S["kivi"][0], S["kivi"][1], wk, wv, 1.0 / math.sqrt(S["d"]))
    else:
        # no window: the new token is quantized into its page slot
        prm = S["prm"]
        kr = oracle_keys(S, S["new_k"])
        vr = OC.quantize_mse(S["new_v"], S["kind"], prm["v_rot"][0], S["v_cb"])
        c = S["comp"]
        comp = {"knorm": np.concatenate([c["knorm"][:, 1:], kr["norm"][None]], axis=1),
                "krnorm": np.concatenate([c["krnorm"][:, 1:], kr["rnorm"][None]], axis=1),
                "kidx": np.concatenate([c["kidx"][:, 1:], kr["idx"][None]], axis=1),
                "ksigns": np.concatenate([c["ksigns"][:, 1:], kr["signs"][None]], axis=1),
                "vnorm": np.concatenate([c["vnorm"][:, 1:], vr["norm"][None]], axis=1),
                "vidx": np.concatenate([c["vidx"][:, 1:], vr["idx"][None]], axis=1)}
        wk = wv = None
    OC.qjl_constant(S["d"])
    return OA.decode_one(S["q"], comp, wk, wv, S["prm"], 1.0 / math.sqrt(S["d"]))


def host_cores():
    """(os.cpu_count(), CPUs this process may run on)."""
    n = os.cpu_count() or 1
    try:
        return n, len(os.sched_getaffinity(0))
    except AttributeError:
        return n, n


def _one_thread_env():
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        os.environ[k] = "1"


def _decode_worker(name, seq, head, steps, barrier, conn):
    """Spawned worker: set up one (sequence, KV head) unit, then time `steps` oracle
    steps (after the barrier) or, with steps == 0, run one step per request on conn."""
    _one_thread_env()
    S = oracle_sample_setup(name, seq, head)
    oracle_step(S)  # warm-up
    barrier.wait()
    if steps > 0:
        t0 = time.perf_counter()
        for _ in range(steps):
            oracle_step(S)
        conn.send((S["bytes"] * steps, time.perf_counter() - t0))
        return
    conn.send(S["bytes"])
    while conn.recv():
        oracle_step(S)
        conn.send(True)


def _quantize_worker(n_vec, kind, layer, barrier, conn):
    """Spawned worker: the oracle's bulk quantize (keys 3b + QJL, values 4b, d = 128) of
    n_vec token-heads of the bulk recipe (bf16 N(0,1) x lognormal channel scales)."""
    _one_thread_env()
    import synthetic_kv as SK
    from oracle import codebook as OCB
    from oracle import codec as OC
    from oracle import transforms as OT

    w = SK.workload("bulk", kind=kind)
    H, d = w.n_kv_heads, w.d
    kv = SK.keys_values(w, layer=layer, ctx=n_vec // H)
    K, V = kv["K"][0], kv["V"][0]                      # [T, H, d]
    kcb, vcb = OCB.lloyd_max(d, w.key_bits), OCB.lloyd_max(d, w.value_bits)
    tr = [(OT.build_transform(kind, d, 0, layer, h, 0), OT.build_transform(kind, d, 0, layer, h, 1),
           OT.build_transform(kind, d, 0, layer, h, 2)) for h in range(H)]
    barrier.wait()
    t0 = time.perf_counter()
    for h in range(H):
        kr = OC.quantize_prod(K[:, h], kind, tr[h][0], kcb, tr[h][2])
        vr = OC.quantize_mse(V[:, h], kind, tr[h][1], vcb)
        OC.pack_codes(kr["idx"], w.key_bits), OC.pack_bits(kr["signs"]), OC.pack_codes(vr["idx"], w.value_bits)
    conn.send((K.shape[0] * H, time.perf_counter() - t0))


def _spawn_timed(target, argsets):
    """Run target(*args, barrier, conn) in one spawned process per argset, all timed
    from a common barrier; returns their (work, seconds) results."""
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(len(argsets), timeout=600)
    procs, conns = [], []
    for a in argsets:
        r, w_ = ctx.Pipe(duplex=False)
        p = ctx.Process(target=target, args=(*a, barrier, w_))
        p.start()
        w_.close()  # a worker that dies then ends our recv with EOFError
        procs.append(p)
        conns.append(r)
    try:
        out = [_recv(c, 900) for c in conns]
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
    return out


def _recv(conn, timeout):
    if not conn.poll(timeout):
        raise TimeoutError("oracle worker did not answer")
    return conn.recv()


def run_cpu_sample(name="qwen"):
    """The oracle on the host cores: decode of the workload on (sequence, KV head) units,
    one per core in parallel and one on a single core, and the bulk quantize of the bulk
    recipe (FWHT and dense Pi), multi- and single-core.  Bounded samples."""
    import synthetic_kv as SK

    ncpu, cores = host_cores()
    w = SK.workload(name)
    units = [(b, g) for b in range(w.batch) for g in range(w.n_kv_heads)]
    par = max(1, min(cores, len(units), 16))
    steps = 2
    one = _spawn_timed(_decode_worker, [(name, 0, 0, steps)])[0]
    multi = _spawn_timed(_decode_worker, [(name, b, g, steps) for b, g in units[:par]])
    mbytes, msec = sum(x[0] for x in multi), max(x[1] for x in multi)
    out = {"value": mbytes / msec / 1e9, "unit": "GB/s", "cores": par, "kind": "oracle",
           "sample": (f"decode: {par} (sequence, KV head) units of the workload in parallel (one process per core, "
                      f"1 BLAS thread each), {steps} append + decode steps each, T={w.ctx}"),
           "host_cpu_count": ncpu, "host_cpus_usable": cores,
           "single_core": {"value": one[0] / one[1] / 1e9, "unit": "GB/s", "cores": 1,
                           "sample": f"1 unit, {steps} steps"}}
    qn1, qn = 1 << 15, 1 << 15
    qpar = max(1, min(cores, 16))
    quant = {}
    for kname, kind in (("fwht", SK.FWHT), ("dense", SK.DENSE)):
        s1 = _spawn_timed(_quantize_worker, [(qn1, kind, 0)])[0]
        sm = _spawn_timed(_quantize_worker, [(qn, kind, l) for l in range(qpar)])
        quant[kname] = {"token_heads_per_s": sum(x[0] for x in sm) / max(x[1] for x in sm), "cores": qpar,
                        "single_core_token_heads_per_s": s1[0] / s1[1]}
    quant["sample"] = (f"keys 3b + QJL and values 4b, d = 128, bulk recipe; {qn} token-heads per core "
                       f"({qpar} cores, one process each), {qn1} on one core")
    out["quantize"] = quant
    return out


def cpu_baseline_subprocess(name="qwen"):
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", "--workload", name],
                       capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "failed"}
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_reference(args):
    """The oracle as the reference arm: each step runs one append + decode on one
    (sequence, KV head) unit per host core, in parallel (spawned processes, one BLAS
    thread each); the step's bytes are the units' algorithmic bytes."""
    import multiprocessing as mp

    ws, rank, _ = dist_info()
    if rank != 0:
        return
    import synthetic_kv as SK

    w = SK.workload(args.workload)
    _, cores = host_cores()
    units = [(b, g) for b in range(w.batch) for g in range(w.n_kv_heads)]
    par = max(1, min(cores, len(units), 16))
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(par, timeout=600)
    procs, conns = [], []
    for b, g in units[:par]:
        a, c = ctx.Pipe()
        p = ctx.Process(target=_decode_worker, args=(args.workload, b, g, 0, barrier, c))
        p.start()
        c.close()
        procs.append(p)
        conns.append(a)
    step_bytes_ = sum(_recv(c, 900) for c in conns)

    def one_step():
        t0 = time.perf_counter()
        for c in conns:
            c.send(True)
        for c in conns:
            _recv(c, 300)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one_step()
    times = [one_step() for _ in range(args.steps)]
    for c in conns:
        c.send(False)
    for p in procs:
        p.join(timeout=30)
        if p.is_alive():
            p.terminate()
    dt = sum(times) / len(times)
    value = step_bytes_ / dt / 1e9
    sample = (f"each step: {par} (sequence, KV head) units of the workload ({w.n_q_heads // w.n_kv_heads} q heads "
              f"each), one per host core in parallel, T={w.ctx}, {step_bytes_ / 1e6:.1f} MB algorithmic bytes")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(w), "sample": f"{par} (sequence, KV head) units per step"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": par, "kind": "oracle", "sample": sample,
                             "host_cpu_count": os.cpu_count()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU path

QUANT_BYTES_PER_TOKEN_HEAD = 2 * 128 * 2 + 140   # bf16 K and V in, 140 B of records out (d = 128, 3b + QJL / 4b)


def quantize_roofline(ms, n, kind, peaks, structured=False):
    """Roofline of bulk quantize over n token-heads: max(bytes / HBM bandwidth, flops / tensor
    peak).  Algorithmic flops per token-head: 2 d^2 for each dense product (Pi k, S r, Pi_v v)
    and 2 d log2 d for each fast transform."""
    d = 128
    dense, fwht = 2 * d * d, 2 * d * int(math.log2(d))
    flops = (3 * dense if kind == 0 else (2 * fwht + (fwht if structured else dense))) * n
    nbytes = QUANT_BYTES_PER_TOKEN_HEAD * n
    bw = peaks.get("hbm_gbs", 6800.0) * 1e9
    tc = peaks.get("bf16_tflops", 1900.0) * 1e12
    t_b, t_f = nbytes / bw, flops / tc
    t = ms * 1e-3
    bound = "hbm" if t_b >= t_f else "tensor"
    return {"bound": bound, "achieved": (nbytes / t / 1e9) if bound == "hbm" else (flops / t / 1e12),
            "peak": bw / 1e9 if bound == "hbm" else tc / 1e12, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": max(t_b, t_f) / t, "flops_per_token_head": flops / n, "bytes_per_token_head": nbytes / n}


def bench_quantize(tq, torch, peaks, n=1 << 20):
    """Bulk prefill quantize of n token-heads (d = 128, 8 KV heads, keys 3b + QJL, values 4b) on
    the bulk recipe: bf16 N(0,1) K and V times lognormal(sigma = 1) channel scales per head.
    Keys and values are timed separately (inputs of 256 MB each, larger than L2)."""
    import synthetic_kv as SK

    out = {}
    w = SK.workload("bulk")
    K, V, _ = SK.keys_values_torch(w, ctx=n // w.n_kv_heads)
    x = K.reshape(n, w.d).contiguous()        # vector index = token * Hkv + head
    y = V.reshape(n, w.d).contiguous()
    del K, V
    for name, kind, structured in (("fwht", tq.TQ_FWHT, False), ("dense", tq.TQ_DENSE, False),
                                   ("fwht_structured_sketch", tq.TQ_FWHT, True)):
        L = tq.TQLayer(128, 8, 8, 3, 4, kind, qjl_structured=structured)
        codes = torch.empty(n, 12, dtype=torch.int32, device="cuda")
        signs = torch.empty(n, 4, dtype=torch.int32, device="cuda")
        nk = torch.empty(n, device="cuda")
        rk = torch.empty(n, device="cuda")
        vcodes = torch.empty(n, 16, dtype=torch.int32, device="cuda")
        nv = torch.empty(n, device="cuda")

        def keys():
            tq.quantize_keys(L.params, x, n, codes, signs, nk, rk)

        def values():
            tq.quantize_values(L.params, y, n, vcodes, nv)

        ms = {}
        for role, f in (("keys", keys), ("values", values)):
            for _ in range(3):
                f()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
            e0.record()
            for _ in range(5):
                f()
            e1.record()
            torch.cuda.synchronize()
            ms[role] = e0.elapsed_time(e1) / 5
        tot = ms["keys"] + ms["values"]
        out[name] = {"token_heads_per_s": n / (tot * 1e-3), "ms": tot, "keys_ms": ms["keys"],
                     "values_ms": ms["values"], "GB_per_s": n * QUANT_BYTES_PER_TOKEN_HEAD / tot / 1e6,
                     "roofline": quantize_roofline(tot, n, kind, peaks, structured)}
    return out


def bench_prefill_quantize(tq, torch, L, w, peaks, calls=3):
    """Prefill of the workload's cache: every sequence's n_c compressed tokens quantized
    straight into their pages in one direct-slot append call (keys and values), as
    PagedCache.prefill does.  Bytes per token-head: bf16 K, V in, one record out."""
    import synthetic_kv as SK

    B, Hkv, T, W = w.batch, w.n_kv_heads, w.ctx, w.window
    nc = 16 * (max(0, T - W) // 16)
    pc = tq.PagedCache(L, B, T)
    K, V, _ = SK.keys_values_torch(w, layer=7, ctx=nc)
    kk = K.reshape(B * nc, Hkv, w.dh).contiguous()
    vv = V.reshape(B * nc, Hkv, w.dh).contiguous()
    del K, V
    slots = pc.slot_mapping(nc)
    tq.append_page(L.params, pc.cache, kk, vv, B * nc, slots, None)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
    e0.record()
    for _ in range(calls):
        tq.append_page(L.params, pc.cache, kk, vv, B * nc, slots, None)
    e1.record()
    torch.cuda.synchronize()
    if tq.check_device_error():
        raise RuntimeError("device error in the prefill benchmark")
    ms = e0.elapsed_time(e1) / calls
    kr, vr = workload_records(w)
    per = 2 * 2 * w.dh + kr + vr
    n = B * nc * Hkv
    bw = peaks.get("hbm_gbs", 6800.0)
    gbs = n * per / (ms * 1e-3) / 1e9
    return {"token_heads": n, "ms": ms, "token_heads_per_s": n / (ms * 1e-3), "GB_per_s": gbs,
            "hbm_fraction": gbs / bw, "bytes_per_token_head": per,
            "config": f"{B} sequences x {nc} tokens x {Hkv} KV heads into pages (one call)"}


def quality_report(tq, torch, T=4096):
    """Attention quality on the long-context workload's first T tokens (d = 256, 2 KV / 16 q heads,
    FWHT, keys 2b + QJL, values 2b, no window): the GPU decode over the compressed cache against
    exact attention in float64 on the same bf16 K, V and q.  Reports the largest output error, the
    output cosine and KL(p_exact || p_tq) of the attention weights per query head
    ([Reconstruction] §15, Experiment A's metric).  A report, not a gate."""
    import numpy as np

    import synthetic_kv as SK

    w = SK.workload("long")
    K, V, q = SK.keys_values_torch(w, ctx=T)
    L = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=w.window, seed=w.seed)
    pc = tq.PagedCache(L, 1, T)
    pc.prefill(K, V)
    ws = torch.empty(tq.decode_workspace_size(L.params, 1, T), dtype=torch.uint8, device="cuda")
    out = torch.zeros(1, w.n_q_heads, w.d, device="cuda")
    scores = torch.zeros(1, w.n_q_heads, T, device="cuda")
    tq.decode_attention(L.params, pc.cache, q, 1.0 / math.sqrt(w.d), out, None, scores, ws, T)
    torch.cuda.synchronize()
    if tq.check_device_error():
        raise RuntimeError("device error in the quality report")
    G = w.n_q_heads // w.n_kv_heads
    Kf = K[0].double().cpu().numpy()          # [T, Hkv, d]
    Vf = V[0].double().cpu().numpy()
    qf = q[0].double().cpu().numpy()          # [Hq, d]
    kv = np.arange(w.n_q_heads) // G
    logits = np.einsum("hd,thd->ht", qf, Kf[:, kv]) / math.sqrt(w.d)
    pe = np.exp(logits - logits.max(1, keepdims=True))
    pe /= pe.sum(1, keepdims=True)
    oe = np.einsum("ht,thd->hd", pe, Vf[:, kv])
    st = scores[0].double().cpu().numpy()
    pt = np.exp(st - st.max(1, keepdims=True))
    pt /= pt.sum(1, keepdims=True)
    ot = out[0].double().cpu().numpy()
    kl = np.sum(pe * (np.log(pe) - np.log(pt)), axis=1)
    cos = np.sum(oe * ot, 1) / (np.linalg.norm(oe, axis=1) * np.linalg.norm(ot, axis=1))
    return {"tokens": T,
            "workload": "long-context first 4096 tokens: d=256, 2 KV / 16 q heads, FWHT, keys 2b+QJL, values 2b",
            "max_abs_out_err": float(np.abs(ot - oe).max()), "out_cosine_mean": float(cos.mean()),
            "out_cosine_min": float(cos.min()), "kl_mean": float(kl.mean()), "kl_max": float(kl.max()),
            "logit_max_abs_err": float(np.abs(st - logits).max())}


def bench_prefill(tq, torch, L, pc, w, recs, nq=64, calls=5):
    """Prefill attention: the last nq appended tokens of every sequence of one layer
    cache attend causally to it (one tq_prefill_attention call: query tiles of 16
    (query, head) rows per page pass where the layer allows it, else batch x nq
    virtual decode sequences).  Algorithmic bytes: every query's visible records,
    window, q and output, as for a decode call of its length."""
    B, Hkv, Hq, d, W = w.batch, w.n_kv_heads, w.n_q_heads, w.d, w.window
    T = int(pc.seq_len[0].item())
    q = torch.randn(B, nq, Hq, d, device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(tq.prefill_workspace_size(L.params, B, nq, T), dtype=torch.uint8, device="cuda")
    out = torch.empty(B, nq, Hq, d, device="cuda")
    for _ in range(2):
        tq.prefill_attention(L.params, pc.cache, nq, q, 1.0 / math.sqrt(d), out, None, ws, T)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
    e0.record()
    for _ in range(calls):
        tq.prefill_attention(L.params, pc.cache, nq, q, 1.0 / math.sqrt(d), out, None, ws, T)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / calls
    nbytes = sum(decode_bytes(T - nq + i + 1, W, B, Hkv, Hq, d, w.key_bits, w.value_bits, rec=recs)
                 for i in range(nq))
    return {"n_query": nq, "ctx": T, "ms": ms, "query_tokens_per_s": B * nq / (ms * 1e-3),
            "visible_GB_per_s": nbytes / (ms * 1e-3) / 1e9,
            "note": "visible bytes count every query's records; a page pass serves 16 (query, head) rows"}


def bench_append_batch256(tq, torch, steps=200):
    """Decode-step append latency: 256 sequences x 8 KV heads, d = 128, keys 3b + QJL,
    values 4b, dense Pi, no window, into partially filled pages (37 tokens each at
    the start); one call quantizes and stores one token per sequence."""
    import synthetic_kv as SK

    w = SK.workload("llama", batch=256, ctx=37, n_q_heads=8)
    L = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=0, seed=w.seed)
    pc = tq.PagedCache(L, w.batch, w.ctx + steps + 32)
    K, V, _ = SK.keys_values_torch(w, ctx=w.ctx + steps + 8)
    pc.prefill(K[:, :w.ctx], V[:, :w.ctx])
    news = [(K[:, t].contiguous(), V[:, t].contiguous()) for t in range(w.ctx, w.ctx + steps + 8)]
    for i in range(5):
        pc.append(*news[i])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
    e0.record()
    for i in range(steps):
        pc.append(*news[5 + i])
    e1.record()
    torch.cuda.synchronize()
    if tq.check_device_error():
        raise RuntimeError("device error in the append benchmark")
    us = e0.elapsed_time(e1) * 1e3 / steps
    return {"us_per_call": us, "token_heads_per_s": w.batch * w.n_kv_heads / (us * 1e-6),
            "config": "256 seqs x 8 KV heads, d=128, keys 3b+QJL, values 4b, dense Pi, 1 token per call"}


def run_gpu(args):
    import torch

    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    from kv_cache_vector_head_gb300 import build

    build.build()
    import kv_cache_vector_head_gb300 as tq
    import synthetic_kv as SK

    w = SK.workload(args.workload, seed=1000 * rank)
    B, Hkv, Hq, d, T0, W = w.batch, w.n_kv_heads, w.n_q_heads, w.d, w.ctx, w.window
    recs = workload_records(w)
    if args.layers <= 0:
        args.layers = DEFAULT_LAYERS[args.workload]
    total_steps = args.warmup + 2 * args.steps
    per_layer = (total_steps + args.layers - 1) // args.layers + 1
    max_ctx = T0 + per_layer + 16
    layers, caches, qs, news = [], [], [], []
    for l in range(args.layers):
        L = tq.TQLayer(d, Hkv, Hq, w.key_bits, w.value_bits, w.kind, window=W, key_qjl=w.key_qjl, seed=w.seed,
                       layer=l, key_split=w.key_split, key_norm_range=w.key_norm_range, kivi=w.kivi)
        pc = tq.PagedCache(L, B, max_ctx)
        K, V, q = SK.keys_values_torch(w, layer=l, ctx=T0 + per_layer)
        pc.prefill(K[:, :T0], V[:, :T0])
        news.append((K[:, T0:].transpose(0, 1).contiguous(), V[:, T0:].transpose(0, 1).contiguous()))
        del K, V
        layers.append(L)
        caches.append(pc)
        qs.append(q.contiguous())
    torch.cuda.synchronize()
    if tq.check_device_error():
        raise RuntimeError("device error after prefill")
    wsz = tq.decode_workspace_size(layers[0].params, B, max_ctx)
    work = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    out = torch.empty(B, Hq, d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    T = [T0] * args.layers
    used = [0] * args.layers

    def step(i, k=None, v=None, q=None, dec_ev=None, o=None):
        l = i % args.layers
        j = used[l]
        used[l] += 1
        kk = news[l][0][j] if k is None else k
        vv = news[l][1][j] if v is None else v
        caches[l].append(kk, vv)
        T[l] += 1
        if dec_ev is not None:
            dec_ev[0].record()
        tq.decode_attention(layers[l].params, caches[l].cache, qs[l] if q is None else q, scale,
                            out if o is None else o, None, None, work, max_ctx)
        if dec_ev is not None:
            dec_ev[1].record()
        return step_bytes(T[l], W, B, Hkv, Hq, d, w.key_bits, w.value_bits, rec=recs)

    props = torch.cuda.get_device_properties(local)
    bus = (f"{getattr(props, 'pci_bus_id', 0):02x}:{getattr(props, 'pci_device_id', 0):02x}"
           if hasattr(props, "pci_bus_id") else None)
    clocks = Clocks(bus)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # the clock sampler sees the GPU under this load for ~0.4 s before the timed steps (decode
    # calls only: the caches are not appended to)
    t_soak = time.monotonic()
    while time.monotonic() - t_soak < 0.4:
        for l in range(args.layers):
            tq.decode_attention(layers[l].params, caches[l].cache, qs[l], scale, out, None, None, work, max_ctx)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    ev = [(torch.cuda.Event(True), torch.cuda.Event(True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(True), torch.cuda.Event(True)
    clocks.mark("timed", "start")
    torch.cuda.nvtx.range_push("timed")
    t0.record()
    total_bytes = 0
    for i in range(args.steps):
        total_bytes += step(args.warmup + i, dec_ev=ev[i])
    t1.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    clocks.mark("timed", "end")
    clocks.stop()
    clk = clocks.summary("timed")
    ms = t0.elapsed_time(t1)
    dec_ms = [a.elapsed_time(b) for a, b in ev]
    if tq.check_device_error():
        raise RuntimeError("device error during the timed steps")
    ms = max_over_ranks(ms)
    # end to end through the public API with host buffers: H2D of the step's K, V, q
    # from pinned memory and D2H of the output, inside the timed region.  The copies run on a
    # stream of their own into double buffers, so step i + 1's inputs and step i's output move
    # while the compute stream runs (events order every buffer's reuse)
    npool = 16  # pinned host copies of step inputs, used cyclically
    hk = [news[i % args.layers][0][i // args.layers].cpu().pin_memory() for i in range(npool)]
    hv = [news[i % args.layers][1][i // args.layers].cpu().pin_memory() for i in range(npool)]
    hq = [qs[i % args.layers].cpu().pin_memory() for i in range(npool)]
    houts = [torch.empty(B, Hq, d).pin_memory() for _ in range(2)]
    dks = [torch.empty_like(news[0][0][0]) for _ in range(2)]
    dvs = [torch.empty_like(news[0][1][0]) for _ in range(2)]
    dqs = [torch.empty_like(qs[0]) for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    cs, xs = torch.cuda.current_stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b copied
    ev_used = [torch.cuda.Event() for _ in range(2)]  # the step on buffer b done (its inputs free, its output written)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # output b copied to the host (free again)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
    e0.record(cs)
    xs.wait_event(e0)

    def h2d(i):
        b = i % 2
        with torch.cuda.stream(xs):
            if i >= 2:
                xs.wait_event(ev_used[b])  # step i - 2 has read buffer b
            dks[b].copy_(hk[i % npool], non_blocking=True)
            dvs[b].copy_(hv[i % npool], non_blocking=True)
            dqs[b].copy_(hq[i % npool], non_blocking=True)
            ev_in[b].record(xs)

    e2e_bytes = 0
    if args.steps > 0:
        h2d(0)
    for i in range(args.steps):
        b = i % 2
        if i + 1 < args.steps:
            h2d(i + 1)
        cs.wait_event(ev_in[b])
        if i >= 2:
            cs.wait_event(ev_out[b])  # the host has step i - 2's output: buffer b may be overwritten
        e2e_bytes += step(args.warmup + args.steps + i, dks[b], dvs[b], dqs[b], o=outs[b])
        ev_used[b].record(cs)
        with torch.cuda.stream(xs):
            xs.wait_event(ev_used[b])
            houts[b].copy_(outs[b], non_blocking=True)
            ev_out[b].record(xs)
    cs.wait_stream(xs)
    e1.record(cs)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms)
    peaks = measured_peaks() or {}
    pre = bench_prefill(tq, torch, layers[0], caches[0], w, recs)
    del caches
    pre_q = bench_prefill_quantize(tq, torch, layers[0], w, peaks) if not w.kivi else None
    quant = bench_quantize(tq, torch, peaks)
    app = bench_append_batch256(tq, torch)
    qual = quality_report(tq, torch)
    if rank != 0:
        return
    peak = peaks["hbm_gbs"] if "hbm_gbs" in peaks else 6800.0
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    value = total_bytes * ws / (ms * 1e-3) / 1e9
    # roofline of the decode call (prologue + tensor-core split-K kernel + combine),
    # algorithmic bytes of its reads and writes per launch over its measured duration
    dec_bytes = decode_bytes(T0 + 1 + args.warmup // args.layers, W, B, Hkv, Hq, d, w.key_bits, w.value_bits,
                             rec=recs)
    dec_avg = statistics.mean(dec_ms)
    achieved = dec_bytes / (dec_avg * 1e-3) / 1e9
    traffic = profiled_traffic() if args.workload == "qwen" else None  # the capture is of the Qwen-like call
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded torch Philox on the device)",
        "config": {"workload": workload_name(w), "batch": B, "ctx": T0, "kv_heads": Hkv, "q_heads": Hq, "d": d,
                   "key_bits": w.key_bits + (0.5 if w.key_split else (1 if int(w.key_qjl) == 1 and not w.kivi else 0)),
                   "value_bits": w.value_bits, "window": W, "page": 16,
                   "layer_caches": args.layers, "l2": f"inputs larger than L2: {args.layers} rotating layer caches "
                   f"of {step_bytes(T0, W, B, Hkv, Hq, d, w.key_bits, w.value_bits, rec=recs) / 1e6:.0f} MB",
                   "parallelism": f"replicas x{ws}"},
        "hbm_fraction": value / ws / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": "tq_decode_attention (prologue + split-K tensor-core + combine)",
                     "peak_source": peak_src},
        "quantize": {"metric": ("bulk quantize token-heads/s (d=128, 8 KV heads, keys 3b+QJL, values 4b, 2^20 "
                                "token-heads of the bulk recipe: bf16 N(0,1) x lognormal(sigma=1) channel scales)"),
                     "fwht": dict(quant["fwht"], hbm_fraction=quant["fwht"]["GB_per_s"] / peak),
                     "dense": dict(quant["dense"], hbm_fraction=quant["dense"]["GB_per_s"] / peak),
                     "fwht_structured_sketch": dict(quant["fwht_structured_sketch"],
                                                    hbm_fraction=quant["fwht_structured_sketch"]["GB_per_s"] / peak)},
        "prefill_quantize": pre_q,
        "append_batch256": app,
        "prefill": pre,
        "quality": qual,
        "e2e": {"value": e2e_bytes * ws / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in (dks[0], dvs[0], dqs[0]))),
                "d2h_bytes_per_step": int(houts[0].numel() * houts[0].element_size()),
                "copies": "own stream, double-buffered, overlapping the compute stream"},
        "gpu_launches": args.steps * launches_per_step(w),
        "clocks": clk,
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args.workload)
    print(json.dumps(line), flush=True)


def run_gpu_part(args):
    """One measurement of run_gpu on its own (bulk quantize, or the workload's prefill into pages)."""
    import torch

    from kv_cache_vector_head_gb300 import build

    build.build()
    import kv_cache_vector_head_gb300 as tq
    import synthetic_kv as SK

    peaks = measured_peaks() or {}
    if args.quantize_only:
        print(json.dumps(bench_quantize(tq, torch, peaks)))
        return
    w = SK.workload(args.workload)
    if args.prefill_attention_only:
        L = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=w.window,
                       key_qjl=w.key_qjl, seed=w.seed, layer=0, key_split=w.key_split,
                       key_norm_range=w.key_norm_range, kivi=w.kivi)
        pc = tq.PagedCache(L, w.batch, w.ctx + 16)
        K, V, _ = SK.keys_values_torch(w, layer=0, ctx=w.ctx)
        pc.prefill(K, V)
        del K, V
        torch.cuda.synchronize()
        if tq.check_device_error():
            raise RuntimeError("device error after prefill")
        print(json.dumps(bench_prefill(tq, torch, L, pc, w, workload_records(w))))
        return
    if w.kivi:
        raise SystemExit("--prefill-only: the KIVI arm fills pages in its own layout")
    L = tq.TQLayer(w.d, w.n_kv_heads, w.n_q_heads, w.key_bits, w.value_bits, w.kind, window=w.window,
                   key_qjl=w.key_qjl, seed=w.seed, layer=0, key_split=w.key_split, key_norm_range=w.key_norm_range)
    print(json.dumps(bench_prefill_quantize(tq, torch, L, w, peaks)))


def main():
    args = parse()
    if args.cpu_sample:
        print(json.dumps(run_cpu_sample(args.workload)))
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.quantize_only or args.prefill_only or args.prefill_attention_only:
        run_gpu_part(args)
        return
    run_gpu(args)


if __name__ == "__main__":
    main()
