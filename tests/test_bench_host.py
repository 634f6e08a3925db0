"""Host-side logic of bench.py: byte accounting and the cross-rank reduction
(two gloo ranks on the CPU; the GPU bench runs one replica per rank)."""

import os
import socket

import pytest

import bench
from oracle import paging as PG


def test_byte_accounting_matches_record_formulas():
    d, kb, vb = 256, 2, 2
    kr, vr = bench.record_bytes(d, kb, True, vb)
    assert kr + vr == PG.record_bytes(d, kb, True, vb) == 172
    B, Hkv, Hq, W = 8, 4, 24, 128
    T = 32768
    nc = PG.n_compressed(T, W)
    exp = B * Hkv * (nc * 172 + (T - nc) * d * 4) + B * Hq * d * 6
    assert bench.decode_bytes(T, W, B, Hkv, Hq, d, kb, vb) == exp
    assert bench.step_bytes(T, W, B, Hkv, Hq, d, kb, vb) == exp + B * Hkv * d * 8
    assert abs(exp / 1e6 - 183.8) < 0.5


@pytest.mark.parametrize("name", ["qwen", "llama", "long", "mixed", "kivi"])
def test_workload_records_match_the_page_formats(name):
    """bench.py's bytes per (token, kv head) for every bench workload equal the oracle's page
    layouts divided by the 16 tokens of a page (key and value parts separately where the
    layout splits them)."""
    import synthetic_kv as SK
    from oracle import kivi as OKV

    w = SK.workload(name)
    kr, vr = bench.workload_records(w)
    if w.kivi:
        lay = OKV.subblock_layout(w.d, w.key_bits, w.value_bits)
        assert 16 * kr == lay["value_scale"] and 16 * vr == lay["bytes"] - lay["value_scale"]
    else:
        lay = PG.subblock_layout(w.d, w.key_bits, int(w.key_qjl), w.value_bits, key_split=w.key_split,
                                 key_norm_u8=int(w.key_norm_range is not None))
        assert 16 * kr == lay["value_norm"] and 16 * vr == lay["bytes"] - lay["value_norm"]
    assert bench.workload_name(w).startswith(name)


def _worker(rank, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    q.put((rank, bench.max_over_ranks(10.0 + rank)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]
    assert bench.max_over_ranks(3.5) == 3.5  # single process: identity


def test_clock_summary_picks_the_gpu_and_the_window():
    """The sampler keeps the rows of the bench's GPU (PCI bus:device) and the samples inside the
    timed window; a window shorter than the sampling period is bracketed by its neighbours."""
    c = bench.Clocks("1b:00")
    row = lambda t, bus, sm, why=(): {"t": t, "bus": bus, "sm": sm, "max": 2070.0, "reasons": list(why)}
    c.samples = [row(1.00, "00000000:1B:00.0", 2070.0), row(1.05, "00000000:1C:00.0", 300.0),
                 row(1.50, "00000000:1B:00.0", 1900.0, ["sw_power_cap"]), row(3.0, "00000000:1B:00.0", 2070.0)]
    c.windows = {"timed": [1.2, 1.3]}
    s = c.summary("timed")
    assert s["how"].startswith("bracketing") and s["samples"] == 2 and s["sm_mhz"] == 1985.0
    assert s["reasons"] == ["sw_power_cap"]
    c.windows = {"timed": [0.9, 1.6]}
    s = c.summary("timed")
    assert s["how"] == "inside the window" and s["samples"] == 2 and s["sm_max_mhz"] == 2070.0
    assert bench.Clocks.bus_key("00000009:01:00.0") == "01:00"
    assert bench.Clocks(None).summary("timed") is None  # no samples, no window


def test_quantize_roofline_bounds():
    """Dense-mode bulk quantize is HBM-bound at the measured peaks: 652 B and 3 x 2 d^2 flops per
    token-head (d = 128); FWHT mode keeps one dense product (the Gaussian sketch)."""
    peaks = {"hbm_gbs": 6694.2, "bf16_tflops": 1942.3}
    n = 1 << 20
    r = bench.quantize_roofline(1.0, n, 0, peaks)
    assert r["bound"] == "hbm" and r["bytes_per_token_head"] == 652 and r["flops_per_token_head"] == 3 * 2 * 128 ** 2
    assert abs(r["frac"] - 652 * n / 6694.2e9 / 1e-3) < 1e-12
    f = bench.quantize_roofline(1.0, n, 1, peaks)
    assert f["flops_per_token_head"] == 2 * 128 ** 2 + 2 * 2 * 128 * 7
    s = bench.quantize_roofline(1.0, n, 1, peaks, structured=True)
    assert s["flops_per_token_head"] == 3 * 2 * 128 * 7


def test_launch_count_follows_the_workload():
    """Kernels a timed step launches: append kernel(s), counters, then the decode call."""
    import synthetic_kv as SK

    assert bench.launches_per_step(SK.workload("qwen")) == 5    # step kernel, counters, 3 decode kernels
    assert bench.launches_per_step(SK.workload("long")) == 5
    assert bench.launches_per_step(SK.workload("mixed")) == 5
    assert bench.launches_per_step(SK.workload("llama")) == 6   # key and value warp tiles, counters, 3
    assert bench.launches_per_step(SK.workload("kivi")) == 4    # step kernel, counters, page kernel, merge
