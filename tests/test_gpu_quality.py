"""Attention quality of the compressed decode against exact attention on the long-context
workload's first 4096 tokens ([Reconstruction] §15, Experiment A: KL divergence of the
attention weights, plus output error and cosine).  A report, not a parity gate: the test
prints the numbers and checks only that they are finite and of a sane size for 2-bit keys
with a 1-bit sketch and 2-bit values."""

import math

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_long_context_quality_report():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from kv_cache_vector_head_gb300 import build

    build.build()
    import kv_cache_vector_head_gb300 as tq

    import bench

    r = bench.quality_report(tq, torch)
    print("\nquality, long-context slice:", r)
    for k in ("max_abs_out_err", "out_cosine_mean", "kl_mean", "kl_max", "logit_max_abs_err"):
        assert math.isfinite(r[k]), k
    assert 0.5 < r["out_cosine_min"] <= 1.0 + 1e-9
    assert 0.0 <= r["kl_mean"] <= r["kl_max"] < 1.0
