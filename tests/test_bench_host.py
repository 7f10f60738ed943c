"""Host-side arithmetic of bench.py without a GPU: the clock-record summary that
decides whether a timed run is kept, the allowed-pair count behind the cross-
attention flops, the per-kernel matmul flops and the whole-job throughput."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from attention_forward_backward_gb300 import synth  # noqa: E402


def test_clock_summary_median_max_and_reasons():
    lines = [
        "0, 1965, 2070, 801.2, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1205.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1500, 2070, 1390.9, 0x0000000000000044, Not Active, Not Active, Active, Active",
    ]
    out = bench.summarize_clocks(lines)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 1965.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    assert bench.summarize_clocks(["", "x, y"]) is None


def _pairs_brute(Lq, Lk, mask):
    off = (Lk - Lq) if mask == "causal_bottom_right" else 0
    n = 0
    for i in range(Lq):
        for j in range(Lk):
            n += mask == "none" or j <= i + off
    return n


@pytest.mark.parametrize("mask", ["none", "causal", "causal_bottom_right"])
@pytest.mark.parametrize("Lq,Lk", [(1, 1), (1, 7), (7, 1), (5, 5), (64, 200), (200, 64), (33, 97)])
def test_allowed_pairs_matches_brute_force(Lq, Lk, mask):
    assert bench.allowed_pairs(Lq, Lk, mask) == _pairs_brute(Lq, Lk, mask)


def test_allowed_pairs_closed_forms():
    L = 8192
    assert bench.allowed_pairs(L, L, "causal") == L * (L + 1) // 2
    assert bench.allowed_pairs(L, L, "causal_bottom_right") == L * (L + 1) // 2
    # bottom-right with Lk = Lq + d: every row sees d more keys than in the square case
    assert bench.allowed_pairs(100, 130, "causal_bottom_right") == 100 * 101 // 2 + 100 * 30


def test_kernel_matmul_flops_follow_the_convention():
    w = synth.WORKLOADS[5]
    # 4 B H L^2 D forward, halved when causal; 2.5x that in the backward
    assert w.flops_fwd() == pytest.approx(4 * 2 * 32 * 8192 ** 2 * 128 / 2)
    assert bench.kernel_matmul_flops("accel_fwd", w) == pytest.approx(w.flops_fwd())
    assert bench.kernel_matmul_flops("accel_dkdv_dq", w) == pytest.approx(2.5 * w.flops_fwd())
    assert bench.kernel_matmul_flops("strict_dkdv_dq", w) == pytest.approx(2.5 * w.flops_fwd())
    assert bench.kernel_matmul_flops("dvec", w) is None


def test_job_tflops():
    # 2 ranks x 10 steps x 3.85 PFLOP in 45 ms (the slowest rank)
    v = bench.job_tflops(3.85e15, 10, 45.0, 2)
    assert v == pytest.approx(2 * 10 * 3.85e15 / 0.045 / 1e12)
    assert np.isfinite(v)
