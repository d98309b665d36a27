"""bench.py's host-side arithmetic (no GPU): the algorithmic bytes and FLOPs
its roofline lines use, and the DRAM-traffic figures it reads from the
committed profile summaries."""
import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from expert_routed_ffn_gemm_gb300 import synth  # noqa: E402


def args_for(**kw):
    a = argparse.Namespace(workload="decode", experts=0, ffn_width=0, weights="bf16")
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_decode_bytes_and_flops():
    shape = synth.FLASH_DECODE
    d, F, E, T, k = shape.d, shape.F, shape.E, shape.T, shape.k
    # 281 routed experts touched + the shared one, bf16 weights: 3 d F 2 bytes each
    b = bench.algorithmic_bytes(shape, 281)
    assert b == 282 * 3 * d * F * 2 + E * d * 4 + T * d * 2 * 2
    assert 8.8e9 < b < 8.9e9
    b8 = bench.algorithmic_bytes(shape, 281, fp8=True)
    assert b8 == 282 * (3 * d * F + (2 * F + d) * 4) + E * d * 4 + T * d * 2 * 2
    rows = T * k + T
    assert bench.gateup_bytes(shape, 281) == 282 * 2 * F * d * 2 + rows * d * 2 + rows * F * 2
    assert bench.gateup_flops(shape) == 2 * rows * d * 2 * F
    assert bench.layer_flops(shape) == T * ((k + 1) * 6 * d * F + 2 * d * E)


def test_traffic_comes_from_the_profiles():
    t = bench.measured_traffic(args_for())
    t8 = bench.measured_traffic(args_for(weights="fp8"))
    assert t is not None and 5.9e9 < t < 6.0e9
    assert t8 is not None and 2.95e9 < t8 < 3.05e9
    assert bench.measured_traffic(args_for(workload="prefill")) is None
    assert bench.measured_traffic(args_for(experts=32)) is None
    assert bench.measured_traffic(args_for(ffn_width=128)) is None


def test_workloads_resolve():
    for name in ("decode", "prefill", "skew", "T=32"):
        shape, _ = bench.workload(name)
        assert shape.d == 4096 and shape.E == 288
    shape, _ = bench.workload("prefill", experts=32, ffn_width=128)
    assert shape.E == 32 and shape.F == 128 and shape.T == 8192


def test_clock_window_and_summary():
    # Samples before the timed region are dropped, the first one after it is
    # kept; throttle reasons are collected and the median taken under load.
    clk = bench.ClockSampler(0)
    row = "0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, {thermal}, Active"
    clk.lines = [(0.9, row.format(sm=345, thermal="Not Active")),
                 (1.01, row.format(sm=2070, thermal="Not Active")),
                 (1.03, row.format(sm=2055, thermal="Active")),
                 (1.05, row.format(sm=2070, thermal="Not Active")),
                 (1.07, row.format(sm=1000, thermal="Not Active"))]
    clk.t0, clk.t1 = 1.0, 1.04
    s = clk.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    clk.t0 = clk.t1 = None  # unmarked: every sample
    assert clk.summary()["samples"] == 5
    assert bench.ClockSampler(0).summary()["reasons"] == ["unsampled"]
