"""bench.py's host-side arithmetic (no GPU): the algorithmic bytes and FLOPs
its roofline lines use, and the DRAM-traffic figures it reads from the
committed capture file (profiles/traffic.json)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from expert_routed_ffn_gemm_gb300 import synth  # noqa: E402


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


def _capture_file(tmp_path, monkeypatch, fresh: bool):
    """The committed capture file with its source digests set as if the
    kernels were (fresh) or were not (stale) the ones captured."""
    import json
    doc = json.load(open(bench.TRAFFIC_FILE))
    for e in doc["entries"]:
        e["sources_sha256_16"] = bench.sources_digest(e["sources"]) if fresh else "0" * 16
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(doc))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))


def test_traffic_comes_from_the_profiles(tmp_path, monkeypatch):
    _capture_file(tmp_path, monkeypatch, fresh=True)
    dec = synth.FLASH_DECODE
    alg = bench.gateup_bytes(dec, 281)
    t, src = bench.measured_traffic("decode", "bf16", dec, alg)
    t8, _ = bench.measured_traffic("decode", "fp8", dec, bench.gateup_bytes(dec, 281, fp8=True))
    assert t is not None and 5.85e9 < t < 6.0e9 and src.startswith("ncu ")
    assert t8 is not None and 2.9e9 < t8 < 3.1e9
    # the prefill entry was captured on a smaller case and scales with the
    # algorithmic bytes of the workload
    pre = synth.FLASH_PREFILL
    alg_p = bench.gateup_bytes(pre, 288)
    tp, _ = bench.measured_traffic("prefill", "bf16", pre, alg_p)
    assert tp is not None and 1.0 <= tp / alg_p < 1.05
    # workloads or shapes without a capture
    assert bench.measured_traffic("skew", "bf16", synth.FLASH_SKEW, 1.0)[0] is None
    from dataclasses import replace
    assert bench.measured_traffic("decode", "bf16", replace(dec, E=32), alg)[0] is None


def test_stale_capture_gives_no_traffic(tmp_path, monkeypatch):
    _capture_file(tmp_path, monkeypatch, fresh=False)
    t, src = bench.measured_traffic("decode", "bf16", synth.FLASH_DECODE, 1.0)
    assert t is None and src.startswith("stale")


def test_committed_captures_name_existing_sources():
    import json
    for e in json.load(open(bench.TRAFFIC_FILE))["entries"]:
        assert e["capture"].startswith("ncu ") and "--clock-control none" in e["capture"]
        bench.sources_digest(e["sources"])  # every file exists


def test_workloads_resolve():
    for name in ("decode", "prefill", "skew", "T=32"):
        shape, _ = bench.workload(name)
        assert shape.d == 4096 and shape.E == 288
    shape, _ = bench.workload("prefill", experts=32, ffn_width=128)
    assert shape.E == 32 and shape.F == 128 and shape.T == 8192


def test_clock_window_and_summary():
    # Samples before the timed region are dropped; the first one after it
    # adds its throttle reasons, and its clock only when the region holds no
    # sample; the median is taken under load.
    clk = bench.ClockSampler(0)
    row = "0, {sm}, 2070, 900.0, 0x0, {hw}, Not Active, {thermal}, Active"
    clk.lines = [(0.9, row.format(sm=345, hw="Not Active", thermal="Not Active")),
                 (1.01, row.format(sm=2070, hw="Not Active", thermal="Not Active")),
                 (1.02, row.format(sm=2070, hw="Not Active", thermal="Not Active")),
                 (1.03, row.format(sm=2055, hw="Not Active", thermal="Active")),
                 (1.05, row.format(sm=1500, hw="Active", thermal="Not Active")),
                 (1.07, row.format(sm=1000, hw="Not Active", thermal="Not Active"))]
    clk.t0, clk.t1 = 1.0, 1.04
    s = clk.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    clk.t0, clk.t1 = 1.035, 1.04  # no sample inside: the one after it
    s = clk.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 1500.0
    clk.t0 = clk.t1 = None  # unmarked: every sample
    assert clk.summary()["samples"] == 6
    assert bench.ClockSampler(0).summary()["reasons"] == ["unsampled"]
