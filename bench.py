"""Benchmark of the sparse-MoE layer (Step 3.5 Flash shape) on GB300.

One step = one moe_forward over one batch of synthetic tokens: router,
softmax/top-8, dispatch, the grouped expert GEMMs (288 routed + 1 shared
expert), and the combine.  Default workload: the decode batch, T=128 tokens,
d=4096, 288+1 experts, top-8, expert width 1280 (bf16 weights, 9.09 GB).

Prints one JSON line.  `value` = tokens/s over the timed steps (device time,
CUDA events, inputs resident in HBM); `e2e` = the same through the host-buffer
entry point (pinned host x in, host y out, copies inside the timed region);
`roofline` = the gate/up grouped GEMM (the dominant kernel) against its binding
roof (HBM copy bandwidth, or the burst bf16 tensor rate for these passes of a
few milliseconds; the sustained rate is reported beside it), its time from a
second pass of the same steps with per-stage events; `routing` = the
per-expert load of the batch (moe_route_stats) and its near-ties;
`cpu_baseline` = the CPU oracle on a bounded sample of the same workload, on
one thread and on every host core.  With the default decode workload the line
also carries `prefill` (T=8192) and `skew` (Zipf-skewed routing, T=4096):
the same measurements on the same weights, nested.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--workload decode|prefill|skew|T=<n>] [--weights bf16|fp8]
                  [--experts E] [--ffn-width F] [--no-cpu-baseline] [--no-nested]

Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of
the layer on its own batch (weak scaling, no data-path collective); the
time is the max over ranks and `value` counts every rank's tokens.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "MoE-layer tokens/s at 1 GB300 (d=4096,E=288,top-8) and % of HBM/tensor roofline"
N_X_BUFFERS = 4  # distinct token batches cycled through the timed steps


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def workload(name: str, experts: int = 0, ffn_width: int = 0):
    """(shape, skew) of a named workload; `experts` > 0 replaces E and
    `ffn_width` > 0 replaces F (smaller cases of the same kernels, e.g. for
    profiler captures of the routing, gather and combine kernels)."""
    from dataclasses import replace

    from expert_routed_ffn_gemm_gb300 import synth

    if name == "decode":
        shape, skew = synth.FLASH_DECODE, None
    elif name == "prefill":
        shape, skew = synth.FLASH_PREFILL, None
    elif name == "skew":
        shape, skew = synth.FLASH_SKEW, "zipf"
    elif name.startswith("T="):
        shape, skew = synth.FLASH_DECODE.with_tokens(int(name[2:])), None
    else:
        raise SystemExit(f"unknown workload {name}")
    if experts > 0:
        shape = replace(shape, E=experts)
    if ffn_width > 0:
        shape = replace(shape, F=ffn_width)
    return shape, skew


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms by a
    background nvidia-smi whose lines a reader thread timestamps.  Entering
    waits (up to 5 s) for the first sample, so the sampler is running before
    the timed region starts; mark_start() / mark_end() bracket the timed
    region, and summary() keeps the samples taken inside it plus the first
    one after it, which covers its last interval: its throttle reasons count,
    but its clock only when the region holds no sample (the GPU idles while
    the sampler stops, so that sample's clock can be an idle one)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []  # (time.perf_counter(), line)
        self.t0 = self.t1 = None
        self._reader = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line))

    def __enter__(self):
        import threading

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()
        deadline = time.perf_counter() + 5.0
        while not self.lines and time.perf_counter() < deadline and self.proc.poll() is None:
            time.sleep(0.005)
        return self

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(2 * self.INTERVAL_MS / 1000.0)  # the sample that covers the end of the region
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self._reader is not None:
                self._reader.join(timeout=5)

    def window(self):
        """The timed region's sampled lines as (line, its clock counts) pairs
        (every line, counted, if the region was not marked)."""
        if self.t0 is None or self.t1 is None:
            return [(l, True) for _, l in self.lines]
        inside = [l for t, l in self.lines if self.t0 <= t <= self.t1]
        after = [l for t, l in self.lines if t > self.t1][:1]
        return [(l, True) for l in inside] + [(l, not inside) for l in after]

    def summary(self):
        lines = self.window()
        if not lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line, clock_counts in lines:
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                clock, smax = float(f[1]), float(f[2])
            except ValueError:
                continue
            if clock_counts:
                sm.append(clock)
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        load = [v for v in sm if smax and v > 0.3 * smax] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "interval_ms": self.INTERVAL_MS}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist

    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, steps: int, elapsed_s_per_rank: float, world: int) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    slowest = max_over_ranks(elapsed_s_per_rank, world)
    return tokens_per_rank * steps * world / slowest


def algorithmic_bytes(shape, touched: int, fp8: bool = False):
    """Bytes the layer must move: the weights of every expert group with at
    least one row (routed experts touched + the shared expert; fp8: one byte
    per weight plus a 4-byte scale per weight row), the router weights, x in
    and y out."""
    d, F, E, T = shape.d, shape.F, shape.E, shape.T
    per_group = 3 * d * F + (2 * F + d) * 4 if fp8 else 3 * d * F * 2
    return (touched + (1 if shape.has_shared else 0)) * per_group + E * d * 4 + T * d * 2 * 2


def gateup_bytes(shape, touched: int, fp8: bool = False):
    """Algorithmic bytes of one gate/up GEMM launch: W_gu of every group with
    rows (fp8: codes + row scales), the R dispatch-ordered token rows read
    once, H written once."""
    d, F, T, k = shape.d, shape.F, shape.T, shape.k
    groups = touched + (1 if shape.has_shared else 0)
    R = T * k + (T if shape.has_shared else 0)
    w = 2 * F * d + 2 * F * 4 if fp8 else 2 * F * d * 2
    return groups * w + R * d * 2 + R * F * 2


def gateup_flops(shape):
    d, F, T, k = shape.d, shape.F, shape.T, shape.k
    R = T * k + (T if shape.has_shared else 0)
    return 2 * R * d * 2 * F


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def sources_digest(files) -> str:
    """sha256 (first 16 hex digits) over the named kernel sources, in order."""
    import hashlib

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload_name: str, weights: str, shape, gu_alg_bytes: float):
    """DRAM bytes per launch of the gate/up GEMM from the committed ncu
    captures (profiles/traffic.json): (bytes or None, source note).  An entry
    whose kernel sources have changed since the capture gives None.  Each
    entry was captured on a smaller case of the same kernel, with L2 emptied
    before the kernel, and carries the ratio of its traffic to its
    algorithmic bytes; in a layer call the routing kernels have already
    brought the shared expert's weights into L2, so the figure is that ratio
    times this workload's algorithmic bytes without them."""
    try:
        with open(TRAFFIC_FILE) as f:
            entries = json.load(f)["entries"]
    except (OSError, ValueError, KeyError):
        return None, "no capture file"
    for e in entries:
        if e.get("workload") != workload_name or e.get("weights") != weights:
            continue
        if tuple(e.get("shape", ())) != (shape.T, shape.d, shape.E, shape.k, shape.F):
            continue
        try:
            digest = sources_digest(e["sources"])
        except OSError:
            return None, "kernel sources missing"
        if digest != e.get("sources_sha256_16"):
            return None, f"stale: the kernel changed since the capture ({e['capture']})"
        if e.get("traffic_over_algorithmic") is not None:
            shared = shared_weight_bytes(shape, weights == "fp8") if shape.has_shared else 0
            return float(e["traffic_over_algorithmic"]) * (gu_alg_bytes - shared), e["capture"]
    return None, "no capture of this workload"


def shared_weight_bytes(shape, fp8: bool = False) -> int:
    """The shared expert's gate/up weight bytes (codes and row scales for FP8)."""
    return 2 * shape.F * shape.d + 2 * shape.F * 4 if fp8 else 2 * shape.F * shape.d * 2


def layer_flops(shape):
    d, F, E, T, k = shape.d, shape.F, shape.E, shape.T, shape.k
    return T * ((k + (1 if shape.has_shared else 0)) * 6 * d * F + 2 * d * E)


def cpu_oracle_rate(inp_host, shape, budget_s: float, max_tokens: int, fp8=None, threads: int = 0):
    """CPU oracle throughput (tokens/s) on the batch's tokens in order, in
    chunks, cycling through the batch, until `budget_s` seconds are spent or
    `max_tokens` tokens are done.  fp8 = host (q_gate_up, s_gate_up, q_down,
    s_down): the FP8 oracle forward.  threads: OpenMP threads (0 = all).
    Returns (tokens/s, tokens, seconds, threads used)."""
    import numpy as np

    import oracle

    xb, wr, wgu, wd = inp_host
    n, spent, chunk = 0, 0.0, 4
    while spent < budget_s and n < max_tokens:
        m = min(chunk, max_tokens - n)
        toks = ((n + np.arange(m)) % shape.T).astype(np.int32)
        if toks.size == 0:
            break
        t0 = time.perf_counter()
        if fp8 is None:
            oracle.forward(xb, wr, wgu, wd, shape.k, has_shared=shape.has_shared, tokens=toks, threads=threads)
        else:
            oracle.forward_fp8(xb, wr, *fp8, shape.k, has_shared=shape.has_shared, tokens=toks, threads=threads)
        spent += time.perf_counter() - t0
        n += toks.size
        chunk = min(64, chunk * 2)
    return n / spent, n, spent, (threads if threads > 0 else oracle.max_threads())


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip() + f" ({platform.machine()})"
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def host_copy(inp):
    from expert_routed_ffn_gemm_gb300 import synth

    return (synth.bf16_bits(inp.x), inp.w_router.detach().cpu().numpy(), synth.bf16_bits(inp.w_gate_up),
            synth.bf16_bits(inp.w_down))


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, timed per step on a
    bounded sample of the workload's tokens."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from expert_routed_ffn_gemm_gb300 import synth

    shape, skew = workload(args.workload, args.experts, args.ffn_width)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.make_inputs(shape, seed=0, device=dev, skew=skew)
    xb, wr, wgu, wd = host_copy(inp)
    del inp
    sample = min(shape.T, args.ref_tokens)
    for _ in range(args.warmup):
        oracle.forward(xb, wr, wgu, wd, shape.k, tokens=np.arange(min(2, sample), dtype=np.int32))
    t0 = time.perf_counter()
    for s in range(args.steps):
        start = (s * sample) % shape.T
        toks = (np.arange(sample) + start) % shape.T
        oracle.forward(xb, wr, wgu, wd, shape.k, tokens=toks.astype(np.int32))
    el = time.perf_counter() - t0
    tok_s = sample * args.steps / el
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02) weights)",
        "config": {"workload": f"{args.workload}: T={shape.T}, d={shape.d}, E={shape.E}+1, k={shape.k}, "
                               f"F={shape.F}", "tokens_per_step_sampled": sample},
        "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} tokens of the T={shape.T} batch per step", "cpu_model": cpu_model()},
        "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


GATEUP_KERNEL = {
    "bf16": "gate_up_gemm (tcgen05 grouped GEMM, fused SiLU gate)",
    "fp8": "gate_up_gemm (tcgen05 kind::f8f6f4 grouped GEMM on E4M3 weights and two-term E4M3 token rows, "
           "fused SiLU gate)",
}


def routing_report(layer, x, shape, n_groups: int = 8):
    """Per-expert load of one batch from moe_route_stats (max/mean load,
    experts without rows, EP-group balance L_EP over n_groups groups of
    consecutive experts, mean router entropy) and the tokens whose k-th and
    (k+1)-th probabilities differ by less than 1e-6 (near-ties, from the
    GPU's own gap)."""
    import numpy as np

    g = n_groups if shape.E % n_groups == 0 else 1
    counts, _, _, summary = layer.route_stats(x, g)
    _, _, _, _, gap = layer.route(x, with_gap=True)
    c = counts.cpu().numpy()
    s = summary.cpu().numpy().astype(float)
    gp = gap.float().cpu().numpy()
    return {"max_over_mean_load": float(s[1]), "empty_experts": int(s[3]), "max_rows": int(c.max()),
            "mean_rows": float(c.mean()), "l_ep": float(s[0]), "ep_groups": g, "router_entropy": float(s[2]),
            "near_ties": int(np.count_nonzero(gp < 1e-6))}


def measure(layer, xs, shape, args, fp8, world, local, stream, label):
    """One workload on one handle: the timed pass (step time, no per-stage
    events), the same steps again with per-stage events, the clocks of the
    timed pass, and the roofline figures of the layer and its gate/up GEMM."""
    import numpy as np

    from expert_routed_ffn_gemm_gb300 import binding

    hbm_gbs, tf_burst, tf_sust, peak_kind = peaks()
    y = torch.empty((shape.T, shape.d), dtype=torch.bfloat16, device=xs[0].device)
    # units of work of each batch: routed experts with at least one row
    touched = []
    for x in xs:
        _, _, _, offsets, _ = layer.route(x, with_gap=False)
        off = offsets.cpu().numpy()
        touched.append(int(np.count_nonzero(np.diff(off[:shape.E + 1]))))
    for i in range(args.warmup):
        layer.forward(xs[i % len(xs)], y)
    torch.cuda.synchronize()
    if layer.check() != binding.MOE_OK:
        raise RuntimeError(f"{label}: device error during warm-up")

    # The layer's kernels overlap their launch and set-up with the end of the
    # kernel before them (programmatic dependent launch); events recorded
    # between kernels would serialise them, so the step time is taken without
    # the per-stage events, and the per-stage times in a second timed pass of
    # the same steps with them.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark_start()
        ev0.record(stream)
        launches = 0
        for i in range(args.steps):
            layer.forward(xs[i % len(xs)], y)
            launches += layer.last_kernel_count()
        ev1.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world)
    if layer.check() != binding.MOE_OK:
        raise RuntimeError(f"{label}: device error in the timed region")
    if not torch.isfinite(y.float()).all():
        raise RuntimeError(f"{label}: non-finite output")

    layer.profile_enable(True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(args.steps):
        layer.forward(xs[i % len(xs)], y)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms_staged = ev0.elapsed_time(ev1)
    stages, n_prof = layer.profile_read()
    layer.profile_enable(False)
    if layer.check() != binding.MOE_OK:
        raise RuntimeError(f"{label}: device error in the staged pass")

    steps_prof = max(1, n_prof)
    gu_ms = stages["gate_up_gemm"] / steps_prof
    mean_touched = sum(touched[i % len(xs)] for i in range(args.steps)) / args.steps
    gu_bytes = gateup_bytes(shape, mean_touched, fp8)
    gu_gbs = gu_bytes / (gu_ms / 1e3) / 1e9
    gu_tfs = gateup_flops(shape) / (gu_ms / 1e3) / 1e12
    # the binding roof of the kernel: the larger of its HBM and tensor floors
    # (burst tensor rate: these passes last milliseconds)
    tensor_bound = gateup_flops(shape) / (tf_burst * 1e12) > gu_bytes / (hbm_gbs * 1e9)
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": gu_tfs, "peak": tf_burst, "unit": "TFLOP/s",
                "frac": gu_tfs / tf_burst, "peak_kind": peak_kind + " (burst bf16)"}
    else:
        roof = {"bound": "hbm", "achieved": gu_gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gu_gbs / hbm_gbs,
                "peak_kind": peak_kind + " (copy bandwidth)"}
    wname = "fp8" if fp8 else "bf16"
    traffic, traffic_src = measured_traffic(args.workload if label == "headline" else label, wname, shape, gu_bytes)
    layer_bytes = algorithmic_bytes(shape, mean_touched, fp8)
    step_s = ms_max / 1e3 / args.steps
    return {
        "ms_per_step": ms_max / args.steps,
        "value": shape.T * args.steps * world / (ms_max / 1e3),
        "tokens_per_step_per_gpu": shape.T,
        "experts_touched_mean": mean_touched,
        "roofline": {"kernel": GATEUP_KERNEL[wname], **roof, "traffic": traffic, "traffic_source": traffic_src,
                     "ms_per_launch": gu_ms, "algorithmic_bytes_per_launch": gu_bytes,
                     "flops_per_launch": gateup_flops(shape), "hbm_frac": gu_gbs / hbm_gbs,
                     "tensor_frac_burst": gu_tfs / tf_burst, "tensor_frac_sustained": gu_tfs / tf_sust},
        "layer_roofline": {"hbm_frac": layer_bytes / step_s / 1e9 / hbm_gbs,
                           "tensor_frac_burst": layer_flops(shape) / step_s / 1e12 / tf_burst,
                           "tensor_frac_sustained": layer_flops(shape) / step_s / 1e12 / tf_sust,
                           "bytes_per_step": layer_bytes, "flops_per_step": layer_flops(shape),
                           "peaks": {"hbm_gbs": hbm_gbs, "bf16_tflops_burst": tf_burst,
                                     "bf16_tflops_sustained": tf_sust, "kind": peak_kind}},
        "stage_ms_per_step": {k: v / steps_prof for k, v in stages.items()},
        "ms_per_step_with_stage_events": ms_staged / args.steps,
        "routing": routing_report(layer, xs[0], shape),
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }


def nested_workload(name, inp, q, args, world, rank, local, stream):
    """The prefill or skew workload on the headline's expert weights (a
    second handle borrowing the same tensors), for the nested objects."""
    from expert_routed_ffn_gemm_gb300 import binding, synth

    skew = "zipf" if name == "skew" else None
    shape = synth.FLASH_PREFILL if name == "prefill" else synth.FLASH_SKEW
    dev = inp.w_router.device
    xs = [synth.make_tokens(shape, seed=2000 + 31 * rank + i, device=dev, skew=skew) for i in range(N_X_BUFFERS)]
    wr = synth.skewed_router(inp.w_router, seed=rank) if skew else inp.w_router
    if q is not None:
        layer = binding.MoeLayer.fp8(wr, *q, shape.k, shape.T)
    else:
        layer = binding.MoeLayer(wr, inp.w_gate_up, inp.w_down, shape.k, shape.T)
    try:
        out = measure(layer, xs, shape, args, q is not None, world, local, stream, name)
    finally:
        layer.close()
    out["workload"] = (f"{name}: T={shape.T} tokens, d={shape.d}, E={shape.E} routed + 1 shared, top-{shape.k}, "
                       f"expert width {shape.F}" + (", Zipf-skewed router bias (40 experts never chosen)"
                                                    if skew else ""))
    return out


def run_native(args, world, rank, local):
    from expert_routed_ffn_gemm_gb300 import binding, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape, skew = workload(args.workload, args.experts, args.ffn_width)

    inp = synth.make_inputs(shape, seed=rank, device=dev, skew=skew)
    xs = [inp.x] + [synth.make_tokens(shape, seed=1000 + 31 * rank + i, device=dev, skew=skew)
                    for i in range(N_X_BUFFERS - 1)]
    fp8 = args.weights == "fp8"
    q = None
    if fp8:
        # E4M3 codes + row scales of the same synthetic weights, made on the device
        q_gu, s_gu = binding.moe_quantize_fp8(inp.w_gate_up)
        q_d, s_d = binding.moe_quantize_fp8(inp.w_down)
        q = (q_gu, s_gu, q_d, s_d)
        inp.w_gate_up = inp.w_down = None
        torch.cuda.synchronize()
        layer = binding.MoeLayer.fp8(inp.w_router, q_gu, s_gu, q_d, s_d, shape.k, shape.T)
    else:
        layer = binding.MoeLayer(inp.w_router, inp.w_gate_up, inp.w_down, shape.k, shape.T)
    stream = torch.cuda.current_stream(dev)

    head = measure(layer, xs, shape, args, fp8, world, local, stream, "headline")

    # ---- end to end through the host-buffer entry point ---------------------
    x_host = [x.cpu().pin_memory() for x in xs]
    y_host = torch.empty((shape.T, shape.d), dtype=torch.bfloat16).pin_memory()
    for i in range(2):
        layer.forward_host(x_host[i % N_X_BUFFERS], y_host)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(args.steps):
        layer.forward_host(x_host[i % N_X_BUFFERS], y_host)
    e2e_s = time.perf_counter() - t0
    barrier(world)
    e2e = aggregate(shape.T, args.steps, e2e_s, world)
    layer.close()

    layer_bytes = head["layer_roofline"]["bytes_per_step"]
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3-weights/bf16-x" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) bf16 tokens, N(0,0.02) weights, random init)",
        "config": {
            "workload": f"{args.workload}: T={shape.T} tokens, d={shape.d}, E={shape.E} routed + 1 shared, "
                        f"top-{shape.k}, expert width {shape.F}, SiLU-gated"
                        + (", E4M3 expert weights with fp32 row scales" if fp8 else ""),
            "tokens_per_step_per_gpu": shape.T,
            "l2": f"inputs larger than L2: {layer_bytes / 1e9:.2f} GB of expert weights read per step; "
                  f"{N_X_BUFFERS} token batches cycled",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "experts_touched_mean": head["experts_touched_mean"],
        },
        "roofline": head["roofline"],
        "layer_roofline": head["layer_roofline"],
        "stage_ms_per_step": head["stage_ms_per_step"],
        "ms_per_step_with_stage_events": head["ms_per_step_with_stage_events"],
        "routing": head["routing"],
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": shape.T * shape.d * 2,
                "d2h_bytes_per_step": shape.T * shape.d * 2},
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }

    # ---- the prefill chunk and the skewed batch on the same weights ---------
    if args.workload == "decode" and not args.no_nested and not args.experts and not args.ffn_width:
        for name in ("prefill", "skew"):
            line[name] = nested_workload(name, inp, q, args, world, rank, local, stream)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if fp8:
            inp_host = (synth.bf16_bits(inp.x), inp.w_router.detach().cpu().numpy(), None, None)
            fp8_host = tuple(t.cpu().numpy() for t in q)
        else:
            inp_host, fp8_host = host_copy(inp), None
        budget = args.cpu_budget / 2
        rate, n, spent, cores = cpu_oracle_rate(inp_host, shape, budget_s=budget,
                                                max_tokens=max(shape.T, 16 * 1024), fp8=fp8_host)
        rate1, n1, spent1, _ = cpu_oracle_rate(inp_host, shape, budget_s=budget, max_tokens=max(shape.T, 1024),
                                               fp8=fp8_host, threads=1)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{n} tokens of the T={shape.T} batch, in order and cycled "
                                          f"({spent:.1f} s on {cores} threads)",
                                "cpu_model": cpu_model(),
                                "one_thread": {"value": rate1, "unit": "tokens/s", "cores": 1,
                                               "sample": f"{n1} tokens of the same batch ({spent1:.1f} s)"}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--experts", type=int, default=0, help="override the routed expert count (smaller cases)")
    ap.add_argument("--ffn-width", type=int, default=0, help="override the expert width F, a multiple of 128 (smaller cases)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-nested", action="store_true", help="decode only: leave out the nested prefill and skew runs")
    ap.add_argument("--weights", choices=["bf16", "fp8"], default="bf16",
                    help="expert weight format (fp8: E4M3 codes with fp32 row scales)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        import __graft_entry__

        if rank == 0 or world == 1:
            __graft_entry__.build()
        barrier(world)
        run_native(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
