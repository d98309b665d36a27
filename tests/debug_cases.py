"""Layer calls run in a process that loaded libmoe_debug.so (the build whose
kernels check every index they take from the dispatch; see kernels.cuh), each
checked against the oracle; run by test_debug_build_gpu.py with
MOE_LIBRARY=debug.  Prints one line per case and exits non-zero on the first
failure."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from expert_routed_ffn_gemm_gb300 import binding, synth  # noqa: E402

from moe_check import check_output, check_routing, cpu, host_bits, sample_tokens  # noqa: E402

DEV = torch.device("cuda:0")


def case(shape, seed, tiles=(0, 0), env=None, n_sample=None, fp8=False):
    inp = synth.make_inputs(shape, seed=seed, device=DEV)
    old = {k: os.environ.get(k) for k in ("MOE_TILE_N_GATEUP", "MOE_TILE_N_DOWN", "MOE_GEMM_KSPLIT")}
    os.environ["MOE_TILE_N_GATEUP"], os.environ["MOE_TILE_N_DOWN"] = str(tiles[0]), str(tiles[1])
    os.environ.update(env or {})
    try:
        if fp8:
            q = binding.moe_quantize_fp8(inp.w_gate_up) + binding.moe_quantize_fp8(inp.w_down)
            layer = binding.MoeLayer.fp8(inp.w_router, *q, shape.k, shape.T, has_shared=shape.has_shared,
                                         out_fp32=True)
        else:
            layer = binding.MoeLayer(inp.w_router, inp.w_gate_up, inp.w_down, shape.k, shape.T,
                                     has_shared=shape.has_shared, out_fp32=True)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    idx, prob, perm, offsets, gap = layer.route(inp.x)
    y = layer.forward(inp.x)
    rc = layer.check()
    assert rc == binding.MOE_OK, f"device error word set: {binding.moe_status_string(rc)}"
    xb, wr, wgu, wd = host_bits(inp)
    idx_h = cpu(idx)
    near, _ = check_routing(xb, wr, shape.k, idx_h, cpu(prob), cpu(gap), cpu(perm), cpu(offsets),
                            has_shared=shape.has_shared)
    tokens = np.arange(shape.T, dtype=np.int32) if n_sample is None else sample_tokens(shape.T, idx_h, n_sample, seed,
                                                                                      near)
    fp8_h = tuple(cpu(t) for t in q) if fp8 else None
    ratio = check_output(xb, wr, wgu, wd, shape.k, cpu(y.float())[tokens], idx_h, tokens=tokens,
                         has_shared=shape.has_shared, out_bf16=False, fp8=fp8_h)
    layer.close()
    return ratio


def main():
    assert binding.library_path().endswith("libmoe_debug.so"), binding.library_path()
    S = synth.LayerShape
    cases = [
        ("tiny", lambda: case(synth.TINY, 1)),
        ("16-row tiles, ragged", lambda: case(S(T=300, d=256, E=16, k=2, F=128), 2, tiles=(16, 16))),
        ("256-row tiles on CTA pairs, ragged", lambda: case(S(T=300, d=256, E=16, k=2, F=128), 3, tiles=(256, 256))),
        ("chunked dispatch, 9-term combine", lambda: case(S(T=1500, d=256, E=32, k=8, F=128), 4, n_sample=96)),
        ("pairs over many tokens", lambda: case(S(T=5000, d=256, E=16, k=2, F=128), 5, n_sample=64)),
        ("K split in 3 parts", lambda: case(S(T=3, d=512, E=16, k=2, F=256), 6, tiles=(16, 32),
                                            env={"MOE_GEMM_KSPLIT": "3"})),
        ("K split in balanced ranges", lambda: case(S(T=5, d=1024, E=16, k=2, F=384), 8, tiles=(32, 32),
                                                    env={"MOE_GEMM_KSPLIT": "b"})),
        ("FP8 two-term rows", lambda: case(S(T=600, d=512, E=24, k=2, F=256), 7, fp8=True, n_sample=64)),
        # no shared expert: k terms per token in the combine, no shared group
        ("no shared expert, generic combine", lambda: case(S(T=50, d=256, E=12, k=3, F=128, has_shared=False), 9)),
        ("no shared expert, FP8", lambda: case(S(T=70, d=256, E=12, k=3, F=128, has_shared=False), 10, fp8=True)),
    ]
    for name, run in cases:
        r = run()
        print(f"ok  {name}: max|err|/RMS {r:.3e}", flush=True)


if __name__ == "__main__":
    main()
