"""The allocation-free dispatch entry point, moe_dispatch_noalloc.

It serves callers that cannot call cudaMalloc (their device memory belongs to
another allocator, or cudaMalloc's implicit synchronisation is not allowed on
their path).  Its scratch is a fixed array inside the library, shared by every
call and never freed, so these tests check that two calls in a row, on
different routings, each give exactly what the allocating path (moe_route)
gives: the array must be cleared by every call.  This file is collected last
so that a failure here cannot hide the other tests.
"""
import ctypes

import pytest
import torch

from expert_routed_ffn_gemm_gb300 import binding, synth


def test_rejects_sizes_beyond_its_fixed_scratch():
    lib = binding.load()
    # 600 experts do not fit the 512-entry array: refused before any device work
    assert lib.moe_dispatch_noalloc(None, 0, 600, 8, 1, ctypes.c_void_p(16), None, None) == \
        binding.MOE_ERR_UNSUPPORTED
    assert lib.moe_dispatch_noalloc(None, 4, 16, 2, 1, None, None, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_noalloc(None, 0, 16, 17, 1, ctypes.c_void_p(16), None, None) == \
        binding.MOE_ERR_INVALID_ARG


@pytest.mark.gpu
def test_two_calls_match_the_allocating_route():
    dev = torch.device("cuda:0")
    shape = synth.LayerShape(T=300, d=256, E=16, k=2, F=128)
    inp = synth.make_inputs(shape, seed=77)
    layer = binding.MoeLayer(inp.w_router.to(dev), inp.w_gate_up.to(dev), inp.w_down.to(dev), shape.k, shape.T)
    batches = [inp.x.to(dev), synth.make_tokens(shape, seed=78, device=dev)]
    for x in batches:  # two calls in a row on different routings
        idx, _, perm, offsets, _ = layer.route(x, with_gap=False)
        off2 = torch.full_like(offsets, -1)
        perm2 = torch.full_like(perm, -1)
        binding.moe_dispatch_noalloc(idx, shape.T, shape.E, shape.k, True, off2, perm2)
        torch.cuda.synchronize()
        assert torch.equal(off2, offsets)
        assert torch.equal(perm2, perm)
    layer.close()
