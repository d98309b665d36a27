"""The allocation-free dispatch entry point, moe_dispatch_noalloc.

It serves callers that cannot call cudaMalloc (their device memory belongs to
another allocator, or cudaMalloc's implicit synchronisation is not allowed on
their path).  Its scratch is a fixed array inside the library, shared by every
call and never freed, so these tests check that calls in a row, on different
routings, each give exactly what the oracle's dispatch and the allocating path
(moe_route) give: the array must be cleared by every call.  This file is
collected last so that a failure here cannot hide the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gemm_gb300 import binding, synth


def test_rejects_sizes_beyond_its_fixed_scratch():
    lib = binding.load()
    # 600 experts do not fit the 512-entry array: refused before any device work
    assert lib.moe_dispatch_noalloc(None, 0, 600, 8, 1, ctypes.c_void_p(16), None, None) == \
        binding.MOE_ERR_UNSUPPORTED
    assert lib.moe_dispatch_noalloc(None, 4, 16, 2, 1, None, None, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_noalloc(None, 0, 16, 17, 1, ctypes.c_void_p(16), None, None) == \
        binding.MOE_ERR_INVALID_ARG


def random_routing(T, E, k, seed):
    """k distinct experts per token, uniformly at random."""
    rng = np.random.default_rng(seed)
    if T == 0:
        return np.zeros((0, k), np.int32)
    return np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)


def noalloc(idx_h, E, k, has_shared, dev):
    T = idx_h.shape[0]
    idx = torch.from_numpy(idx_h).to(dev) if T else torch.zeros((1, k), dtype=torch.int32, device=dev)
    off = torch.full((E + 2,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((max(1, T * k),), -1, dtype=torch.int32, device=dev)
    binding.moe_dispatch_noalloc(idx, T, E, k, has_shared, off, perm)
    torch.cuda.synchronize()
    return off.cpu().numpy(), perm.cpu().numpy()[:T * k]


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
        # and the oracle's dispatch of the same routing
        _, o_off, o_perm = oracle.dispatch(idx.cpu().numpy(), shape.E)
        np.testing.assert_array_equal(off2.cpu().numpy(), o_off)
        np.testing.assert_array_equal(perm2.cpu().numpy(), o_perm)
    layer.close()


@pytest.mark.gpu
@pytest.mark.parametrize("T,E,k,has_shared", [
    (0, 16, 2, 1),       # no tokens: offsets all zero
    (1, 16, 2, 1),
    (1025, 40, 6, 1),
    (128, 288, 8, 1),    # the flash shape's decode batch
    (8192, 288, 8, 1),   # and its prefill chunk
    (300, 24, 8, 0),     # without the shared expert
])
def test_matches_the_oracle_dispatch(T, E, k, has_shared):
    dev = torch.device("cuda:0")
    for call, seed in enumerate((T + E, T + E + 1)):  # two calls in a row
        idx_h = random_routing(T, E, k, seed)
        off, perm = noalloc(idx_h, E, k, has_shared, dev)
        _, o_off, o_perm = oracle.dispatch(idx_h, E)
        np.testing.assert_array_equal(off[:E + 1], o_off[:E + 1])
        assert off[E + 1] == o_off[E] + (T if has_shared else 0)
        np.testing.assert_array_equal(perm, o_perm)


@pytest.mark.gpu
def test_ids_outside_the_expert_range_are_skipped():
    # entries -1 and E are not counted, and no perm slot is written for them:
    # the valid entries are dispatched as if the others were absent
    dev = torch.device("cuda:0")
    T, E, k = 200, 16, 2
    idx_h = random_routing(T, E, k, 5)
    idx_h[3, 1] = -1
    idx_h[50, 0] = E
    idx_h[199, 1] = -7
    off, perm = noalloc(idx_h, E, k, 1, dev)
    valid = (idx_h >= 0) & (idx_h < E)
    counts = np.bincount(idx_h[valid], minlength=E)
    np.testing.assert_array_equal(off[:E + 1], np.concatenate([[0], np.cumsum(counts)]))
    n = int(valid.sum())
    # brute force: assignment ids a = t*k + j of the valid entries, by (expert, token)
    want = sorted((int(idx_h[t, j]), t, t * k + j) for t in range(T) for j in range(k) if valid[t, j])
    np.testing.assert_array_equal(perm[:n], [a for _, _, a in want])
    assert np.all(perm[n:] == -1)
