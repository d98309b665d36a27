"""Per-call routing variants (top-k below the handle's k, renormalised
weights) and the EP-group routing statistics, through the C ABI, against
the CPU oracle.  Same bars as test_parity_gpu.py (see moe_check.py)."""
import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gemm_gb300 import binding, synth

from moe_check import NEAR_TIE, check_output, check_routing, compare, cpu, host_bits, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def layer_of(inp, max_tokens=None, out_fp32=False):
    x, wr, wgu, wd = to_dev(inp, DEV)
    return binding.MoeLayer(wr, wgu, wd, inp.shape.k, max_tokens or inp.shape.T, out_fp32=out_fp32), x


@pytest.mark.parametrize("out_fp32", [False, True])
@pytest.mark.parametrize("kk", [1, 4])
def test_smaller_top_k_per_call(kk, out_fp32):
    # bf16 y: measured max|err|/RMS 2.46e-2 at top-1, one element near 6 RMS
    # where half a bf16 ulp of y alone is 2.0e-2 RMS; fp32 y meets the plain bound
    shape = synth.LayerShape(T=100, d=256, E=32, k=8, F=128)
    inp = synth.make_inputs(shape, seed=60 + kk)
    layer, x = layer_of(inp, out_fp32=out_fp32)
    idx, prob, perm, offsets, gap = layer.route(x, top_k=kk)
    y = layer.forward(x, top_k=kk)
    assert layer.check() == binding.MOE_OK
    xb, wr, wgu, wd = host_bits(inp)
    slack = not out_fp32
    check_routing(xb, wr, kk, cpu(idx), cpu(prob), cpu(gap), cpu(perm), cpu(offsets))
    check_output(xb, wr, wgu, wd, kk, cpu(y.float()), cpu(idx), out_bf16=not out_fp32, storage_slack=slack)
    # the default call still routes to the handle's k
    y8 = layer.forward(x)
    idx8, _, _, _, _ = layer.route(x)
    check_output(xb, wr, wgu, wd, 8, cpu(y8.float()), cpu(idx8), out_bf16=not out_fp32, storage_slack=slack)
    layer.close()


@pytest.mark.parametrize("kk,T", [(2, 120), (8, 120), (4, 1100), (4, 6000)])
def test_renormalized_weights(kk, T):
    # T = 1100: the one-warp-per-token top-k kernel (1024 tokens and more)
    shape = synth.LayerShape(T=T, d=256, E=32, k=8, F=128)
    inp = synth.make_inputs(shape, seed=70 + kk)
    layer, x = layer_of(inp)
    idx, prob, perm, offsets, gap = layer.route(x, top_k=kk, renormalize=True)
    y = layer.forward(x, top_k=kk, renormalize=True)
    assert layer.check() == binding.MOE_OK
    xb, wr, wgu, wd = host_bits(inp)
    idx_h, prob_h = cpu(idx), cpu(prob).astype(np.float64)
    o_idx, o_w, o_gap, o_p = oracle.route(xb, wr, kk, want_p=True)
    sure = o_gap >= NEAR_TIE
    np.testing.assert_array_equal(idx_h[sure], o_idx[sure])
    sel_p = o_p[np.arange(shape.T)[:, None], idx_h]
    want = sel_p / sel_p.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(prob_h, want, rtol=2e-5, atol=1e-7)
    np.testing.assert_allclose(prob_h.sum(axis=1), 1.0, rtol=0, atol=1e-5)
    y_ref = oracle.forward(xb, wr, wgu, wd, kk, sel=idx_h, renormalize=True)
    # bf16 y: measured max|err|/RMS 2.55e-2 at 6000 tokens, four elements near
    # 6 RMS where half a bf16 ulp of y alone is 2.0e-2 RMS
    compare(cpu(y.float()), y_ref, storage_slack=True)
    layer.close()


def test_flash_decode_top4_renormalized(flash_small_weights):
    inp = flash_small_weights
    layer, x = layer_of(inp)
    y = layer.forward(x, top_k=4, renormalize=True)
    idx, prob, _, _, _ = layer.route(x, top_k=4, renormalize=True)
    assert layer.check() == binding.MOE_OK
    xb, wr, wgu, wd = host_bits(inp)
    y_ref = oracle.forward(xb, wr, wgu, wd, 4, sel=cpu(idx), renormalize=True)
    compare(cpu(y.float()), y_ref)
    layer.close()


@pytest.fixture(scope="module")
def flash_small_weights():
    # d=4096, 288 routed + 1 shared, top-8, width 1280; a decode batch of 64
    return synth.make_inputs(synth.FLASH_DECODE.with_tokens(64), seed=5, device=DEV)


@pytest.mark.parametrize("case", ["tiny", "tiny_many_tokens", "tiny_256_tiles", "flash"])
def test_route_stats_match_oracle(case, flash_small_weights):
    if case.startswith("tiny"):
        # 1500 and 6000 tokens: the one-warp-per-token top-k kernel writes the
        # statistics (6000: 256-token router tiles)
        T = {"tiny": 300, "tiny_many_tokens": 1500, "tiny_256_tiles": 6000}[case]
        inp = synth.make_inputs(synth.LayerShape(T=T, d=256, E=16, k=2, F=128), seed=80)
        G = 4
    else:
        inp = flash_small_weights
        G = 8
    layer, x = layer_of(inp)
    counts, gf, gp, summary = layer.route_stats(x, G)
    assert layer.check() == binding.MOE_OK
    xb, wr, _, _ = host_bits(inp)
    o_counts, o_f, o_p, o_sum = oracle.route_stats(xb, wr, inp.shape.k, G)
    _, _, o_gap, _ = oracle.route(xb, wr, inp.shape.k)
    c = cpu(counts)
    if np.all(o_gap >= NEAR_TIE):
        np.testing.assert_array_equal(c, o_counts)
    T, k, E = inp.shape.T, inp.shape.k, inp.shape.E
    # group shares and the load figures follow from the GPU's own counts exactly
    per = E // G
    f_from_c = np.array([c[g * per:(g + 1) * per].sum() for g in range(G)]) / (T * k)
    np.testing.assert_allclose(cpu(gf), f_from_c, rtol=1e-6)
    np.testing.assert_allclose(cpu(gp), o_p, rtol=1e-5, atol=1e-7)
    s = cpu(summary).astype(np.float64)
    np.testing.assert_allclose(s[0], G * (f_from_c * o_p).sum(), rtol=1e-5)
    np.testing.assert_allclose(s[1], c.max() / (T * k / E), rtol=1e-6)
    np.testing.assert_allclose(s[2], o_sum[2], rtol=1e-5)
    assert s[3] == (c == 0).sum()
    # deterministic run to run
    again = layer.route_stats(x, G)
    for u, v in zip((counts, gf, gp, summary), again):
        assert torch.equal(u, v)
    layer.close()


def test_bad_options_are_rejected():
    inp = synth.make_inputs(synth.TINY, seed=90)
    layer, x = layer_of(inp)
    with pytest.raises(binding.MoeError) as e:
        layer.forward(x, top_k=3)  # the handle's top_k is 2
    assert e.value.status == binding.MOE_ERR_INVALID_ARG
    with pytest.raises(binding.MoeError) as e:
        layer.route_stats(x, 5)  # 5 does not divide 16 experts
    assert e.value.status == binding.MOE_ERR_INVALID_ARG
    assert layer.check() == binding.MOE_OK
    layer.close()
