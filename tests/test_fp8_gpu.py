"""FP8 expert weights on the GPU (moe_quantize_fp8, moe_init_fp8 + the
forward) against the oracle: codes and scales bit-exact, routing as in the
bf16 path, the layer output within the same bound (see moe_check.py) of the
oracle's forward on the same E4M3 weights ("Step3.5 Flash 大模型技术深度解析"
§8.1, FP8/FP16 mixed-precision inference)."""
import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gemm_gb300 import binding, synth

from moe_check import check_output, check_routing, compare, cpu, sample_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def quantised(inp):
    """Device E4M3 codes and scales of the synthetic bf16 expert weights."""
    q_gu, s_gu = binding.moe_quantize_fp8(inp.w_gate_up.to(DEV))
    q_d, s_d = binding.moe_quantize_fp8(inp.w_down.to(DEV))
    torch.cuda.synchronize()
    return q_gu, s_gu, q_d, s_d


def test_quantiser_bit_exact():
    rng = np.random.default_rng(5)
    w = rng.normal(0, 0.02, (300, 384)).astype(np.float32)
    w[7] = 0.0
    w[9, :5] = [3.0, -500.0, 1e-6, -1e-9, 0.0]
    w[11] *= 1e-4
    wb = torch.from_numpy(w).to(torch.bfloat16)
    q, s = binding.moe_quantize_fp8(wb.to(DEV))
    oq, os_ = oracle.quantize_e4m3(synth.bf16_bits(wb))
    np.testing.assert_array_equal(cpu(s), os_)
    np.testing.assert_array_equal(cpu(q), oq)


def fp8_case(shape, seed, tiles=(0, 0), n_sample=None, max_tokens=None, out_fp32=False, x2=True, ksplit=None,
             storage_slack=False):
    """x2: the gate/up GEMM on E4M3 tensor cores with the token rows as two
    E4M3 terms (the default), or on fp16 tensor cores with the weights widened
    (MOE_FP8_X2=0).  ksplit: K parts forced on the expert GEMMs (None: by
    work items).  storage_slack: see moe_check.check_output."""
    import os
    inp = synth.make_inputs(shape, seed=seed, device=DEV)
    q_gu, s_gu, q_d, s_d = quantised(inp)
    inp.w_gate_up = inp.w_down = None  # the bf16 copies are not needed any more
    old = {k: os.environ.get(k) for k in ("MOE_TILE_N_GATEUP", "MOE_TILE_N_DOWN", "MOE_FP8_X2", "MOE_GEMM_KSPLIT")}
    os.environ["MOE_TILE_N_GATEUP"], os.environ["MOE_TILE_N_DOWN"] = str(tiles[0]), str(tiles[1])
    os.environ["MOE_FP8_X2"] = "1" if x2 else "0"
    if ksplit is None:
        os.environ.pop("MOE_GEMM_KSPLIT", None)
    else:
        os.environ["MOE_GEMM_KSPLIT"] = str(ksplit)
    try:
        layer = binding.MoeLayer.fp8(inp.w_router, q_gu, s_gu, q_d, s_d, shape.k,
                                     max_tokens or shape.T, has_shared=shape.has_shared, out_fp32=out_fp32)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    x = inp.x
    idx, prob, perm, offsets, gap = layer.route(x)
    y = layer.forward(x)
    assert layer.check() == binding.MOE_OK
    xb = synth.bf16_bits(inp.x)
    wr = cpu(inp.w_router)
    idx_h = cpu(idx)
    near, _ = check_routing(xb, wr, shape.k, idx_h, cpu(prob), cpu(gap), cpu(perm), cpu(offsets),
                            has_shared=shape.has_shared)
    fp8 = (cpu(q_gu), cpu(s_gu), cpu(q_d), cpu(s_d))
    tokens = np.arange(shape.T, dtype=np.int32) if n_sample is None else sample_tokens(shape.T, idx_h, n_sample,
                                                                                      seed, near)
    y_h = cpu(y[torch.from_numpy(tokens).long().to(DEV)].float())
    ratio = check_output(xb, wr, None, None, shape.k, y_h, idx_h, tokens=tokens, has_shared=shape.has_shared,
                         out_bf16=not out_fp32, fp8=fp8, storage_slack=storage_slack)
    y2 = layer.forward(x)
    assert torch.equal(y, y2)
    layer.close()
    return ratio


@pytest.mark.parametrize("out_fp32", [False, True])
@pytest.mark.parametrize("x2", [True, False])
def test_fp8_tiny(x2, out_fp32):
    # bf16 y: measured max|err|/RMS 2.21e-2, one element at 6.1 RMS where half
    # a bf16 ulp of y alone is 2.0e-2 RMS; fp32 y meets the plain bound
    fp8_case(synth.TINY, seed=0, x2=x2, out_fp32=out_fp32, storage_slack=not out_fp32)


@pytest.mark.parametrize("x2", [True, False])
@pytest.mark.parametrize("tiles", [(16, 16), (32, 32), (64, 64), (128, 128), (16, 128), (128, 16), (256, 256)])
def test_fp8_tile_widths_ragged(tiles, x2):
    # 300 tokens, 16 experts, top-2: ragged tiles of every width; d = 512 gives
    # 4 K steps of 128 per gate/up tile (wraps the 4-slot A ring once)
    fp8_case(synth.LayerShape(T=300, d=512, E=16, k=2, F=256), seed=21, tiles=tiles, x2=x2)


@pytest.mark.parametrize("x2", [True, False])
def test_fp8_long_k_and_fp32_output(x2):
    # d = 2048: 16 K steps per gate/up tile (rings wrap several times)
    fp8_case(synth.LayerShape(T=96, d=2048, E=8, k=2, F=256), seed=22, out_fp32=True, x2=x2)


@pytest.mark.parametrize("x2", [True, False])
def test_fp8_without_shared_expert(x2):
    fp8_case(synth.LayerShape(T=50, d=256, E=12, k=3, F=128, has_shared=False), seed=23, x2=x2)


def test_fp8_two_term_rows_with_wide_dynamic_range():
    # token rows whose values span many binades (tiny and huge entries, a zero
    # row): the per-token power-of-two scale and the lo terms below E4M3's
    # normal range must still keep the output within the bound
    shape = synth.LayerShape(T=64, d=256, E=8, k=2, F=128)
    import os
    inp = synth.make_inputs(shape, seed=27, device=DEV)
    inp.x[3] = 0.0
    inp.x[5] *= 1e-6
    inp.x[7, :16] *= 300.0
    inp.x[9, ::3] *= 1e-4
    q_gu, s_gu, q_d, s_d = quantised(inp)
    old = os.environ.get("MOE_FP8_X2")
    os.environ["MOE_FP8_X2"] = "1"
    try:
        layer = binding.MoeLayer.fp8(inp.w_router, q_gu, s_gu, q_d, s_d, shape.k, shape.T)
    finally:
        if old is None:
            os.environ.pop("MOE_FP8_X2", None)
        else:
            os.environ["MOE_FP8_X2"] = old
    y = layer.forward(inp.x)
    assert layer.check() == binding.MOE_OK
    xb = synth.bf16_bits(inp.x)
    wr = cpu(inp.w_router)
    idx, _, _, _, _ = layer.route(inp.x)
    fp8 = (cpu(q_gu), cpu(s_gu), cpu(q_d), cpu(s_d))
    # bf16 y: rows scaled by 300 put y at up to 16 RMS, where half a bf16 ulp
    # of y alone is 4.8e-2 RMS (measured max|err|/RMS 5.55e-2)
    check_output(xb, wr, None, None, shape.k, cpu(y.float()), cpu(idx), fp8=fp8, storage_slack=True)
    # a zero token row: every expert's input is zero, so is every output
    assert torch.all(y[3] == 0)
    layer.close()


@pytest.mark.parametrize("x2", [True, False])
@pytest.mark.parametrize("T", [1, 128])
def test_fp8_flash_decode(T, x2):
    # d=4096, 288 routed + 1 shared, top-8, width 1280
    fp8_case(synth.FLASH_DECODE.with_tokens(T), seed=24, n_sample=None if T == 1 else 48, x2=x2)


@pytest.mark.parametrize("x2", [True, False])
def test_fp8_many_tokens(x2):
    # 2000 tokens over 24 experts: chunked dispatch, every row (the shared
    # expert's too) scattered, ~170 rows per group in 128-row tiles
    fp8_case(synth.LayerShape(T=2000, d=512, E=24, k=2, F=256), seed=26, n_sample=64, x2=x2)


def test_fp8_smaller_top_k_renormalized():
    # per-call top-4 with renormalised weights on an FP8 handle built for top-8:
    # the two-term scatter and the requantisation of H follow the call's k
    shape = synth.LayerShape(T=100, d=256, E=32, k=8, F=128)
    inp = synth.make_inputs(shape, seed=28, device=DEV)
    q_gu, s_gu, q_d, s_d = quantised(inp)
    layer = binding.MoeLayer.fp8(inp.w_router, q_gu, s_gu, q_d, s_d, shape.k, shape.T)
    y = layer.forward(inp.x, top_k=4, renormalize=True)
    assert layer.check() == binding.MOE_OK
    assert layer.last_kernel_count() == 8  # 7 + the requantisation of H
    xb = synth.bf16_bits(inp.x)
    wr = cpu(inp.w_router)
    idx, _, _, _, _ = layer.route(inp.x, top_k=4, renormalize=True)  # the GPU's selection (near-ties)
    y_ref = oracle.forward_fp8(xb, wr, cpu(q_gu), cpu(s_gu), cpu(q_d), cpu(s_d), 4, sel=cpu(idx),
                               renormalize=True)
    compare(cpu(y.float()), y_ref)
    layer.close()


def test_fp8_two_term_128_row_tiles():
    # 128-row tiles of the two-term kernel (N = 256, 4 ring stages): ~150 rows
    # per group, ragged second tiles, d = 1024 gives 8 K steps per gate/up tile
    fp8_case(synth.LayerShape(T=1200, d=1024, E=16, k=2, F=256), seed=29, tiles=(128, 128), n_sample=64)


@pytest.mark.parametrize("parts", [2, 3, 4])
@pytest.mark.parametrize("T,d,F,tiles", [(1, 512, 256, (32, 32)), (5, 1024, 512, (16, 32)), (20, 512, 256, (16, 16))])
def test_fp8_gemm_k_split(parts, T, d, F, tiles):
    # Two-term E4M3 GEMMs with every item's K range in parts (fewer where K
    # has fewer steps of 128): each part's hi + lo sum, the parts summed in
    # order, then the row and token scales; run to run identical (fp8_case).
    shape = synth.LayerShape(T=T, d=d, E=16, k=2, F=F)
    fp8_case(shape, seed=90 + T + parts, tiles=tiles, max_tokens=64, ksplit=parts)



# ---------------------------------------------------------------- full size --

@pytest.fixture(scope="module")
def flash_fp8_weights():
    """E4M3 codes and scales of the flash-shaped layer's weights (d=4096, 288
    routed + 1 shared, width 1280), made once for the module."""
    shape = synth.FLASH_DECODE
    inp = synth.make_inputs(shape, seed=0, device=DEV)
    q = quantised(inp)
    wr = inp.w_router
    del inp
    host = tuple(cpu(t) for t in q)
    yield wr, q, host


def flash_fp8_case(weights, T, seed, x2, n_sample=64, skew=None):
    """T tokens on the flash-shaped FP8 layer: routing and dispatch on every
    token, the output on a seeded sample plus every near-tie token plus one
    token per expert used."""
    import os
    wr, (q_gu, s_gu, q_d, s_d), fp8_host = weights
    shape = synth.FLASH_DECODE.with_tokens(T)
    x = synth.make_tokens(shape, seed=seed, device=DEV, skew=skew)
    if skew is not None:
        wr = synth.skewed_router(wr, seed, skew)
    old = os.environ.get("MOE_FP8_X2")
    os.environ["MOE_FP8_X2"] = "1" if x2 else "0"
    try:
        layer = binding.MoeLayer.fp8(wr, q_gu, s_gu, q_d, s_d, shape.k, T)
    finally:
        if old is None:
            os.environ.pop("MOE_FP8_X2", None)
        else:
            os.environ["MOE_FP8_X2"] = old
    idx, prob, perm, offsets, gap = layer.route(x)
    y = layer.forward(x)
    assert layer.check() == binding.MOE_OK
    xb = synth.bf16_bits(x)
    wr_h = cpu(wr)
    idx_h = cpu(idx)
    near, _ = check_routing(xb, wr_h, shape.k, idx_h, cpu(prob), cpu(gap), cpu(perm), cpu(offsets))
    tokens = sample_tokens(T, idx_h, n_sample, seed, near)
    y_h = cpu(y[torch.from_numpy(tokens).long().to(DEV)].float())
    ratio = check_output(xb, wr_h, None, None, shape.k, y_h, idx_h, tokens=tokens, fp8=fp8_host)
    y2 = layer.forward(x)
    assert torch.equal(y, y2)
    layer.close()
    return ratio


@pytest.mark.parametrize("x2", [True, False])
@pytest.mark.parametrize("T", [512, 2048, 8192])
def test_fp8_flash_many_tokens(flash_fp8_weights, T, x2):
    # the E4M3 kernels at the flash shape with many rows per group: 64- and
    # 128-row tiles, thousands of two-term rows, the chunked dispatch
    flash_fp8_case(flash_fp8_weights, T, seed=300 + T, x2=x2)


@pytest.mark.parametrize("x2", [True, False])
def test_fp8_flash_skewed(flash_fp8_weights, x2):
    # Zipf-skewed routing, T=4096: the hottest expert ~10x the mean rows,
    # 40 experts unused
    flash_fp8_case(flash_fp8_weights, 4096, seed=102, x2=x2, skew="zipf")
