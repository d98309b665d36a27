"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars (see moe_check.py): routing and dispatch bit-exact outside near-ties,
probabilities within the derived fp32 bound, layer output within
2e-2 * RMS of the oracle.
"""
import os

import numpy as np
import pytest
import torch

from expert_routed_ffn_gemm_gb300 import binding, synth

from moe_check import check_output, check_routing, cpu, host_bits, sample_tokens, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def make_layer(inp, max_tokens=None, tiles=(0, 0), out_fp32=False, has_shared=True, env=None):
    x, wr, wgu, wd = to_dev(inp, DEV)
    env = dict(env or {})
    env.setdefault("MOE_TILE_N_GATEUP", str(tiles[0]))
    env.setdefault("MOE_TILE_N_DOWN", str(tiles[1]))
    old = {kk: os.environ.get(kk) for kk in env}
    os.environ.update(env)
    try:
        layer = binding.MoeLayer(wr, wgu, wd, inp.shape.k, max_tokens or max(1, inp.shape.T),
                                 has_shared=has_shared, out_fp32=out_fp32)
    finally:
        for kk, v in old.items():
            if v is None:
                os.environ.pop(kk, None)
            else:
                os.environ[kk] = v
    return layer, x


def run_and_check(inp, tiles=(0, 0), tokens=None, out_fp32=False, max_tokens=None, storage_slack=False):
    shape = inp.shape
    layer, x = make_layer(inp, max_tokens=max_tokens, tiles=tiles, out_fp32=out_fp32,
                          has_shared=shape.has_shared)
    idx, prob, perm, offsets, gap = layer.route(x)
    y = layer.forward(x)
    assert layer.check() == binding.MOE_OK
    xb, wr, wgu, wd = host_bits(inp)
    idx_h = cpu(idx)
    near, _ = check_routing(xb, wr, shape.k, idx_h, cpu(prob), cpu(gap), cpu(perm), cpu(offsets),
                            has_shared=shape.has_shared)
    y_h = cpu(y.float())
    if tokens is None:
        tokens = np.arange(shape.T, dtype=np.int32)
    else:
        tokens = sample_tokens(shape.T, idx_h, tokens, seed=1, extra=near)
    ratio = check_output(xb, wr, wgu, wd, shape.k, y_h[tokens], idx_h, tokens=tokens,
                         has_shared=shape.has_shared, out_bf16=not out_fp32, storage_slack=storage_slack)
    layer.close()
    return ratio, len(near)


def test_tiny_workload():
    inp = synth.make_inputs(synth.TINY, seed=0)
    run_and_check(inp)


@pytest.mark.parametrize("tiles", [(16, 16), (32, 32), (64, 64), (128, 128), (256, 256), (16, 256), (128, 16)])
def test_tile_widths_ragged(tiles):
    # 300 tokens over 16 experts (top-2): ~37 rows per expert, ragged in every
    # tile width, several token tiles per group for the small widths.
    shape = synth.LayerShape(T=300, d=256, E=16, k=2, F=128)
    inp = synth.make_inputs(shape, seed=3)
    run_and_check(inp, tiles=tiles)


@pytest.mark.parametrize("T", [1, 2, 7, 33, 129])
def test_token_counts(T):
    shape = synth.LayerShape(T=T, d=256, E=16, k=2, F=128)
    inp = synth.make_inputs(shape, seed=10 + T)
    run_and_check(inp, max_tokens=200)


@pytest.mark.parametrize("T", [5000, 20000])
def test_many_tokens_small_layer(T):
    # Many tokens over few experts: 256-token router tiles, one warp per token
    # in the top-k, groups of hundreds of rows on CTA pairs with ragged tails.
    shape = synth.LayerShape(T=T, d=256, E=16, k=2, F=128)
    inp = synth.make_inputs(shape, seed=50 + T % 7)
    run_and_check(inp, tokens=64)


@pytest.mark.parametrize("shape", [
    synth.LayerShape(T=300, d=384, E=24, k=8, F=128, has_shared=False),  # 8 terms, no shared expert
    synth.LayerShape(T=300, d=384, E=24, k=7, F=128),                    # 8 terms with the shared expert
    synth.LayerShape(T=1500, d=256, E=32, k=8, F=128),                   # 9 terms, chunked dispatch
    synth.LayerShape(T=1024, d=256, E=40, k=6, F=128),                   # first token count of the chunked path
    synth.LayerShape(T=1025, d=128, E=300, k=8, F=128),                  # 16 slots per lane in the top-k
])
@pytest.mark.parametrize("out_fp32", [False, True])
def test_combine_terms_and_chunked_dispatch(shape, out_fp32):
    # bf16 y: measured max|err|/RMS 2.62e-2 on the 1024-token case, two
    # elements near 6 RMS where half a bf16 ulp of y alone is 2.0e-2 RMS; fp32
    # y meets the plain bound
    inp = synth.make_inputs(shape, seed=60 + shape.T % 11 + shape.k)
    run_and_check(inp, tokens=96 if shape.T > 1000 else None, out_fp32=out_fp32, storage_slack=not out_fp32)


def test_chunked_dispatch_ties_and_one_hot():
    # Many tokens choosing the same experts: W_r = 0 (every token picks 0..3,
    # all rows of a chunk land in four experts) and a one-hot bias.
    shape = synth.LayerShape(T=2000, d=256, E=16, k=4, F=128)
    inp = synth.make_inputs(shape, seed=12)
    inp.w_router.zero_()
    layer, x = make_layer(inp)
    idx, prob, perm, offsets, gap = layer.route(x)
    assert np.all(cpu(idx) == np.arange(4)[None, :])
    off = cpu(offsets)
    assert list(off[:6]) == [0, 2000, 4000, 6000, 8000, 8000]
    perm_h = cpu(perm)
    for e in range(4):  # rows of expert e: tokens in order, slot e
        np.testing.assert_array_equal(perm_h[e * 2000:(e + 1) * 2000], np.arange(2000) * 4 + e)
    layer.close()
    inp = synth.make_inputs(shape, seed=13)
    inp.x[:, 0] = 1.0
    inp.w_router[:, 0] = -20.0
    inp.w_router[5, 0] = 20.0
    run_and_check(inp, tokens=64)


@pytest.mark.parametrize("parts", ["2", "3", "4", "b", "auto"])
@pytest.mark.parametrize("T,d,F,tiles", [(1, 256, 128, (32, 32)), (3, 512, 256, (16, 32)),
                                         (20, 512, 256, (16, 16)), (7, 256, 128, (32, 16)),
                                         (5, 1024, 384, (32, 32)), (2, 4096, 128, (16, 16))])
def test_gemm_k_split(parts, T, d, F, tiles):
    # Few work items: every item's K range in 2..4 parts (fewer where K has
    # fewer steps of 64), summed in part order by the last part to finish;
    # "b": the K steps of all items in one contiguous range per CTA (an
    # item's parts are the ranges it spans, 1..4 of them).
    shape = synth.LayerShape(T=T, d=d, E=16, k=2, F=F)
    inp = synth.make_inputs(shape, seed=70 + T + d // 128)
    env = {} if parts == "auto" else {"MOE_GEMM_KSPLIT": parts}
    layer, x = make_layer(inp, tiles=tiles, env=env)
    y1 = layer.forward(x)
    y2 = layer.forward(x)
    assert layer.check() == binding.MOE_OK
    assert torch.equal(y1, y2)  # fixed summation order: run to run identical
    xb, wr, wgu, wd = host_bits(inp)
    idx, prob, perm, offsets, gap = layer.route(x)
    check_output(xb, wr, wgu, wd, shape.k, cpu(y1.float()), cpu(idx), tokens=np.arange(T, dtype=np.int32))
    layer.close()


@pytest.mark.parametrize("T,d,E,F,tiles", [(1, 512, 16, 256, (0, 0)), (24, 256, 16, 128, (32, 32)),
                                           (128, 1024, 8, 128, (16, 16)), (6, 256, 40, 384, (32, 32))])
def test_down_weight_prefetch(T, d, E, F, tiles):
    # The single-CTA gate/up brings the down launch's first weights into L2
    # when that launch has at most two waves of items (all of these): a hint
    # only, so the output is bit-identical with it off, with one or two waves
    # of it, and within the bound of the oracle.
    shape = synth.LayerShape(T=T, d=d, E=E, k=2, F=F)
    inp = synth.make_inputs(shape, seed=90 + T + E)
    ys = []
    for waves in ("0", "1", "2"):
        layer, x = make_layer(inp, tiles=tiles, env={"MOE_PF_DOWN_WAVES": waves})
        ys.append(layer.forward(x))
        assert layer.check() == binding.MOE_OK
        if waves == "1":
            idx = layer.route(x)[0]
        layer.close()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
    xb, wr, wgu, wd = host_bits(inp)
    check_output(xb, wr, wgu, wd, shape.k, cpu(ys[1].float()), cpu(idx), tokens=np.arange(T, dtype=np.int32))


def test_several_weight_tiles_and_k_steps():
    # F = 256 -> 2 gate/up weight tiles, d = 512 -> 4 down weight tiles and 8 K steps.
    shape = synth.LayerShape(T=200, d=512, E=32, k=4, F=256)
    inp = synth.make_inputs(shape, seed=5)
    run_and_check(inp)


def test_kernel_count_reported():
    inp = synth.make_inputs(synth.TINY, seed=41)
    layer, x = make_layer(inp)
    layer.forward(x)
    assert layer.last_kernel_count() == 7
    big = synth.make_inputs(synth.TINY.with_tokens(1024), seed=42)
    layer2, x2 = make_layer(big)
    layer2.forward(x2)
    assert layer2.last_kernel_count() == 9  # chunked dispatch from 1024 tokens on
    layer2.close()
    binding.moe_forward(layer.handle, x[:0], 0, torch.empty_like(x[:0]))
    assert layer.last_kernel_count() == 0
    layer.close()


def test_every_expert_selected():
    # k == E: all experts run for every token; gap is +inf.
    shape = synth.LayerShape(T=40, d=256, E=8, k=8, F=128)
    inp = synth.make_inputs(shape, seed=6)
    run_and_check(inp)


def test_without_shared_expert():
    shape = synth.LayerShape(T=50, d=256, E=12, k=3, F=128, has_shared=False)
    inp = synth.make_inputs(shape, seed=7)
    run_and_check(inp)


def test_one_hot_expert_and_empty_experts():
    # A huge bias on expert 5 (feature 0 set to 1): every token picks it first;
    # most experts receive no rows.
    shape = synth.LayerShape(T=96, d=256, E=16, k=2, F=128)
    inp = synth.make_inputs(shape, seed=8)
    inp.x[:, 0] = 1.0
    inp.w_router[:, 0] = -20.0
    inp.w_router[5, 0] = 20.0
    inp.w_router[9, 0] = 10.0
    layer, x = make_layer(inp)
    idx, prob, perm, offsets, gap = layer.route(x)
    off = cpu(offsets)
    assert off[5 + 1] - off[5] == 96
    run_and_check(inp)


def test_uniform_router_tie_rule():
    # W_r = 0: every probability is 1/E and the lower indices win.
    shape = synth.LayerShape(T=20, d=256, E=16, k=4, F=128)
    inp = synth.make_inputs(shape, seed=9)
    inp.w_router.zero_()
    layer, x = make_layer(inp)
    idx, prob, perm, offsets, gap = layer.route(x)
    assert np.all(cpu(idx) == np.arange(4)[None, :])
    assert np.all(cpu(prob) == np.float32(1.0 / 16))
    y = layer.forward(x)
    xb, wr, wgu, wd = host_bits(inp)
    check_output(xb, wr, wgu, wd, 4, cpu(y.float()), cpu(idx))
    layer.close()


def test_fp32_output():
    inp = synth.make_inputs(synth.TINY, seed=11)
    run_and_check(inp, out_fp32=True)


def test_deterministic_run_to_run():
    shape = synth.LayerShape(T=500, d=256, E=16, k=2, F=128)
    inp = synth.make_inputs(shape, seed=12)
    layer, x = make_layer(inp)
    a = [t.clone() for t in layer.route(x)]
    y1 = layer.forward(x).clone()
    b = layer.route(x)
    y2 = layer.forward(x)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert torch.equal(y1, y2)
    layer.close()


def test_host_entry_point_matches_device_entry_point():
    inp = synth.make_inputs(synth.TINY, seed=13)
    layer, x = make_layer(inp)
    y_dev = layer.forward(x)
    x_host = inp.x.clone().pin_memory()
    y_host = layer.forward_host(x_host)
    assert torch.equal(y_dev.cpu(), y_host)
    layer.close()


def test_zero_tokens_and_limits():
    inp = synth.make_inputs(synth.TINY, seed=14)
    layer, x = make_layer(inp, max_tokens=64)
    y = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    binding.moe_forward(layer.handle, x[:0], 0, y)
    big = torch.zeros((65, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(binding.MoeError) as e:
        layer.forward(big)
    assert e.value.status == binding.MOE_ERR_TOO_MANY_TOKENS
    with pytest.raises(binding.MoeError) as e:
        binding.moe_forward(layer.handle, x.cpu(), 64, torch.empty_like(x))
    assert e.value.status == binding.MOE_ERR_INVALID_ARG
    assert layer.check() == binding.MOE_OK
    layer.close()


def test_bounded_wait_reports_instead_of_hanging():
    # A barrier nothing arrives at: the kernel gives up after 1 ms and the
    # host reads the error status; the context stays usable.
    assert binding.moe_selftest_wait_timeout(1_000_000) == binding.MOE_ERR_DEVICE
    inp = synth.make_inputs(synth.TINY, seed=15)
    run_and_check(inp)


# ---------------------------------------------------------------- full size --

@pytest.fixture(scope="module")
def flash_weights():
    shape = synth.FLASH_DECODE
    inp = synth.make_inputs(shape, seed=0, device=DEV)
    host = host_bits(inp)
    yield inp, host
    del inp


def flash_case(flash_weights, T, seed, n_sample=None, skew=None, out_fp32=False):
    inp, (_, wr_h, wgu_h, wd_h) = flash_weights
    shape = synth.FLASH_DECODE.with_tokens(T)
    x = synth.make_tokens(shape, seed=seed, device=DEV, skew=skew)
    wr = inp.w_router
    wr_h2 = wr_h
    if skew is not None:
        wr = synth.skewed_router(inp.w_router, seed, skew)
        wr_h2 = cpu(wr)
    layer = binding.MoeLayer(wr, inp.w_gate_up, inp.w_down, shape.k, T, out_fp32=out_fp32)
    idx, prob, perm, offsets, gap = layer.route(x)
    y = layer.forward(x)
    assert layer.check() == binding.MOE_OK
    xb = synth.bf16_bits(x)
    idx_h = cpu(idx)
    near, _ = check_routing(xb, wr_h2, shape.k, idx_h, cpu(prob), cpu(gap), cpu(perm), cpu(offsets))
    tokens = np.arange(T, dtype=np.int32) if n_sample is None else sample_tokens(T, idx_h, n_sample, seed, near)
    y_h = cpu(y[torch.from_numpy(tokens).long().to(DEV)].float())
    ratio = check_output(xb, wr_h2, wgu_h, wd_h, shape.k, y_h, idx_h, tokens=tokens, out_bf16=not out_fp32)
    layer.close()
    return ratio


def test_flash_back_to_back_calls_match_calls_alone(flash_weights):
    # The flash shape's regimes (1-4 tokens with the routing finished in the
    # gate/up launch over replicated token rows, the decode batch, 37 tokens
    # with K-split GEMMs, the chunked dispatch with CTA pairs and the second
    # stream) enqueued back to back with no host synchronisation, switching
    # between two token sets: every result bit for bit that of the same call
    # run alone (consecutive calls overlap on the device; a stale or clobbered
    # buffer would show).
    inp, _ = flash_weights
    shape = synth.FLASH_PREFILL
    xs = [synth.make_tokens(shape, seed=s, device=DEV) for s in (71, 72)]
    layer = binding.MoeLayer(inp.w_router, inp.w_gate_up, inp.w_down, shape.k, shape.T)
    calls = [(i % 2, T) for i, T in enumerate([1, 128, 4, 8192, 2, 37, 2048, 3, 1, 128] * 2)]
    ref = {}
    for w, T in sorted(set(calls)):
        ref[(w, T)] = layer.forward(xs[w][:T]).clone()
        torch.cuda.synchronize()
        assert layer.check() == binding.MOE_OK
    outs = [torch.empty((T, shape.d), dtype=torch.bfloat16, device=DEV) for _, T in calls]
    torch.cuda.synchronize()
    for (w, T), y in zip(calls, outs):
        layer.forward(xs[w][:T], y)
    torch.cuda.synchronize()
    assert layer.check() == binding.MOE_OK
    bad = [c for c, y in zip(calls, outs) if not torch.equal(y, ref[c])]
    assert not bad, bad
    layer.close()


@pytest.mark.parametrize("out_fp32", [False, True])
def test_flash_decode_all_tokens(flash_weights, out_fp32):
    # d=4096, 288 routed + 1 shared, top-8, width 1280, T=128 (decode batch)
    flash_case(flash_weights, 128, seed=100, out_fp32=out_fp32)


def test_flash_prefill_sampled(flash_weights):
    # T=8192: routing and dispatch on every token, output on a seeded sample
    # plus every near-tie token plus one token per used expert.
    flash_case(flash_weights, 8192, seed=101, n_sample=128)


@pytest.mark.parametrize("out_fp32", [False, True])
def test_flash_skewed_sampled(flash_weights, out_fp32):
    # Zipf-skewed routing, T=4096: hottest expert ~10x the mean, 40 unused.
    flash_case(flash_weights, 4096, seed=102, n_sample=64, skew="zipf", out_fp32=out_fp32)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 8, 32, 512, 2048])
def test_flash_sweep_points(flash_weights, T):
    # 1 to 3 tokens: balanced K ranges in the gate/up GEMM; 1 to 4: the
    # few-token routing launch (with one or two tokens also the row copy)
    flash_case(flash_weights, T, seed=200 + T, n_sample=None if T <= 32 else 64)


def test_flash_largest_sweep_point(flash_weights):
    # T=32768: routing and dispatch on every token, output on a sample; fp32 y
    flash_case(flash_weights, 32768, seed=232, n_sample=48, out_fp32=True)


@pytest.mark.parametrize("T,d,F", [(200, 256, 128), (1, 2048, 256), (3, 2048, 256)])
def test_forward_captured_in_a_cuda_graph(T, d, F):
    # moe_forward enqueues only kernels and a memset on the caller's stream
    # (no host synchronisation, no allocation), so it can be captured once
    # and replayed; replays on new inputs match the eager call bit for bit.
    # 1 and 3 tokens: the routing finished in the gate/up launch, K split in
    # balanced ranges (the part counters reset by each launch), and with one
    # token the L2 prefetch of the down launch's first weights.
    shape = synth.LayerShape(T=T, d=d, E=16, k=2, F=F)
    inp = synth.make_inputs(shape, seed=16 + T)
    layer, x = make_layer(inp)
    y = torch.empty((shape.T, shape.d), dtype=torch.bfloat16, device=DEV)
    layer.forward(x, y)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer.forward(x, y, stream=s)
    for seed in (17, 18):
        x.copy_(synth.make_tokens(shape, seed=seed, device=DEV))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, layer.forward(x))
    assert layer.check() == binding.MOE_OK
    layer.close()


def test_forward_from_a_new_thread():
    # A host thread that has not used CUDA yet: the library binds the handle's
    # device before its first driver call (1500 tokens take the chunked
    # dispatch, whose first call is the tensor-map encoding of x).
    import threading

    inp = synth.make_inputs(synth.LayerShape(T=1500, d=256, E=16, k=2, F=128), seed=47)
    layer, x = make_layer(inp)
    y_main = layer.forward(x)
    torch.cuda.synchronize()
    out, errs = {}, []

    def work():
        try:
            out["y"] = layer.forward(x)
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001 - reported below
            errs.append(e)

    t = threading.Thread(target=work)
    t.start()
    t.join(timeout=120)
    assert not errs, errs
    assert torch.equal(out["y"], y_main)
    layer.close()


@pytest.mark.parametrize("fused", ["1", "0"])
@pytest.mark.parametrize("T,d,E,k", [(1, 256, 16, 2), (3, 512, 64, 4), (4, 256, 300, 8), (4, 1024, 24, 8)])
def test_few_token_routing_both_paths(fused, T, d, E, k):
    # From 1 to 4 tokens routing and dispatch run as one launch (fp32 FMA dot
    # products, MOE_SMALL_ROUTE=0 turns it off for the tensor-core router):
    # both paths against the oracle.
    shape = synth.LayerShape(T=T, d=d, E=E, k=k, F=128)
    inp = synth.make_inputs(shape, seed=400 + T + E)
    layer, x = make_layer(inp, env={"MOE_SMALL_ROUTE": fused})
    idx, prob, perm, offsets, gap = layer.route(x)
    y = layer.forward(x)
    assert layer.check() == binding.MOE_OK
    # fused: one launch for the logits and copies of the token rows, the
    # top-k and dispatch in the gate/up launch
    assert layer.last_kernel_count() == (4 if fused == "1" else 7)
    xb, wr, wgu, wd = host_bits(inp)
    check_routing(xb, wr, k, cpu(idx), cpu(prob), cpu(gap), cpu(perm), cpu(offsets))
    check_output(xb, wr, wgu, wd, k, cpu(y.float()), cpu(idx), storage_slack=False)
    y2 = layer.forward(x)
    assert torch.equal(y, y2)
    layer.close()


@pytest.mark.parametrize("T,d,E,k,F,shared,top_k,renorm", [
    (1, 256, 16, 2, 128, True, None, False),
    (2, 512, 64, 4, 256, True, None, False),
    (3, 256, 300, 8, 128, False, None, False),
    (4, 1024, 24, 8, 384, True, 4, True),
    (4, 256, 512, 32, 128, True, None, False),  # T*k = 128 picks over 512 experts, the limits
    (3, 256, 6, 2, 128, True, None, False),  # fewer experts (routing blocks) than copies of the rows
])
def test_routing_in_gate_up_launch(T, d, E, k, F, shared, top_k, renorm):
    # 1 to 4 tokens, bf16 weights: the routing launch writes the logits and
    # copies of the token rows only, and every gate/up CTA ranks the tokens
    # (the same softmax and top-k code), lays out the dispatch and reads its
    # copy of the rows; CTA 0 writes the routing results for the down GEMM and
    # the combine.  Bit-identical to the routing launch doing it all
    # (MOE_ROUTE_IN_GEMM=0), with per-call top-k and renormalisation too, and
    # against the oracle.  The last case also has more terms per token (33)
    # than the combine has threads (32 for d = 256).
    shape = synth.LayerShape(T=T, d=d, E=E, k=k, F=F, has_shared=shared)
    inp = synth.make_inputs(shape, seed=700 + T + E)
    ys = {}
    for v in ("1", "0"):
        layer, x = make_layer(inp, has_shared=shared, env={"MOE_ROUTE_IN_GEMM": v})
        ys[v] = [layer.forward(x), layer.forward(x, top_k=top_k, renormalize=renorm)]
        assert layer.check() == binding.MOE_OK
        assert layer.last_kernel_count() == (4 if v == "1" else 5 if T > 2 else 4)
        if v == "1":
            idx, prob, perm, offsets, gap = layer.route(x)
        layer.close()
    assert torch.equal(ys["1"][0], ys["0"][0]) and torch.equal(ys["1"][1], ys["0"][1])
    xb, wr, wgu, wd = host_bits(inp)
    check_routing(xb, wr, k, cpu(idx), cpu(prob), cpu(gap), cpu(perm), cpu(offsets), has_shared=shared)
    check_output(xb, wr, wgu, wd, k, cpu(ys["1"][0].float()), cpu(idx), has_shared=shared)


@pytest.mark.parametrize("tiles", [(0, 0), (128, 128)])
@pytest.mark.parametrize("overlap", ["1", "0"])
def test_shared_expert_on_a_second_stream(overlap, tiles):
    # From 2048 tokens on the shared expert's gate/up runs on a second stream
    # beside the dispatch and row scatter (MOE_SHARED_OVERLAP=0: in the one
    # gate/up launch): same results bit for bit, against the oracle, and the
    # fork and join capture into a CUDA graph whose replays match the eager call.
    # tiles (128, 128): single-CTA token tiles forced, the shared expert stays
    # in the routed launches either way.
    shape = synth.LayerShape(T=2500, d=256, E=16, k=2, F=128)
    inp = synth.make_inputs(shape, seed=501)
    layer, x = make_layer(inp, tiles=tiles, env={"MOE_SHARED_OVERLAP": overlap})
    y = layer.forward(x)
    assert layer.check() == binding.MOE_OK
    assert layer.last_kernel_count() == (11 if overlap == "1" and tiles == (0, 0) else 9)
    other, _ = make_layer(inp, tiles=tiles, env={"MOE_SHARED_OVERLAP": "0" if overlap == "1" else "1"})
    assert torch.equal(y, other.forward(x))
    other.close()
    idx, prob, perm, offsets, gap = layer.route(x)
    xb, wr, wgu, wd = host_bits(inp)
    near, _ = check_routing(xb, wr, shape.k, cpu(idx), cpu(prob), cpu(gap), cpu(perm), cpu(offsets))
    tokens = sample_tokens(shape.T, cpu(idx), 96, seed=5, extra=near)
    check_output(xb, wr, wgu, wd, shape.k, cpu(y.float())[tokens], cpu(idx), tokens=tokens)
    yg = torch.empty_like(y)
    layer.forward(x, yg)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            layer.forward(x, yg, stream=st)
    for seed in (502, 503):
        x.copy_(synth.make_tokens(shape, seed=seed, device=DEV))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(yg, layer.forward(x))
    assert layer.check() == binding.MOE_OK
    layer.close()


@pytest.mark.parametrize("case", range(12))
def test_random_small_layers(case):
    # Seeded random small layers (token count, width, experts, top-k, expert
    # width, token tiles, K split) against the oracle, run to run identical:
    # the corners of the work decomposition (balanced K ranges whose parts
    # span 1..4 CTAs, ragged token tiles, groups without rows) that the named
    # cases may miss.
    rng = np.random.default_rng(900 + case)
    T = int(rng.integers(1, 48))
    d = int(rng.choice([256, 512, 1024, 2048]))
    E = int(rng.integers(4, 65))
    k = int(rng.integers(1, min(8, E) + 1))
    F = int(rng.choice([128, 256, 384]))
    tiles = [(0, 0), (16, 16), (32, 32), (16, 32)][int(rng.integers(0, 4))]
    split = ["auto", "b", "2", "1"][int(rng.integers(0, 4))]
    shape = synth.LayerShape(T=T, d=d, E=E, k=k, F=F)
    inp = synth.make_inputs(shape, seed=910 + case)
    env = {} if split == "auto" else {"MOE_GEMM_KSPLIT": split}
    # fp32 y: the bound then measures the arithmetic, not y's bf16 storage
    layer, x = make_layer(inp, tiles=tiles, env=env, out_fp32=True)
    y = layer.forward(x)
    assert layer.check() == binding.MOE_OK
    assert torch.equal(layer.forward(x), y)
    idx, prob, perm, offsets, gap = layer.route(x)
    xb, wr, wgu, wd = host_bits(inp)
    check_routing(xb, wr, k, cpu(idx), cpu(prob), cpu(gap), cpu(perm), cpu(offsets))
    check_output(xb, wr, wgu, wd, k, cpu(y), cpu(idx), out_bf16=False)
    layer.close()
