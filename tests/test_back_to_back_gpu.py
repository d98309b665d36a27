"""Layer calls enqueued back to back, with no host synchronisation between
them, give bit for bit what each gives alone.

Consecutive calls overlap on the device: every kernel may start while the one
before it ends (programmatic dependent launch), and from 2048 tokens on the
shared expert's GEMMs run on a second stream.  A call that read a buffer the
previous call was still writing, or wrote one it was still reading, would
show up here: the sequence switches between two inputs, token counts from
every dispatch regime (1-4 tokens with the routing finished in the gate/up
launch, the single-block dispatch with K-split GEMMs, the chunked dispatch,
256-token tiles on CTA pairs, the second stream) and per-call top-k, so a
stale value from the call before is never the right one.  The reference for
every (input, token count, top-k) is the same call run alone and synchronised.
"""
import pytest
import torch

from expert_routed_ffn_gemm_gb300 import binding, synth

from moe_check import to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# (tokens, top_k or None for the layer's k, renormalise)
SEQUENCE = [(1, None, False), (37, None, False), (4, None, False), (600, None, False), (2500, None, False),
            (3, None, False), (130, 1, True), (2048, None, False), (1, None, False), (2, None, False),
            (1100, None, False), (4, 1, True), (2500, 1, True), (37, None, False)]


def _layer(fp8: bool, seed: int = 901):
    shape = synth.LayerShape(T=2500, d=256, E=16, k=2, F=128)
    inp = synth.make_inputs(shape, seed=seed)
    x, wr, wgu, wd = to_dev(inp, DEV)
    if fp8:
        q = binding.moe_quantize_fp8(wgu) + binding.moe_quantize_fp8(wd)
        layer = binding.MoeLayer.fp8(wr, *q, shape.k, shape.T)
    else:
        layer = binding.MoeLayer(wr, wgu, wd, shape.k, shape.T)
    x2 = to_dev(synth.make_inputs(shape, seed=seed + 1), DEV)[0]
    return layer, (x, x2)


def _call(layer, x, T, top_k, renorm, y, stream=None):
    if top_k is None:
        return layer.forward(x[:T], y, stream=stream)
    return layer.forward(x[:T], y, stream=stream, top_k=top_k, renormalize=renorm)


@pytest.mark.parametrize("fp8", [False, True])
def test_back_to_back_calls_match_calls_alone(fp8):
    layer, xs = _layer(fp8)
    calls = [(i % 2, T, kk, rn) for i, (T, kk, rn) in enumerate(SEQUENCE * 3)]
    ref = {}
    for c in dict.fromkeys(calls):
        w, T, kk, rn = c
        y = torch.empty((T, 256), dtype=torch.bfloat16, device=DEV)
        _call(layer, xs[w], T, kk, rn, y)
        torch.cuda.synchronize()
        assert layer.check() == binding.MOE_OK
        ref[c] = y.clone()
    outs = [torch.full((T, 256), float("nan"), dtype=torch.bfloat16, device=DEV) for (_, T, _, _) in calls]
    torch.cuda.synchronize()
    for c, y in zip(calls, outs):
        w, T, kk, rn = c
        _call(layer, xs[w], T, kk, rn, y)
    torch.cuda.synchronize()
    assert layer.check() == binding.MOE_OK
    bad = [i for i, (c, y) in enumerate(zip(calls, outs)) if not torch.equal(y, ref[c])]
    assert not bad, [calls[i] for i in bad]
    layer.close()


def test_two_layers_on_two_streams_at_once():
    # Two handles (bf16 and FP8 weights, different seeds) each enqueue on a
    # stream of their own, their calls alternating and running side by side on
    # the device with no synchronisation: nothing is shared between handles,
    # so each result is bit for bit that of the same call alone.
    layers = [_layer(False, seed=911), _layer(True, seed=921)]
    seqs = [[(T, None, False) for T in (2500, 4, 600, 1, 2048, 37, 130, 3)],
            [(T, None, False) for T in (1, 2048, 37, 2500, 3, 600, 4, 1100)]]
    seqs[1][2] = (37, 1, True)
    refs = [[], []]
    for h in range(2):
        layer, xs = layers[h]
        for i, (T, kk, rn) in enumerate(seqs[h]):
            y = torch.empty((T, 256), dtype=torch.bfloat16, device=DEV)
            _call(layer, xs[i % 2], T, kk, rn, y)
            torch.cuda.synchronize()
            assert layer.check() == binding.MOE_OK
            refs[h].append(y)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[torch.empty((T, 256), dtype=torch.bfloat16, device=DEV) for T, _, _ in seqs[h]] for h in range(2)]
    torch.cuda.synchronize()
    for i in range(len(seqs[0])):
        for h in range(2):
            layer, xs = layers[h]
            T, kk, rn = seqs[h][i]
            _call(layer, xs[i % 2], T, kk, rn, outs[h][i], stream=streams[h])
    torch.cuda.synchronize()
    for h in range(2):
        assert layers[h][0].check() == binding.MOE_OK
        bad = [seqs[h][i] for i in range(len(seqs[h])) if not torch.equal(outs[h][i], refs[h][i])]
        assert not bad, (h, bad)
        layers[h][0].close()


def test_two_host_threads_each_with_a_handle():
    # Two host threads, each driving its own handle on its own stream (the
    # library's host code holds no per-call global state): every result bit for
    # bit the same call alone.
    import threading

    layers = [_layer(False, seed=931), _layer(False, seed=941)]
    seq = [(T, None, False) for T in (2500, 1, 600, 4, 2048, 37, 3, 130)]
    refs = [[], []]
    for h in range(2):
        layer, xs = layers[h]
        for i, (T, kk, rn) in enumerate(seq):
            y = torch.empty((T, 256), dtype=torch.bfloat16, device=DEV)
            _call(layer, xs[i % 2], T, kk, rn, y)
            torch.cuda.synchronize()
            refs[h].append(y)
    outs = [[[torch.empty((T, 256), dtype=torch.bfloat16, device=DEV) for T, _, _ in seq] for _ in range(5)]
            for _ in range(2)]
    torch.cuda.synchronize()
    errors = []

    def drive(h):
        try:
            layer, xs = layers[h]
            st = torch.cuda.Stream()
            for rep in range(5):
                for i, (T, kk, rn) in enumerate(seq):
                    _call(layer, xs[i % 2], T, kk, rn, outs[h][rep][i], stream=st)
            st.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append((h, repr(e)))

    threads = [threading.Thread(target=drive, args=(h,)) for h in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not any(th.is_alive() for th in threads)
    assert not errors, errors
    torch.cuda.synchronize()
    for h in range(2):
        assert layers[h][0].check() == binding.MOE_OK
        bad = [(rep, seq[i]) for rep in range(5) for i in range(len(seq))
               if not torch.equal(outs[h][rep][i], refs[h][i])]
        assert not bad, (h, bad)
        layers[h][0].close()
