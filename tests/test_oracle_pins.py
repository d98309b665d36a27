"""Pins of the CPU oracle against things other than itself.

The oracle restates "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.1
(288 routed + 1 shared expert, independent FFNs) and §3.2.2 (linear router,
softmax, top-8, weighted sum of the 9 expert outputs).  These tests check it
against closed forms, special cases that reduce to library routines (numpy
matmul, scipy softmax, numpy lexsort/bincount, torch float64 matmul and
silu), invariants and a pure-Python brute force, each chosen so that a
plausible slip (dropped shared expert, renormalised weights, gate/up swapped,
a transposed weight, a wrong tie rule, a missing max-subtraction) fails.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from expert_routed_ffn_gemm_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def bits_of(a_f32: np.ndarray) -> np.ndarray:
    """fp32 values that are exact in bf16 -> their bf16 bit patterns."""
    a = np.ascontiguousarray(a_f32, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "values must be exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def f64_of(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_layer(seed, T, d, E, k, F, skew=None):
    shape = synth.LayerShape(T=T, d=d, E=E, k=k, F=F)
    inp = synth.make_inputs(shape, seed=seed, device="cpu", skew=skew)
    return (shape, synth.bf16_bits(inp.x), inp.w_router.numpy(), synth.bf16_bits(inp.w_gate_up),
            synth.bf16_bits(inp.w_down))


def library_forward(x, wr, wgu, wd, k, has_shared=True):
    """The layer recomposed from library routines: numpy matmul for the
    router, scipy softmax, lexsort for the top-k order, torch float64 matmul
    and torch silu for the expert FFNs."""
    X = f64_of(x)
    z = X @ wr.astype(np.float64).T
    p = scipy.special.softmax(z, axis=1)
    T, E = p.shape
    Wgu = torch.from_numpy(f64_of(wgu))
    Wd = torch.from_numpy(f64_of(wd))
    F = Wgu.shape[1] // 2
    Xt = torch.from_numpy(X)
    y = torch.zeros(T, X.shape[1], dtype=torch.float64)
    idx = np.zeros((T, k), np.int64)
    for t in range(T):
        order = np.lexsort((np.arange(E), -p[t]))  # p descending, then index ascending
        idx[t] = order[:k]
    for g in range(E + (1 if has_shared else 0)):
        h = torch.nn.functional.silu(Xt @ Wgu[g, :F].T) * (Xt @ Wgu[g, F:].T)
        o = h @ Wd[g].T
        if g == E:
            y += o
        else:
            wcol = torch.from_numpy(np.where(idx == g, p[np.arange(T)[:, None], idx], 0.0).sum(1))
            y += wcol[:, None] * o
    return y.numpy(), idx, p


def test_uniform_router_picks_lowest_indices():
    # W_r = 0: every logit is 0, p = 1/E exactly, and the tie rule
    # (lower expert index first) makes idx = 0..k-1 for every token.
    shape, x, wr, wgu, wd = rand_layer(1, T=9, d=64, E=12, k=5, F=32)
    wr = np.zeros_like(wr)
    idx, w, gap, p = oracle.route(x, wr, 5, want_p=True)
    assert np.all(p == 1.0 / 12)
    assert np.all(idx == np.arange(5)[None, :])
    assert np.all(w == 1.0 / 12)
    assert np.all(gap == 0.0)


def test_all_experts_selected_when_k_equals_E():
    shape, x, wr, wgu, wd = rand_layer(2, T=7, d=64, E=6, k=6, F=32)
    idx, w, gap, p = oracle.route(x, wr, 6, want_p=True)
    for t in range(7):
        assert sorted(idx[t].tolist()) == list(range(6))
        assert np.all(np.diff(w[t]) <= 0)
    assert np.all(np.isinf(gap))
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)


def test_softmax_matches_scipy_and_sums_to_one():
    shape, x, wr, wgu, wd = rand_layer(3, T=33, d=128, E=40, k=4, F=32)
    idx, w, gap, p = oracle.route(x, wr, 4, want_p=True)
    z = f64_of(x) @ wr.astype(np.float64).T
    np.testing.assert_allclose(p, scipy.special.softmax(z, axis=1), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-12)


def test_softmax_is_stable_for_huge_logits():
    # Logits of order 1e4: exp() without subtracting the maximum overflows.
    shape, x, wr, wgu, wd = rand_layer(4, T=5, d=64, E=10, k=3, F=32)
    wr = wr * 1.0e4
    idx, w, gap, p = oracle.route(x, wr, 3, want_p=True)
    assert np.all(np.isfinite(p))
    z = f64_of(x) @ wr.astype(np.float64).T
    np.testing.assert_allclose(p, scipy.special.softmax(z, axis=1), rtol=1e-9, atol=1e-300)


def test_topk_order_matches_lexsort():
    shape, x, wr, wgu, wd = rand_layer(5, T=50, d=64, E=31, k=7, F=32)
    idx, w, gap, p = oracle.route(x, wr, 7, want_p=True)
    for t in range(50):
        order = np.lexsort((np.arange(31), -p[t]))
        assert idx[t].tolist() == order[:7].tolist()
        assert w[t].tolist() == p[t, order[:7]].tolist()
        assert gap[t] == p[t, order[6]] - p[t, order[7]]


def test_topk_ties_inside_selection():
    # Duplicate router rows give exactly equal logits: the lower index of
    # each equal pair must come first.
    shape, x, wr, wgu, wd = rand_layer(6, T=20, d=64, E=8, k=4, F=32)
    wr = np.concatenate([wr[:4], wr[:4]], axis=0)  # expert e+4 duplicates expert e
    idx, w, gap, p = oracle.route(x, wr, 4, want_p=True)
    for t in range(20):
        order = np.lexsort((np.arange(8), -p[t]))
        assert idx[t].tolist() == order[:4].tolist()
        for e in range(4):
            assert p[t, e] == p[t, e + 4]
        # each chosen duplicate pair appears lower index first
        pos = {e: j for j, e in enumerate(idx[t].tolist())}
        for e in range(4):
            if e in pos and e + 4 in pos:
                assert pos[e] < pos[e + 4]


def test_dispatch_invariants():
    shape, x, wr, wgu, wd = rand_layer(7, T=200, d=64, E=24, k=3, F=32)
    idx, w, gap, _ = oracle.route(x, wr, 3)
    counts, offsets, perm = oracle.dispatch(idx, 24)
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=24))
    np.testing.assert_array_equal(offsets[:-1], np.concatenate([[0], np.cumsum(counts)]))
    assert offsets[-1] == offsets[-2] + 200
    assert sorted(perm.tolist()) == list(range(600))
    e_of = idx.ravel()[perm]
    t_of = perm // 3
    keys = list(zip(e_of.tolist(), t_of.tolist()))
    assert keys == sorted(keys)
    for e in range(24):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(idx.ravel()[seg] == e)


def test_expert_ffn_matches_torch():
    # d != F so that a transposed W_d or a gate/up swap cannot pass.
    shape, x, wr, wgu, wd = rand_layer(8, T=6, d=96, E=3, k=1, F=40)
    Wgu = torch.from_numpy(f64_of(wgu))
    Wd = torch.from_numpy(f64_of(wd))
    X = torch.from_numpy(f64_of(x))
    for g in range(4):
        ref = (torch.nn.functional.silu(X @ Wgu[g, :40].T) * (X @ Wgu[g, 40:].T)) @ Wd[g].T
        got = oracle.expert_ffn(x, wgu, wd, g)
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_shared_only_output_is_dense_swiglu():
    # All routed down-projections zero: the layer is the shared SwiGLU FFN.
    shape, x, wr, wgu, wd = rand_layer(9, T=12, d=64, E=10, k=3, F=32)
    wd = wd.copy()
    wd[:10] = 0
    y = oracle.forward(x, wr, wgu, wd, 3)
    X = torch.from_numpy(f64_of(x))
    Wgu = torch.from_numpy(f64_of(wgu))
    ref = (torch.nn.functional.silu(X @ Wgu[10, :32].T) * (X @ Wgu[10, 32:].T)) @ torch.from_numpy(f64_of(wd[10])).T
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("k", [1, 3, 10])
def test_forward_matches_library_recomposition(k):
    shape, x, wr, wgu, wd = rand_layer(10 + k, T=17, d=64, E=10, k=k, F=48)
    y = oracle.forward(x, wr, wgu, wd, k)
    ref, idx_ref, _ = library_forward(x, wr, wgu, wd, k)
    idx, _, _, _ = oracle.route(x, wr, k)
    np.testing.assert_array_equal(idx, idx_ref)
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-13)


def test_forward_without_shared_expert():
    shape = synth.LayerShape(T=9, d=64, E=6, k=2, F=32, has_shared=False)
    inp = synth.make_inputs(shape, seed=21)
    x, wr = synth.bf16_bits(inp.x), inp.w_router.numpy()
    wgu, wd = synth.bf16_bits(inp.w_gate_up), synth.bf16_bits(inp.w_down)
    y = oracle.forward(x, wr, wgu, wd, 2, has_shared=False)
    ref, _, _ = library_forward(x, wr, wgu, wd, 2, has_shared=False)
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-13)


def test_weights_are_not_renormalised():
    # With k < E the routed part is sum p_j * FFN_j with raw softmax
    # probabilities; renormalising over the top-k would scale it by
    # 1/sum_j p_j > 1.  Zero the shared expert and compare the ratio.
    shape, x, wr, wgu, wd = rand_layer(30, T=8, d=64, E=12, k=2, F=32)
    wd = wd.copy()
    wd[12] = 0
    y = oracle.forward(x, wr, wgu, wd, 2)
    idx, w, _, _ = oracle.route(x, wr, 2)
    for t in range(8):
        o = [oracle.expert_ffn(x, wgu, wd, int(e), rows=np.array([t], np.int32))[0] for e in idx[t]]
        np.testing.assert_allclose(y[t], w[t, 0] * o[0] + w[t, 1] * o[1], rtol=1e-12, atol=1e-14)
        assert w[t].sum() < 1.0


def test_linear_in_one_experts_down_weights():
    shape, x, wr, wgu, wd = rand_layer(31, T=16, d=64, E=8, k=2, F=32)
    y1 = oracle.forward(x, wr, wgu, wd, 2)
    wd2 = wd.copy()
    # doubling a bf16 value is exact: add 1 to the exponent field
    wd2[3] = (wd2[3].astype(np.uint32) + np.where(wd2[3] & 0x7F80, 0x80, 0)).astype(np.uint16)
    y2 = oracle.forward(x, wr, wgu, wd2, 2)
    idx, w, _, _ = oracle.route(x, wr, 2)
    o3 = oracle.expert_ffn(x, wgu, wd, 3)
    extra = np.where(idx == 3, w, 0.0).sum(1)[:, None] * o3
    np.testing.assert_allclose(y2 - y1, extra, rtol=1e-9, atol=1e-13)


def test_token_permutation_equivariance():
    shape, x, wr, wgu, wd = rand_layer(32, T=13, d=64, E=7, k=3, F=32)
    perm = np.random.default_rng(0).permutation(13)
    y = oracle.forward(x, wr, wgu, wd, 3)
    yp = oracle.forward(np.ascontiguousarray(x[perm]), wr, wgu, wd, 3)
    np.testing.assert_array_equal(yp, y[perm])


def test_token_subset_and_selection_override():
    shape, x, wr, wgu, wd = rand_layer(33, T=20, d=64, E=9, k=2, F=32)
    y = oracle.forward(x, wr, wgu, wd, 2)
    idx, _, _, _ = oracle.route(x, wr, 2)
    toks = np.array([19, 0, 7], np.int32)
    np.testing.assert_array_equal(oracle.forward(x, wr, wgu, wd, 2, tokens=toks), y[toks])
    np.testing.assert_array_equal(oracle.forward(x, wr, wgu, wd, 2, tokens=toks, sel=idx[toks]), y[toks])


def test_closed_form_two_experts():
    # d=2, E=2, k=1, F=1, x = (1, 0): every dot product picks one weight.
    # z = (1, 0) -> p0 = e/(1+e); expert 0 wins.  Expert e has gate row
    # (a_e, .), up row (c_e, .), down column (u_e, v_e); the shared expert
    # likewise.  y = p0 * silu(a0) c0 (u0, v0) + silu(a_s) c_s (u_s, v_s).
    x = bits_of(np.array([[1.0, 0.0]], np.float32))
    wr = np.array([[1.0, 0.0], [0.0, 0.0]], np.float32)
    gu = np.array([[[2.0, 5.0], [0.5, -3.0]],      # expert 0: gate (2,5), up (0.5,-3)
                   [[-1.0, 1.0], [4.0, 1.0]],      # expert 1
                   [[-0.25, 7.0], [3.0, 2.0]]],    # shared: gate (-0.25,7), up (3,2)
                  np.float32)
    dn = np.array([[[1.5], [-2.0]], [[9.0], [9.0]], [[0.75], [0.125]]], np.float32)
    y = oracle.forward(x, wr, bits_of(gu), bits_of(dn), 1)

    def silu(v):
        return v / (1.0 + math.exp(-v))

    p0 = math.e / (1.0 + math.e)
    h0 = silu(2.0) * 0.5
    hs = silu(-0.25) * 3.0
    expect = [p0 * h0 * 1.5 + hs * 0.75, p0 * h0 * -2.0 + hs * 0.125]
    np.testing.assert_allclose(y[0], expect, rtol=1e-14, atol=0)


def brute_force(x, wr, wgu, wd, k, has_shared=True):
    """Per-token, per-expert pure-Python loops with a full sorted()."""
    X = f64_of(x).tolist()
    Wr = wr.astype(np.float64).tolist()
    Wgu = f64_of(wgu).tolist()
    Wd = f64_of(wd).tolist()
    T, d, E, F = len(X), len(X[0]), len(Wr), len(Wgu[0]) // 2
    ys, sels = [], []
    for t in range(T):
        z = [sum(X[t][i] * Wr[e][i] for i in range(d)) for e in range(E)]
        m = max(z)
        ex = [math.exp(v - m) for v in z]
        s = sum(ex)
        p = [v / s for v in ex]
        ranked = sorted(range(E), key=lambda e: (-p[e], e))
        chosen = ranked[:k]
        sels.append(chosen)
        y = [0.0] * d
        groups = [(e, p[e]) for e in chosen] + ([(E, 1.0)] if has_shared else [])
        for g, wgt in groups:
            h = []
            for f in range(F):
                gv = sum(Wgu[g][f][i] * X[t][i] for i in range(d))
                uv = sum(Wgu[g][F + f][i] * X[t][i] for i in range(d))
                h.append(gv / (1.0 + math.exp(-gv)) * uv)
            for o in range(d):
                y[o] += wgt * sum(Wd[g][o][f] * h[f] for f in range(F))
        ys.append(y)
    return np.array(ys), np.array(sels)


def test_brute_force_tiny():
    shape, x, wr, wgu, wd = rand_layer(40, T=5, d=16, E=6, k=2, F=8)
    y_b, sel_b = brute_force(x, wr, wgu, wd, 2)
    idx, _, _, _ = oracle.route(x, wr, 2)
    np.testing.assert_array_equal(idx, sel_b)
    np.testing.assert_allclose(oracle.forward(x, wr, wgu, wd, 2), y_b, rtol=1e-12, atol=1e-14)


def test_tiny_workload_routing_properties():
    # The tiny workload (T=64, d=256, 16+1 experts, top-2, width 128).
    inp = synth.make_inputs(synth.TINY, seed=0)
    x, wr = synth.bf16_bits(inp.x), inp.w_router.numpy()
    idx, w, gap, p = oracle.route(x, wr, 2, want_p=True)
    assert idx.shape == (64, 2)
    assert np.all(idx[:, 0] != idx[:, 1])
    assert np.all(w[:, 0] >= w[:, 1])
    assert np.all(gap >= 0)
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-12)


def test_skew_recipe_shape():
    # Zipf-skewed routing: masked experts never chosen, hot experts far above
    # the mean (checked on a reduced d to keep the CPU suite quick).
    shape = synth.LayerShape(T=1024, d=256, E=288, k=8, F=128)
    inp = synth.make_inputs(shape, seed=0, skew="zipf")
    idx, _, _, _ = oracle.route(synth.bf16_bits(inp.x), inp.w_router.numpy(), 8)
    counts = np.bincount(idx.ravel(), minlength=288)
    assert (counts == 0).sum() >= 40
    assert counts.max() / counts.mean() > 4.0


# ---- per-call routing variants and routing statistics ----------------------

def library_forward_renorm(x, wr, wgu, wd, k):
    """library_forward with the k weights divided by their sum."""
    X = f64_of(x)
    p = scipy.special.softmax(X @ wr.astype(np.float64).T, axis=1)
    T, E = p.shape
    Wgu = torch.from_numpy(f64_of(wgu))
    Wd = torch.from_numpy(f64_of(wd))
    F = Wgu.shape[1] // 2
    Xt = torch.from_numpy(X)
    y = torch.zeros(T, X.shape[1], dtype=torch.float64)
    idx = np.stack([np.lexsort((np.arange(E), -p[t]))[:k] for t in range(T)])
    wsel = p[np.arange(T)[:, None], idx]
    wsel = wsel / wsel.sum(axis=1, keepdims=True)
    for g in range(E + 1):
        o = (torch.nn.functional.silu(Xt @ Wgu[g, :F].T) * (Xt @ Wgu[g, F:].T)) @ Wd[g].T
        if g == E:
            y += o
        else:
            y += torch.from_numpy(np.where(idx == g, wsel, 0.0).sum(1))[:, None] * o
    return y.numpy()


@pytest.mark.parametrize("k", [2, 5])
def test_renormalized_forward_matches_library(k):
    shape, x, wr, wgu, wd = rand_layer(50 + k, T=11, d=64, E=9, k=k, F=32)
    y = oracle.forward(x, wr, wgu, wd, k, renormalize=True)
    np.testing.assert_allclose(y, library_forward_renorm(x, wr, wgu, wd, k), rtol=1e-11, atol=1e-13)


def test_renormalize_changes_nothing_when_k_equals_E():
    shape, x, wr, wgu, wd = rand_layer(55, T=6, d=64, E=5, k=5, F=32)
    np.testing.assert_allclose(oracle.forward(x, wr, wgu, wd, 5, renormalize=True),
                               oracle.forward(x, wr, wgu, wd, 5), rtol=1e-13, atol=1e-15)


def test_route_stats_uniform_router_closed_form():
    # W_r = 0: p = 1/E for every expert, the tie rule picks experts 0..k-1, so
    # all T*k rows land in group 0: f = (1, 0, ...), p_g = 1/G, L_EP = 1,
    # max/mean load = E/k, entropy = ln E, E - k experts without rows.
    shape, x, wr, wgu, wd = rand_layer(56, T=10, d=64, E=24, k=3, F=32)
    counts, f, pg, summary = oracle.route_stats(x, np.zeros_like(wr), 3, 6)
    np.testing.assert_array_equal(counts, np.array([10, 10, 10] + [0] * 21))
    np.testing.assert_array_equal(f, np.array([1.0, 0, 0, 0, 0, 0]))
    np.testing.assert_allclose(pg, 1.0 / 6, rtol=1e-14)
    np.testing.assert_allclose(summary, [1.0, 24 / 3, math.log(24), 21], rtol=1e-13)


def test_route_stats_brute_force():
    shape, x, wr, wgu, wd = rand_layer(57, T=7, d=16, E=8, k=2, F=8)
    counts, f, pg, summary = oracle.route_stats(x, wr, 2, 4)
    X = f64_of(x).tolist()
    W = wr.astype(np.float64).tolist()
    c = [0] * 8
    mass = [0.0] * 4
    ent = 0.0
    for t in range(7):
        z = [sum(X[t][i] * W[e][i] for i in range(16)) for e in range(8)]
        m = max(z)
        ex = [math.exp(v - m) for v in z]
        s = sum(ex)
        p = [v / s for v in ex]
        for e in sorted(range(8), key=lambda e: (-p[e], e))[:2]:
            c[e] += 1
        for e in range(8):
            mass[e // 2] += p[e]
            ent -= p[e] * math.log(p[e])
    fb = [(c[2 * g] + c[2 * g + 1]) / 14 for g in range(4)]
    pb = [mv / 7 for mv in mass]
    assert counts.tolist() == c
    np.testing.assert_allclose(f, fb, rtol=1e-14)
    np.testing.assert_allclose(pg, pb, rtol=1e-12)
    np.testing.assert_allclose(summary, [4 * sum(a * b for a, b in zip(fb, pb)), max(c) / (14 / 8), ent / 7,
                                         c.count(0)], rtol=1e-12)
