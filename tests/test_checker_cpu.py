"""The parity checks (moe_check.py) reject wrong results, on the CPU.

The oracle's own routing, dispatch and output, stored the way the GPU path
stores them (probabilities and gap as fp32, y as bf16), must pass the checks;
the same results with one planted error each must fail them; and the valid
alternatives the checks exempt (experts with exactly equal probabilities, in
either order or at the top-k boundary) must pass.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gemm_gb300 import synth

from moe_check import OUT_TOL, PROB_GUARD, check_output, check_routing, host_bits, prob_bound

SHAPE = synth.LayerShape(T=48, d=128, E=16, k=4, F=64)


def _bf16(y: np.ndarray) -> np.ndarray:
    return torch.from_numpy(y).to(torch.bfloat16).double().numpy()


@pytest.fixture(scope="module")
def layer():
    inp = synth.make_inputs(SHAPE, seed=77)
    xb, wr, wgu, wd = host_bits(inp)
    idx, w, gap, _ = oracle.route(xb, wr, SHAPE.k, want_p=True)
    _, offsets, perm = oracle.dispatch(idx, SHAPE.E)
    offsets[SHAPE.E + 1] = offsets[SHAPE.E] + SHAPE.T
    y = _bf16(oracle.forward(xb, wr, wgu, wd, SHAPE.k))
    return dict(xb=xb, wr=wr, wgu=wgu, wd=wd, idx=idx, prob=w.astype(np.float32), gap=gap.astype(np.float32),
                perm=perm, offsets=offsets, y=y, o_gap=gap)


def _routing(L, **over):
    a = dict(idx=L["idx"], prob=L["prob"], gap=L["gap"], perm=L["perm"], offsets=L["offsets"])
    a.update(over)
    return check_routing(L["xb"], L["wr"], SHAPE.k, a["idx"], a["prob"], a["gap"], a["perm"], a["offsets"])


def _output(L, y, sel=None):
    return check_output(L["xb"], L["wr"], L["wgu"], L["wd"], SHAPE.k, y, L["idx"] if sel is None else sel)


def test_the_oracles_own_results_pass(layer):
    _routing(layer)
    assert _output(layer, layer["y"]) < OUT_TOL


def _clear_token(L):
    # a token whose k-th and (k+1)-th probabilities are far apart
    return int(np.argmax(L["o_gap"]))


def test_another_expert_is_rejected(layer):
    t = _clear_token(layer)
    p = oracle.route(layer["xb"], layer["wr"], SHAPE.k + 1)[0]
    idx = layer["idx"].copy()
    idx[t, -1] = p[t, -1]  # the (k+1)-th expert in place of the k-th
    with pytest.raises(AssertionError):
        _routing(layer, idx=idx)


def test_slots_swapped_across_a_clear_gap_are_rejected(layer):
    t = int(np.argmax(layer["prob"][:, 0] - layer["prob"][:, 1]))
    idx = layer["idx"].copy()
    idx[t, [0, 1]] = idx[t, [1, 0]]
    with pytest.raises(AssertionError):
        _routing(layer, idx=idx)
    prob = layer["prob"].copy()
    prob[t, [0, 1]] = prob[t, [1, 0]]
    with pytest.raises(AssertionError):
        _routing(layer, idx=idx, prob=prob)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_a_probability_beyond_its_bound_is_rejected(layer, sign):
    # three times the derived fp32 bound (a worst case, linear in 3d: about
    # 1.5e-4 of p at d = 128) away from the oracle's value
    _, _, _, p = oracle.route(layer["xb"], layer["wr"], SHAPE.k, want_p=True)
    t = 5
    e = layer["idx"][t, 2]
    b = prob_bound(layer["xb"], layer["wr"], np.array([t]), p)[0, e]
    prob = layer["prob"].copy()
    prob[t, 2] = np.float32(p[t, e] + sign * 3 * b)
    prob[t] = np.sort(prob[t])[::-1]  # still ordered along the slots
    with pytest.raises(AssertionError):
        _routing(layer, prob=prob)


def test_a_bf16_router_is_rejected_where_the_derived_bound_is_loose():
    # d = 4096: the derived bound allows some 17 % of p; probabilities from a
    # bf16 copy of W_r (errors of a few 1e-3 of p) must still fail, on the
    # empirical guard
    shape = synth.LayerShape(T=16, d=4096, E=32, k=4, F=64)
    inp = synth.make_inputs(shape, seed=79)
    xb, wr, _, _ = host_bits(inp)
    idx, w, gap, p = oracle.route(xb, wr, shape.k, want_p=True)
    _, off, perm = oracle.dispatch(idx, shape.E)
    off[shape.E + 1] = off[shape.E] + shape.T
    check_routing(xb, wr, shape.k, idx, w.astype(np.float32), gap.astype(np.float32), perm, off)
    wr16 = torch.from_numpy(wr).to(torch.bfloat16).float().numpy()
    _, _, _, p16 = oracle.route(xb, wr16, shape.k, want_p=True)
    prob16 = p16[np.arange(shape.T)[:, None], idx]
    rel = np.abs(prob16 - w) / w
    assert rel.max() > PROB_GUARD  # the bf16 router's error
    assert np.all(np.abs(prob16 - w) <= prob_bound(xb, wr, np.arange(shape.T), p)[np.arange(shape.T)[:, None], idx])
    with pytest.raises(AssertionError, match="guard"):
        check_routing(xb, wr, shape.k, idx, np.sort(prob16, axis=1)[:, ::-1].astype(np.float32),
                      gap.astype(np.float32), perm, off)


def test_dispatch_errors_are_rejected(layer):
    perm = layer["perm"].copy()
    e0, e1 = 0, 1
    i, j = layer["offsets"][e0], layer["offsets"][e1]  # first rows of two experts
    perm[[i, j]] = perm[[j, i]]
    with pytest.raises(AssertionError):
        _routing(layer, perm=perm)
    perm = layer["perm"].copy()
    lo, hi = layer["offsets"][3], layer["offsets"][4]
    assert hi - lo >= 2
    perm[[lo, lo + 1]] = perm[[lo + 1, lo]]  # token order inside one expert
    with pytest.raises(AssertionError):
        _routing(layer, perm=perm)
    for pos, delta in ((3, 1), (SHAPE.E + 1, -1)):
        off = layer["offsets"].copy()
        off[pos] += delta
        with pytest.raises(AssertionError):
            _routing(layer, offsets=off)


def test_a_wrong_gap_is_rejected(layer):
    t = _clear_token(layer)
    gap = layer["gap"].copy()
    gap[t] = -gap[t]
    with pytest.raises(AssertionError):
        _routing(layer, gap=gap)


def test_output_errors_are_rejected(layer):
    L = layer
    y = L["y"]
    rms = np.sqrt((y ** 2).mean())
    bad = y.copy()
    bad[7, 11] += 1.5 * OUT_TOL * rms  # one element over the bound
    with pytest.raises(AssertionError):
        _output(L, bad)
    bad = y.copy()
    bad[[0, 1]] = bad[[1, 0]]  # two tokens' rows swapped
    with pytest.raises(AssertionError):
        _output(L, bad)
    bad = y.copy()
    bad[3, 0] = np.nan
    with pytest.raises(AssertionError):
        _output(L, bad)
    E = SHAPE.E
    no_shared = _bf16(oracle.forward(L["xb"], L["wr"], L["wgu"][:E], L["wd"][:E], SHAPE.k, has_shared=False))
    with pytest.raises(AssertionError):
        _output(L, no_shared)
    renormalised = _bf16(oracle.forward(L["xb"], L["wr"], L["wgu"], L["wd"], SHAPE.k, renormalize=True))
    with pytest.raises(AssertionError):
        _output(L, renormalised)
    other = oracle.route(L["xb"], L["wr"], SHAPE.k + 1)[0]
    sel = L["idx"].copy()
    sel[:, -1] = other[:, -1]  # every token's k-th expert replaced by its (k+1)-th
    with pytest.raises(AssertionError):
        _output(L, _bf16(oracle.forward(L["xb"], L["wr"], L["wgu"], L["wd"], SHAPE.k, sel=sel)))


def test_exact_ties_are_accepted_in_either_order_and_at_the_boundary():
    # experts 14 and 15 with the same router row, far above the others: every
    # token gives them the same probability.  With k = 2 they are the top two
    # (a slot-order tie); with k = 1 they tie at the boundary.  The oracle puts
    # 14 first; 15 first is an equally valid result and must pass, with the
    # output compared to the oracle's for that choice.
    inp = synth.make_inputs(SHAPE, seed=78)
    wr = inp.w_router.clone()
    wr[14] = wr[15] = torch.sign(inp.x[0].float()) * 0.5
    inp = synth.LayerInputs(SHAPE, inp.x, wr, inp.w_gate_up, inp.w_down)
    xb, wr_h, wgu, wd = host_bits(inp)
    for k in (2, 1):
        idx, w, gap, p = oracle.route(xb, wr_h, k, want_p=True)
        tied = np.nonzero(np.isin(idx[:, 0], [14]) & (p[:, 14] == p[:, 15]))[0]
        assert tied.size > 0
        swapped = idx.copy()
        if k == 2:
            swapped[tied] = swapped[tied][:, ::-1]
        else:
            swapped[tied, 0] = 15
        _, off, perm = oracle.dispatch(swapped, SHAPE.E)
        off[SHAPE.E + 1] = off[SHAPE.E] + SHAPE.T
        prob = p[np.arange(SHAPE.T)[:, None], swapped].astype(np.float32)
        check_routing(xb, wr_h, k, swapped, prob, gap.astype(np.float32), perm, off)
        y = _bf16(oracle.forward(xb, wr_h, wgu, wd, k, sel=swapped))
        check_output(xb, wr_h, wgu, wd, k, y, swapped)
