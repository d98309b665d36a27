"""Shared checks of the CUDA path against the CPU oracle (test helpers).

Tolerances (stated once, used by every parity test):
* routing: expert indices and the dispatch permutation bit-exact, except for
  tokens whose oracle gap between the k-th and (k+1)-th probability is below
  NEAR_TIE (1e-6); for those the GPU's choice must still be a valid top-k
  under the oracle's probabilities to within NEAR_TIE, and the output is
  compared with the oracle recomputed for the GPU's choice;
* probabilities: within the fp32 error bound derived in ``prob_bound``;
* layer output: |y_gpu - y_oracle| <= OUT_TOL * RMS(y_oracle) everywhere
  when y is fp32.  When y is stored as bf16, the storage itself moves each
  value by up to half a bf16 ulp of y (2^-9 relative), which past about
  5 RMS alone exceeds 2e-2 RMS; that half ulp of y_oracle is added to the
  bound element by element, so the check measures the computation and not
  the output format.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from expert_routed_ffn_gemm_gb300 import synth

NEAR_TIE = 1e-6
OUT_TOL = 2e-2


def to_dev(inp: synth.LayerInputs, dev):
    return (inp.x.to(dev), inp.w_router.to(dev), inp.w_gate_up.to(dev), inp.w_down.to(dev))


def host_bits(inp: synth.LayerInputs):
    return (synth.bf16_bits(inp.x), inp.w_router.detach().cpu().numpy(), synth.bf16_bits(inp.w_gate_up),
            synth.bf16_bits(inp.w_down))


def prob_bound(x_bits, w_router, tokens, o_p):
    """Per-token bound on |p_gpu - p_oracle| for the fp32-accurate router.

    Each logit is x . W_r computed as x . hi + x . mid + x . lo over three
    bf16 slices of W_r (residual below 2^-24 |w|), every product exact, summed
    in fp32: at most n = 3d terms, each addition off by at most 2u (u = 2^-24,
    2u allowing accumulators that truncate), so |dz| <= gamma * sum_i |x_i w_i|
    with gamma = 2 n u / (1 - 2 n u) + u.  log p_e = z_e - logsumexp(z) then
    moves by at most 2 max_e dz_e.  The fp32 softmax adds: rounding of
    z - max (relative error of exp(.) up to range * u, range = max z - min z),
    expf itself (2 ulp), the E-term sum ((E - 1) u) and the division (u).
    """
    xf = (x_bits[tokens].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wa = np.abs(w_router.astype(np.float64))
    d = xf.shape[1]
    E = wa.shape[0]
    u = 2.0 ** -24
    n = 3 * d
    gamma = 2 * n * u / (1 - 2 * n * u) + u
    dz = gamma * (np.abs(xf) @ wa.T)  # [n_tok, E]
    p = o_p[tokens]
    with np.errstate(divide="ignore"):
        rng = np.log(p.max(axis=1)) - np.log(np.maximum(p.min(axis=1), 1e-300))
    dzm = dz.max(axis=1)
    rel = np.expm1(2.0 * dzm) + (rng + 4 + E) * u
    return rel[:, None] * p + 1e-30


def check_routing(x_bits, w_router, k, idx, prob, gap=None, perm=None, offsets=None, has_shared=True):
    """Returns (near-tie token list, oracle idx).

    Near-ties come in two kinds.  Boundary: the oracle's gap between the
    k-th and (k+1)-th probability is below NEAR_TIE, so the chosen set itself
    is decided by rounding.  Order: two adjacent probabilities inside the
    top-k are closer than NEAR_TIE, so only their order (the slot index j)
    is decided by rounding.  Every other token must match the oracle's idx
    bit for bit; order near-ties must match as a set, with an order that is
    non-increasing under the oracle's probabilities to within NEAR_TIE;
    boundary near-ties must pick k distinct experts none of which is more
    than NEAR_TIE below the oracle's k-th probability.
    """
    T = x_bits.shape[0]
    E = w_router.shape[0]
    o_idx, o_w, o_gap, o_p = oracle.route(x_bits, w_router, k, want_p=True)
    boundary = o_gap < NEAR_TIE
    order = np.zeros(T, bool)
    if k > 1:
        order = (np.diff(o_w, axis=1) > -NEAR_TIE).any(axis=1) & ~boundary
    sure = ~boundary & ~order
    assert idx.shape == (T, k)
    np.testing.assert_array_equal(idx[sure], o_idx[sure])
    assert idx.min() >= 0 and idx.max() < E
    for t in np.nonzero(order)[0]:
        assert sorted(idx[t].tolist()) == sorted(o_idx[t].tolist())
        assert np.all(np.diff(o_p[t, idx[t]]) <= NEAR_TIE)
    for t in np.nonzero(boundary)[0]:
        assert len(set(idx[t].tolist())) == k
        kth = o_w[t, k - 1]
        assert np.all(o_p[t, idx[t]] >= kth - NEAR_TIE)
    near = np.nonzero(~sure)[0]
    # probabilities of the chosen experts
    tok = np.arange(T)
    bound = prob_bound(x_bits, w_router, tok, o_p)
    p_ref = o_p[tok[:, None], idx]
    b_sel = bound[tok[:, None], idx]
    assert np.all(np.abs(prob.astype(np.float64) - p_ref) <= b_sel), \
        f"prob error {np.abs(prob - p_ref).max():.3e}"
    if gap is not None:
        gb = 2 * bound.max(axis=1)
        g_ref = np.where(np.isinf(o_gap), np.inf, o_gap)
        fin = ~np.isinf(g_ref) & sure
        assert np.all(np.abs(gap[fin].astype(np.float64) - g_ref[fin]) <= gb[fin] + 1e-12)
        assert np.all(np.isinf(gap[np.isinf(g_ref)]))
    if perm is not None:
        c_ref, off_ref, perm_ref = oracle.dispatch(idx, E)
        np.testing.assert_array_equal(offsets[:E + 1], off_ref[:E + 1])
        assert offsets[E + 1] == off_ref[E] + (T if has_shared else 0)
        np.testing.assert_array_equal(perm, perm_ref)
    return near, o_idx


def half_ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |v| (8 significand bits): 2^(floor(log2|v|) - 8)."""
    _, e = np.frexp(np.abs(v))  # |v| = m 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 9)


def check_output(x_bits, w_router, wgu_bits, wd_bits, k, y_gpu, sel, tokens=None, has_shared=True, tol=OUT_TOL,
                 out_bf16=True, fp8=None):
    """Compares y_gpu (rows = tokens) with the oracle for the GPU's selection;
    returns max|err| / RMS.  fp8 = (q_gate_up, s_gate_up, q_down, s_down):
    the expert weights are E4M3 codes with row scales (wgu_bits / wd_bits
    unused)."""
    T = x_bits.shape[0]
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    sel_t = np.ascontiguousarray(sel[tokens])
    if fp8 is None:
        y_ref = oracle.forward(x_bits, w_router, wgu_bits, wd_bits, k, has_shared=has_shared, tokens=tokens,
                               sel=sel_t)
    else:
        y_ref = oracle.forward_fp8(x_bits, w_router, *fp8, k, has_shared=has_shared, tokens=tokens, sel=sel_t)
    y = y_gpu.astype(np.float64)
    assert np.all(np.isfinite(y))
    if not y.size:
        return 0.0
    diff = np.abs(y - y_ref)
    rms = np.sqrt((y_ref ** 2).mean())
    bound = tol * rms + (half_ulp_bf16(y_ref) if out_bf16 else 0.0)
    worst = np.unravel_index(np.argmax(diff - bound), diff.shape)
    assert np.all(diff <= bound), (f"|err| {diff[worst]:.4e} > bound {bound[worst] if out_bf16 else bound:.4e} "
                                   f"at {worst} (y_ref {y_ref[worst]:.4e}, rms {rms:.4e})")
    return diff.max() / rms


def sample_tokens(T, idx, n_random, seed, extra=()):
    """A seeded sample of tokens, plus `extra`, plus one token per expert used."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(T, n_random), replace=False).tolist())
    pick.update(int(t) for t in extra)
    first = {}
    for t in range(T):
        for e in idx[t]:
            first.setdefault(int(e), t)
    pick.update(first.values())
    return np.array(sorted(pick), dtype=np.int32)


def cpu(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()
