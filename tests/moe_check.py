"""Shared checks of the CUDA path against the CPU oracle (test helpers).

Tolerances (stated once, used by every parity test):
* routing: expert indices and the dispatch permutation bit-exact, except for
  tokens whose oracle gap between the k-th and (k+1)-th probability is below
  NEAR_TIE (1e-6); for those the GPU's choice must still be a valid top-k
  under the oracle's probabilities to within NEAR_TIE, and the output is
  compared with the oracle recomputed for the GPU's choice;
* probabilities: within the fp32 error bound derived in ``prob_bound``;
* layer output: max |y_gpu - y_oracle| <= OUT_TOL * RMS(y_oracle).
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
    """Per-token bound on |p_gpu - p_oracle| for an fp32 router.

    Each logit is a dot product of length d summed in fp32 (at most d terms
    in one chain): its error is at most gamma_d * sum_i |x_i w_i|, with
    gamma_n = n u / (1 - n u) and u = 2^-24.  log p_e = z_e - logsumexp(z)
    then moves by at most 2 max_e dz_e.  The fp32 softmax adds: rounding of
    z - max (relative error of exp(.) up to range * u, range = max z - min z),
    expf itself (2 ulp), the E-term sum ((E - 1) u) and the division (u).
    """
    xf = (x_bits[tokens].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wa = np.abs(w_router.astype(np.float64))
    d = xf.shape[1]
    E = wa.shape[0]
    u = 2.0 ** -24
    gamma = d * u / (1 - d * u)
    dz = gamma * (np.abs(xf) @ wa.T)  # [n_tok, E]
    p = o_p[tokens]
    with np.errstate(divide="ignore"):
        rng = np.log(p.max(axis=1)) - np.log(np.maximum(p.min(axis=1), 1e-300))
    dzm = dz.max(axis=1)
    rel = np.expm1(2.0 * dzm) + (rng + 4 + E) * u
    return rel[:, None] * p + 1e-30


def check_routing(x_bits, w_router, k, idx, prob, gap=None, perm=None, offsets=None, has_shared=True):
    """Returns (near-tie token list, oracle idx)."""
    T = x_bits.shape[0]
    E = w_router.shape[0]
    o_idx, o_w, o_gap, o_p = oracle.route(x_bits, w_router, k, want_p=True)
    near = np.nonzero(o_gap < NEAR_TIE)[0]
    sure = o_gap >= NEAR_TIE
    assert idx.shape == (T, k)
    np.testing.assert_array_equal(idx[sure], o_idx[sure])
    # every token: k distinct experts in range, ordered by oracle probability
    assert idx.min() >= 0 and idx.max() < E
    for t in near:
        assert len(set(idx[t].tolist())) == k
        kth = o_w[t, k - 1]
        assert np.all(o_p[t, idx[t]] >= kth - NEAR_TIE)
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


def check_output(x_bits, w_router, wgu_bits, wd_bits, k, y_gpu, sel, tokens=None, has_shared=True, tol=OUT_TOL):
    """Compares y_gpu (rows = tokens) with the oracle for the GPU's selection."""
    T = x_bits.shape[0]
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    y_ref = oracle.forward(x_bits, w_router, wgu_bits, wd_bits, k, has_shared=has_shared, tokens=tokens,
                           sel=np.ascontiguousarray(sel[tokens]))
    y = y_gpu.astype(np.float64)
    assert np.all(np.isfinite(y))
    err = np.abs(y - y_ref).max() if y.size else 0.0
    rms = np.sqrt((y_ref ** 2).mean()) if y.size else 1.0
    assert err <= tol * rms, f"max|err| {err:.4e} > {tol} * rms {rms:.4e} (ratio {err / rms:.3e})"
    return err / rms


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
