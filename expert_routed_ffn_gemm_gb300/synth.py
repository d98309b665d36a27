"""Seeded synthetic inputs for the sparse-MoE layer.

This module only draws random numbers and arranges them into the layer's
input tensors; it holds none of the layer's arithmetic.  It serves both the
CUDA path and the CPU oracle in the tests and the benchmark, which then
consume the very same tensors.

Recipe (one torch.Generator seeded with ``seed`` on ``device``, drawn in the
order x, W_r, W_gu, W_d, then the skew ranking):

* x      [T, d]          N(0, 1)    fp32 -> bf16 (round to nearest even)
* W_r    [E, d]          N(0, 0.02) fp32
* W_gu   [G, 2F, d]      N(0, 0.02) fp32 -> bf16, gate rows then up rows
* W_d    [G, d, F]       N(0, 0.02) fp32 -> bf16
with G = E + 1 (group E is the always-on shared expert).

Skewed routing is an input structure, not a change of the method: feature
0 of every token is set to 1 and column 0 of W_r to a per-expert bias
b_e = -alpha * s * ln(rank_e) with s = 1.1 (a Zipf(s) ranking drawn as a
seeded permutation), and experts whose rank is above ``n_live`` get
b_e = -30 so that they are never chosen.  The router's logits then carry
b_e exactly, with no bias term in the layer itself.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class LayerShape:
    """Shape of one MoE layer and the number of tokens of one call."""

    T: int
    d: int
    E: int
    k: int
    F: int
    has_shared: bool = True

    @property
    def groups(self) -> int:
        return self.E + (1 if self.has_shared else 0)

    def with_tokens(self, T: int) -> "LayerShape":
        return replace(self, T=T)


# Named workloads: a tiny layer the oracle runs in well under a second, and
# the Step 3.5 Flash layer (d=4096, 288 routed + 1 shared expert, top-8,
# expert width 1280) at decode, prefill and skewed token counts.
TINY = LayerShape(T=64, d=256, E=16, k=2, F=128)
FLASH_DECODE = LayerShape(T=128, d=4096, E=288, k=8, F=1280)
FLASH_PREFILL = FLASH_DECODE.with_tokens(8192)
FLASH_SKEW = FLASH_DECODE.with_tokens(4096)
FLASH_SWEEP_T = (1, 8, 32, 512, 2048, 32768)

SKEW_ALPHA = 0.35
SKEW_S = 1.1
SKEW_LIVE = 248
SKEW_ALPHA_LITERAL = 2.0


@dataclass
class LayerInputs:
    shape: LayerShape
    x: torch.Tensor  # [T, d] bf16
    w_router: torch.Tensor  # [E, d] fp32
    w_gate_up: torch.Tensor  # [G, 2F, d] bf16
    w_down: torch.Tensor  # [G, d, F] bf16


def _normal_bf16(gen, shape, std, device, chunk_rows=None):
    """N(0, std) drawn in fp32 and rounded to bf16, drawn slice by slice along
    dim 0 when ``chunk_rows`` is set (bounds the fp32 temporary)."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    n0 = shape[0]
    step = max(1, n0 if not chunk_rows else chunk_rows)
    for s in range(0, n0, step):
        e = min(n0, s + step)
        tmp = torch.randn((e - s,) + tuple(shape[1:]), generator=gen, device=device,
                          dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        out[s:e].copy_(tmp)
        del tmp
    return out


def make_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_inputs(shape: LayerShape, seed: int = 0, device="cpu", skew: str | None = None,
                weights_only: bool = False) -> LayerInputs:
    """Draw one layer's inputs.  ``skew`` is None, "zipf" (alpha 0.35, 40
    experts never chosen) or "zipf_literal" (alpha 2, no masking)."""
    device = torch.device(device)
    gen = make_generator(seed, device)
    T, d, E, F, G = shape.T, shape.d, shape.E, shape.F, shape.groups
    x = _normal_bf16(gen, (max(T, 0), d), 1.0, device)
    w_router = torch.randn((E, d), generator=gen, device=device, dtype=torch.float32).mul_(0.02)
    w_gate_up = _normal_bf16(gen, (G, 2 * F, d), 0.02, device, chunk_rows=8)
    w_down = _normal_bf16(gen, (G, d, F), 0.02, device, chunk_rows=8)
    if skew is not None:
        ranks = torch.randperm(E, generator=gen, device=device).to(torch.float64) + 1.0
        if skew == "zipf":
            alpha, live = SKEW_ALPHA, SKEW_LIVE
        elif skew == "zipf_literal":
            alpha, live = SKEW_ALPHA_LITERAL, E
        else:
            raise ValueError(f"unknown skew {skew!r}")
        bias = -alpha * SKEW_S * torch.log(ranks)
        bias = torch.where(ranks > live, torch.full_like(bias, -30.0), bias)
        w_router[:, 0] = bias.to(torch.float32)
        if T > 0:
            x[:, 0] = 1.0
    if weights_only:
        x = x[:0]
    return LayerInputs(shape, x, w_router, w_gate_up, w_down)


def skewed_router(w_router: torch.Tensor, seed: int, skew: str = "zipf") -> torch.Tensor:
    """A copy of ``w_router`` whose column 0 is the skew bias of the recipe
    above, from its own seeded ranking (for weights that already exist; pair
    it with tokens from ``make_tokens(..., skew=skew)``)."""
    E = w_router.shape[0]
    ranks = torch.randperm(E, generator=make_generator(seed, "cpu")).to(torch.float64) + 1.0
    if skew == "zipf":
        alpha, live = SKEW_ALPHA, SKEW_LIVE
    elif skew == "zipf_literal":
        alpha, live = SKEW_ALPHA_LITERAL, E
    else:
        raise ValueError(f"unknown skew {skew!r}")
    bias = -alpha * SKEW_S * torch.log(ranks)
    bias = torch.where(ranks > live, torch.full_like(bias, -30.0), bias)
    w = w_router.clone()
    w[:, 0] = bias.to(torch.float32).to(w.device)
    return w


def make_tokens(shape: LayerShape, seed: int, device="cpu", skew: str | None = None) -> torch.Tensor:
    """A fresh x [T, d] bf16 for an existing set of weights (for repeated
    steps that must not reuse one batch).  Feature 0 is 1 under skew."""
    gen = make_generator(seed, device)
    x = _normal_bf16(gen, (shape.T, shape.d), 1.0, device)
    if skew is not None and shape.T > 0:
        x[:, 0] = 1.0
    return x


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor, as a host numpy array."""
    import numpy as np

    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def expected_touched(shape: LayerShape) -> float:
    """Expected number of routed experts with at least one row when every
    expert is equally likely (used only to size work estimates)."""
    if shape.T <= 0:
        return 0.0
    return shape.E * (1.0 - (1.0 - shape.k / shape.E) ** shape.T)


__all__ = [
    "LayerShape", "LayerInputs", "TINY", "FLASH_DECODE", "FLASH_PREFILL", "FLASH_SKEW",
    "FLASH_SWEEP_T", "make_inputs", "make_tokens", "skewed_router", "bf16_bits", "expected_touched",
]
