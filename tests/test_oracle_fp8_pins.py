"""Pins of the oracle's FP8 pieces (E4M3 codec, per-row quantiser, forward
with E4M3 expert weights) against things other than themselves.

The FP8 weights follow "Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §8.1
(FP8/FP16 mixed-precision inference); the page names no format, so the
reading is OCP FP8 E4M3 codes with one fp32 scale per weight row.  The pins:
values the OCP E4M3 definition fixes (1.0, 448, the smallest normal and
subnormal, NaN), torch's own float8_e4m3fn conversion (a library routine),
round-to-nearest-even at every midpoint, the quantiser's error bound, and the
fp8 forward reducing exactly to the (separately pinned) bf16 forward when
every dequantised weight is a bf16 value.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_gemm_gb300 import synth


def test_e4m3_values_fixed_by_the_format():
    v = oracle.e4m3_decode(np.array([0x38, 0x40, 0x3F, 0x7E, 0xFE, 0x08, 0x07, 0x01, 0x00, 0x80, 0x77],
                                    np.uint8))
    assert list(v[:3]) == [1.0, 2.0, 1.875]
    assert v[3] == 448.0 and v[4] == -448.0          # largest finite magnitude
    assert v[5] == 2.0 ** -6                         # smallest normal
    assert v[6] == 7 * 2.0 ** -9                     # largest subnormal
    assert v[7] == 2.0 ** -9                         # smallest subnormal
    assert v[8] == 0.0 and np.signbit(v[9])          # +0, -0
    assert v[10] == 240.0
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), ~fin)
    np.testing.assert_array_equal(ours[fin], ref[fin])


def test_e4m3_encode_matches_torch_in_range_and_saturates_beyond():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 100, 4000), rng.normal(0, 1e-2, 4000),
                        rng.uniform(-448, 448, 4000)]).astype(np.float32)
    ours = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)
    big = np.array([448.0, 449.0, 464.0, 1e6, -500.0], np.float32)
    assert list(oracle.e4m3_encode(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_e4m3_rounds_midpoints_to_even_codes():
    codes = np.arange(0, 0x7E, dtype=np.uint8)          # 0 .. 447 (positive, finite)
    v = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)                       # codes are ordered by value
    mid = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (v[:-1] + v[1:]) / 2)  # midpoints exact in fp32
    got = oracle.e4m3_encode(mid)
    even = np.where(codes % 2 == 0, codes, codes + 1)
    np.testing.assert_array_equal(got, even)
    # just off the midpoint: the nearer code
    up = np.nextafter(mid, np.float32(np.inf))
    dn = np.nextafter(mid, np.float32(-np.inf))
    np.testing.assert_array_equal(oracle.e4m3_encode(up), codes + 1)
    np.testing.assert_array_equal(oracle.e4m3_encode(dn), codes)


def test_quantiser_scale_and_error_bound():
    rng = np.random.default_rng(1)
    w = rng.normal(0, 0.02, (64, 512)).astype(np.float32)
    w[3] = 0.0                                          # a zero row
    w[5, 17] = 3.0                                      # an outlier
    bits = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    wb = torch.from_numpy(w).to(torch.bfloat16).double().numpy()
    q, s = oracle.quantize_e4m3(bits)
    amax = np.abs(wb).max(axis=1)
    np.testing.assert_array_equal(s, (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32))
    assert s[3] == 0 and np.all(q[3] == 0)
    deq = oracle.e4m3_decode(q) * s[:, None].astype(np.float64)
    # the row maximum maps to the largest code
    top = np.abs(wb).argmax(axis=1)
    for r in range(64):
        if r != 3:
            assert q[r, top[r]] & 0x7F == 0x7E
    # nearest-value bound: half a code spacing, 2^-4 relative (normals) or 2^-10 * s (subnormals)
    bound = np.maximum(np.abs(wb) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert np.all(np.abs(deq - wb) <= bound)


def test_forward_fp8_reduces_to_the_bf16_forward():
    # With power-of-two scales every dequantised weight (4 significant bits)
    # is a bf16 value, so the FP8 forward must equal the bf16 forward on those
    # values exactly (same summation order in the oracle).
    shape = synth.LayerShape(T=24, d=256, E=8, k=2, F=128)
    inp = synth.make_inputs(shape, seed=3)
    rng = np.random.default_rng(2)
    G = shape.E + 1
    q_gu = rng.integers(0, 256, (G, 2 * shape.F, shape.d), dtype=np.uint8)
    q_d = rng.integers(0, 256, (G, shape.d, shape.F), dtype=np.uint8)
    q_gu[(q_gu & 0x7F) == 0x7F] = 0x00  # no NaN codes
    q_d[(q_d & 0x7F) == 0x7F] = 0x00
    s_gu = np.ldexp(1.0, rng.integers(-12, -6, (G, 2 * shape.F))).astype(np.float32)
    s_d = np.ldexp(1.0, rng.integers(-12, -6, (G, shape.d))).astype(np.float32)
    w_gu = oracle.e4m3_decode(q_gu) * s_gu[:, :, None]
    w_d = oracle.e4m3_decode(q_d) * s_d[:, :, None]
    to_bits = lambda a: torch.from_numpy(a.astype(np.float32)).view(torch.int32).numpy().view(np.uint32)
    b_gu, b_d = to_bits(w_gu), to_bits(w_d)
    assert np.all((b_gu & 0xFFFF) == 0) and np.all((b_d & 0xFFFF) == 0)
    xb = synth.bf16_bits(inp.x)
    wr = inp.w_router.numpy()
    y8 = oracle.forward_fp8(xb, wr, q_gu, s_gu, q_d, s_d, shape.k)
    y16 = oracle.forward(xb, wr, (b_gu >> 16).astype(np.uint16), (b_d >> 16).astype(np.uint16), shape.k)
    np.testing.assert_array_equal(y8, y16)


def test_forward_fp8_of_quantised_weights_tracks_bf16_forward():
    # Quantising N(0, 0.02) weights keeps the layer output within the E4M3
    # rounding (relative 2^-4 per weight, averaged over d and F terms).
    shape = synth.LayerShape(T=16, d=256, E=8, k=2, F=128)
    inp = synth.make_inputs(shape, seed=4)
    xb = synth.bf16_bits(inp.x)
    wr = inp.w_router.numpy()
    gu_bits, d_bits = synth.bf16_bits(inp.w_gate_up), synth.bf16_bits(inp.w_down)
    q_gu, s_gu = oracle.quantize_e4m3(gu_bits)
    q_d, s_d = oracle.quantize_e4m3(d_bits)
    y8 = oracle.forward_fp8(xb, wr, q_gu, s_gu, q_d, s_d, shape.k)
    y16 = oracle.forward(xb, wr, gu_bits, d_bits, shape.k)
    rel = np.sqrt(((y8 - y16) ** 2).mean()) / np.sqrt((y16 ** 2).mean())
    assert 1e-3 < rel < 5e-2


def test_two_term_e4m3_rows_reproduce_bf16_values():
    # The reading behind the FP8 kernels' activations: with s the largest power
    # of two keeping s*max|x| <= 448, hi = e4m3(s*x) and lo = e4m3(s*x - hi)
    # give hi + lo == s*x exactly for a bf16 x whenever |s*x| >= 2^-2 (the
    # remainder of an 8-bit significand after rounding to 4 bits has at most 4
    # bits, and its lowest bit stays on E4M3's 2^-9 grid), and within 2^-10
    # below that.  Checked with the oracle's codec (pinned above) on bf16 rows
    # spanning many binades.
    rng = np.random.default_rng(11)
    rows = rng.standard_normal((64, 512)) * np.exp2(rng.integers(-30, 30, size=(64, 1)))
    rows *= np.exp2(rng.integers(-12, 3, size=rows.shape))  # entries far below the row maximum
    x = torch.from_numpy(rows.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    amax = np.abs(x).max(axis=1, keepdims=True)
    e = np.floor(np.log2(448.0 / amax))
    s = np.exp2(e)
    assert np.all(s * amax <= 448.0) and np.all(2 * s * amax > 448.0)
    v = x * s  # exact: power-of-two scaling
    hi = oracle.e4m3_decode(oracle.e4m3_encode(v.astype(np.float32)))
    lo = oracle.e4m3_decode(oracle.e4m3_encode((v - hi).astype(np.float32)))
    err = np.abs(hi + lo - v)
    big = np.abs(v) >= 0.25
    assert big.sum() > 1000 and (~big).sum() > 1000
    assert np.all(err[big] == 0.0)
    assert np.all(err[~big] <= 2.0 ** -10)
