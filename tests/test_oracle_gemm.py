"""Pins for the oracle of the step in the L1 GEMM's epilogue (fp32 NVFP4
quantization, SwiGLU of double accumulators, the float64 GEMM) against exact
rational arithmetic, a 50-digit decimal SwiGLU, and reductions to the
already pinned fused step (one-hot weights make the GEMM a column gather)."""
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

from moe_swiglu_epilogue_gb300 import workloads as W
from test_oracle_pins import _adversarial_blocks, _nearest_f32_of_decimal, exact_block


def test_quantize_f32_against_exact_arithmetic(oracle_mod):
    rng = np.random.default_rng(707)
    blocks = _adversarial_blocks(rng)
    for scale in (1e-3, 0.37, 1.0, 17.0, 3e3):
        for _ in range(40):
            blocks.append((rng.standard_normal(16) * scale).astype(np.float32))
    y = np.stack(blocks).astype(np.float32)
    packed, sf = oracle_mod.quantize_nvfp4_f32(y)
    for i, blk in enumerate(y):
        p, s = exact_block(blk)
        assert sf[i, 0] == s and np.array_equal(packed[i], p), (i, blk)


def test_quantize_f32_equals_the_bf16_quantize_on_bf16_values(oracle_mod):
    x = W.prefill_heavy_tail_quantize(rows=128, K=512, seed=9).data
    p1, s1 = oracle_mod.quantize_nvfp4(x)
    p2, s2 = oracle_mod.quantize_nvfp4_f32(W.bf16_to_f32(x).reshape(x.shape))
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def test_swiglu_f64_reduces_to_the_fp32_form(oracle_mod):
    rng = np.random.default_rng(11)
    g = (rng.standard_normal(5000) * 4).astype(np.float32)
    u = (rng.standard_normal(5000) * 4).astype(np.float32)
    g[:8] = [7.0, -7.0, 7.5, -30.0, 0.0, -0.0, 1e-30, 100.0]
    for L in (7.0, 10.0):
        a = oracle_mod.swiglu_clamped_f64_array(g.astype(np.float64), u.astype(np.float64), L)
        b = oracle_mod.swiglu_clamped_array(g, u, L)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_swiglu_f64_against_decimal(oracle_mod):
    """Double inputs that fp32 cannot hold (accumulator values)."""
    getcontext().prec = 50
    rng = np.random.default_rng(12)
    L = 7.0
    g = rng.standard_normal(600) * 3 + rng.uniform(-1e-7, 1e-7, 600)
    u = rng.standard_normal(600) * 2 + rng.uniform(-1e-7, 1e-7, 600)
    g[:4] = [7.0 + 2.0 ** -40, 7.0 - 2.0 ** -40, -25.123456789, 1e-9]
    u[:4] = [-7.0 - 2.0 ** -40, 6.999999999999, 3.0, -1e-9]
    got = oracle_mod.swiglu_clamped_f64_array(g, u, L)
    for gi, ui, yi in zip(g, u, got):
        a = min(Decimal(float(gi)), Decimal(L))
        b = min(max(Decimal(float(ui)), Decimal(-L)), Decimal(L))
        y = a / (1 + (-a).exp()) * b
        best, runner, undecidable = _nearest_f32_of_decimal(y)
        assert yi == best or (undecidable and yi == runner), (gi, ui, yi, y)


def _selection_case(rng, rows, H, I, offsets):
    x = W.bf16_bits((rng.standard_normal((rows, H)) * 3).astype(np.float32))
    x[0, :8] = W.bf16_bits(np.array([7, -7, 8, -8, 0, -0.0, 1e-3, 60], np.float32))
    E = len(offsets) - 1
    sel = np.stack([rng.integers(0, H, 2 * I) for _ in range(E)])
    w1 = np.zeros((E, 2 * I, H), np.uint16)
    one = W.bf16_bits(np.array([1.0], np.float32))[0]
    for e in range(E):
        w1[e, np.arange(2 * I), sel[e]] = one
    return x, w1, sel


def test_gemm_with_one_hot_weights_is_the_fused_step(oracle_mod):
    """w1[e] row c = unit vector k(e, c): gu[r, c] = x[r, k(e, c)] exactly, so
    the GEMM's output must be the (pinned) fused step on that gathered BF16
    tensor, segment by segment; rows outside the segments stay untouched."""
    rng = np.random.default_rng(13)
    rows, H, I = 40, 64, 128
    offsets = np.array([3, 10, 10, 31, 37], np.int32)     # leading gap, empty expert, tail
    x, w1, sel = _selection_case(rng, rows, H, I, offsets)
    sent_p = np.full((rows, I // 2), 0xA5, np.uint8)
    sent_s = np.full((rows, I // 16), 0x5A, np.uint8)
    p, s = oracle_mod.l1_gemm_swiglu_quantize_nvfp4(x, w1, offsets, 7.0, packed=sent_p, sf=sent_s)
    for e in range(len(offsets) - 1):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        gu = np.ascontiguousarray(x[r0:r1][:, sel[e]])
        rp, rs = oracle_mod.swiglu_quantize_nvfp4(gu, 7.0)
        assert np.array_equal(p[r0:r1], rp) and np.array_equal(s[r0:r1], rs), e
    for r in list(range(0, 3)) + list(range(37, rows)):
        assert np.all(p[r] == 0xA5) and np.all(s[r] == 0x5A)


def test_gemm_accumulators_against_exact_sums(oracle_mod):
    rng = np.random.default_rng(14)
    rows, H, I = 12, 64, 128
    offsets = np.array([0, 5, 12], np.int32)
    x = W.bf16_bits((rng.standard_normal((rows, H)) * 5).astype(np.float32))
    w1 = W.bf16_bits((rng.standard_normal((2, 2 * I, H)) * 0.1).astype(np.float32))
    acc = oracle_mod.l1_gemm_accumulators(x, w1, offsets)
    mag = oracle_mod.l1_gemm_abs_accumulators(x, w1, offsets)
    xf = [[Fraction(float(v)) for v in row] for row in W.bf16_to_f32(x).reshape(rows, H)]
    wf = W.bf16_to_f32(w1).reshape(2, 2 * I, H)
    for r in range(rows):
        e = 0 if r < 5 else 1
        for c in rng.integers(0, 2 * I, 12):
            exact = sum(xf[r][k] * Fraction(float(wf[e, c, k])) for k in range(H))
            absum = sum(abs(xf[r][k] * Fraction(float(wf[e, c, k]))) for k in range(H))
            assert abs(Fraction(acc[r, c]) - exact) <= absum * Fraction(1, 2 ** 40)
            assert abs(Fraction(mag[r, c]) - absum) <= absum * Fraction(1, 2 ** 40)


def test_gemm_deinterleave_pairs_each_output_with_its_gate_and_up(oracle_mod):
    """Gates all 1, up of output c = (c + 1) / 1024: y[c] = silu(1) (c+1)/1024
    by a decimal evaluation, for every column of every group."""
    getcontext().prec = 50
    I = 64
    acc = np.zeros((1, 2 * I))
    c = np.arange(I)
    acc[0, 16 * (c // 8) + c % 8] = 1.0
    acc[0, 16 * (c // 8) + c % 8 + 8] = (c + 1) / 1024
    y = oracle_mod.gemm_swiglu_values(acc, 7.0)[0]
    silu1 = Decimal(1) / (1 + Decimal(-1).exp())
    for ci in range(I):
        best, runner, undecidable = _nearest_f32_of_decimal(silu1 * Decimal(ci + 1) / 1024)
        assert y[ci] == best or (undecidable and y[ci] == runner), ci
