"""Pins for the oracle's extensions (two-level scale, BF16 compat / compact
writer, padded per-expert output, dequantization) against torch's BF16 and
float8_e4m3fn casts, exact rational arithmetic and compositions with the
already pinned single-level functions."""
import numpy as np
import pytest
import torch

from moe_swiglu_epilogue_gb300 import workloads as W
from test_oracle_pins import exact_block, _dense_fp32_below

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)


def torch_bf16_bits(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_round_matches_torch(oracle_mod):
    v = _dense_fp32_below(0x7f000000)[::7]           # all binades, ties and neighbours
    v = np.concatenate([v, -v[::5]])
    want = W.bf16_to_f32(torch_bf16_bits(v))
    got = np.array([oracle_mod.bf16_round(float(x)) for x in v[::997]], np.float32)
    assert np.array_equal(got.view(np.uint32), want[::997].view(np.uint32))


def test_scaled_quantize_reduces_to_single_level(oracle_mod):
    x = W.quantize_normal(rows=64, K=256, seed=5).data
    p1, s1 = oracle_mod.quantize_nvfp4(x)
    p2, s2 = oracle_mod.quantize_nvfp4_scaled(x, 1.0)
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2)
    for k in (-7, -1, 3, 9):                           # power-of-two scale: exact prescaling
        xs = W.bf16_bits(W.bf16_to_f32(x) * np.float32(2.0 ** k))
        assert np.array_equal(W.bf16_to_f32(xs), W.bf16_to_f32(x) * np.float32(2.0 ** k))
        p1, s1 = oracle_mod.quantize_nvfp4(xs)
        p2, s2 = oracle_mod.quantize_nvfp4_scaled(x, 2.0 ** k)
        assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def test_scaled_quantize_against_exact_arithmetic(oracle_mod):
    rng = np.random.default_rng(21)
    x = W.quantize_normal(rows=8, K=64, seed=6).data
    for gs in (0.3711, 17.25, 1e-3 * 3.1, 448.0 * 6 / 5.7):
        gs32 = np.float32(gs)
        p, s = oracle_mod.quantize_nvfp4_scaled(x, gs32)
        v = W.bf16_to_f32(x) * gs32                   # IEEE fp32 product
        for r in range(8):
            for b in range(4):
                ep, es = exact_block(v[r, 16 * b:16 * b + 16])
                assert es == s[r, b] and np.array_equal(ep, p[r, 8 * b:8 * b + 8]), (gs, r, b)


def test_fused_ex_reduces_to_the_plain_step(oracle_mod):
    w = W.fused_normal(rows=40, I=128)
    p1, s1 = oracle_mod.swiglu_quantize_nvfp4(w.data, 7.0)
    p2, s2 = oracle_mod.swiglu_quantize_nvfp4_ex(w.data, 7.0)
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def test_compact_writer_is_the_bf16_rounded_swiglu(oracle_mod):
    w = W.fused_normal(rows=24, I=256)
    y = oracle_mod.swiglu_values(w.data, 7.0)
    assert np.array_equal(oracle_mod.swiglu_bf16(w.data, 7.0), torch_bf16_bits(y))


def test_compat_mode_is_quantize_of_the_compact_tensor(oracle_mod):
    w = W.fused_normal(rows=24, I=256)
    compact = oracle_mod.swiglu_bf16(w.data, 7.0)
    for gs in (1.0, 0.625, 3.3):
        p1, s1 = oracle_mod.quantize_nvfp4_scaled(compact, gs)
        p2, s2 = oracle_mod.swiglu_quantize_nvfp4_ex(w.data, 7.0, global_scale=gs, round_bf16=True)
        assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def test_fused_scaled_against_exact_arithmetic(oracle_mod):
    w = W.fused_normal(rows=4, I=64, seed=9)
    gs = np.float32(5.123)
    p, s = oracle_mod.swiglu_quantize_nvfp4_ex(w.data, 7.0, global_scale=gs)
    y = oracle_mod.swiglu_values(w.data, 7.0) * gs
    for r in range(4):
        for b in range(4):
            ep, es = exact_block(y[r, 16 * b:16 * b + 16])
            assert es == s[r, b] and np.array_equal(ep, p[r, 8 * b:8 * b + 8])


def test_padded_segments_move_rows_and_leave_gaps(oracle_mod):
    w = W.ragged_routing(tokens=64, experts=6, topk=3, I=64)
    rows, I = w.rows, w.width
    counts = np.diff(w.offsets)
    tile = 16
    padded = np.ceil(counts / tile).astype(np.int64) * tile
    out_off = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    out_rows = int(out_off[-1])
    sent_p = np.full((out_rows, I // 2), 0xA5, np.uint8)
    sent_s = np.full((out_rows, I // 16), 0x5A, np.uint8)
    p, s = oracle_mod.swiglu_quantize_nvfp4_ex(w.data, 7.0, w.offsets, out_off, out_rows,
                                               packed=sent_p, sf=sent_s)
    fp, fs = oracle_mod.swiglu_quantize_nvfp4(w.data, 7.0)
    for e in range(len(counts)):
        a, n, o = int(w.offsets[e]), int(counts[e]), int(out_off[e])
        assert np.array_equal(p[o:o + n], fp[a:a + n]) and np.array_equal(s[o:o + n], fs[a:a + n])
        assert np.all(p[o + n:o + padded[e]] == 0xA5) and np.all(s[o + n:o + padded[e]] == 0x5A)
    # destinations past out_rows are skipped, the rest written as before
    short = out_rows - tile
    p2, _ = oracle_mod.swiglu_quantize_nvfp4_ex(w.data, 7.0, w.offsets, out_off, short,
                                                packed=np.full((short, I // 2), 0xA5, np.uint8),
                                                sf=np.full((short, I // 16), 0x5A, np.uint8))
    assert np.array_equal(p2, p[:short])
    # destinations before row 0 are skipped too: shifting every destination
    # 5 rows up drops the first 5 output rows and moves the rest
    p3, s3 = oracle_mod.swiglu_quantize_nvfp4_ex(w.data, 7.0, w.offsets, out_off - 5, out_rows - 5,
                                                 packed=np.full((out_rows - 5, I // 2), 0xA5, np.uint8),
                                                 sf=np.full((out_rows - 5, I // 16), 0x5A, np.uint8))
    assert np.array_equal(p3, p[5:]) and np.array_equal(s3, s[5:])


def test_dequantize_every_nibble_under_every_scale(oracle_mod):
    codes = np.arange(0x7f, dtype=np.uint8)
    nibs = np.arange(16, dtype=np.uint8)
    # one row per code: 16 elements with nibbles 0..15 (8 bytes), one scale
    packed = np.tile((nibs[0::2] | (nibs[1::2] << 4))[None, :], (codes.size, 1))
    sf = codes[:, None]
    out = oracle_mod.dequantize_nvfp4(packed, sf)
    d = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    grid = E2M1[nibs & 7] * np.where(nibs & 8, -1.0, 1.0).astype(np.float32)
    want = grid[None, :] * d[:, None]                  # exact in fp32
    assert np.array_equal(out, torch_bf16_bits(want))
    assert np.array_equal(W.bf16_to_f32(out), want)     # and exact in BF16


def test_dequantize_with_global_scale(oracle_mod):
    x = W.quantize_normal(rows=16, K=128, seed=3).data
    gs = np.float32(2.7)
    p, s = oracle_mod.quantize_nvfp4_scaled(x, gs)
    out = oracle_mod.dequantize_nvfp4(p, s, gs)
    nib = np.stack([p & 15, p >> 4], -1).reshape(16, 128)
    d = torch.from_numpy(s).view(torch.float8_e4m3fn).float().numpy()
    val = E2M1[nib & 7] * np.where(nib & 8, -1.0, 1.0).astype(np.float32) * np.repeat(d, 16, axis=1)
    assert np.array_equal(out, torch_bf16_bits(val / gs))
    # and it approximates x: each element within one E2M1 step of its block scale
    err = np.abs(W.bf16_to_f32(out) - W.bf16_to_f32(x))
    assert np.all(err <= 1.26 * np.repeat(d, 16, axis=1) / gs + 1e-6)


def test_quantize_dequantize_round_trip_of_representable_values(oracle_mod):
    rng = np.random.default_rng(8)
    code = 0x40                                        # d = 2^(8-7) = 2.0
    d = float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).float())
    vals = E2M1[rng.integers(0, 8, (32, 16))] * d * np.where(rng.integers(0, 2, (32, 16)), -1, 1)
    vals[:, 0] = 6 * d                                 # fixes the scale
    x = W.bf16_bits(vals.astype(np.float32))
    p, s = oracle_mod.quantize_nvfp4(x)
    assert np.all(s == code)
    assert np.array_equal(W.bf16_to_f32(oracle_mod.dequantize_nvfp4(p, s)), vals.astype(np.float32))
