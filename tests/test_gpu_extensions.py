"""GPU parity of the extensions (two-level scale, BF16 compat, compact
writer, padded per-expert rows, dequantization) with the oracle, through the
C ABI. All are exact definitions, so every comparison is bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import moe_swiglu_epilogue_gb300 as M
from moe_swiglu_epilogue_gb300 import workloads as W

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from moe_swiglu_epilogue_gb300 import build
    build.build()
    oracle.build()
    M.load_library()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


GS = (1.0, 0.37109375, 3.3, 448.0 * 6.0 / 71.5)


@pytest.mark.parametrize("gs", GS)
def test_quantize_scaled_bit_exact(gs):
    for w in (W.quantize_normal(rows=256, K=2048, seed=11),
              W.prefill_heavy_tail_quantize(rows=512, K=1024)):
        p, s = M.moe_nvfp4_quantize_scaled(dev(w.data), gs)
        rp, rs = oracle.quantize_nvfp4_scaled(w.data, gs)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp)


def test_quantize_scaled_edge_blocks_bit_exact():
    rng = np.random.default_rng(51)
    x = parity.quantize_edge_blocks(rng, 12000).reshape(-1, 256)
    for gs in (0.5, 0.7, 1.3):
        p, s = M.moe_nvfp4_quantize_scaled(dev(x), gs)
        rp, rs = oracle.quantize_nvfp4_scaled(x, gs)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp)


@pytest.mark.parametrize("gs", GS)
@pytest.mark.parametrize("compat", [False, True])
def test_fused_ex_bit_exact(gs, compat):
    w = W.fused_normal(rows=256, I=2048, seed=3)
    p, s = M.moe_swiglu_nvfp4_quantize_ex(dev(w.data), w.clamp_L, global_scale=gs,
                                         round_to_bf16=compat)
    rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data, w.clamp_L, global_scale=gs, round_bf16=compat)
    assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp)


def test_fused_ex_defaults_equal_the_plain_step():
    w = W.prefill_heavy_tail(rows=256, I=3072)
    p1, s1 = M.moe_swiglu_nvfp4_quantize_ex(dev(w.data), w.clamp_L)
    p2, s2 = M.moe_swiglu_nvfp4_quantize(dev(w.data), w.clamp_L)
    assert torch.equal(p1, p2) and torch.equal(s1, s2)


def test_fused_ex_near_tie_blocks_bit_exact():
    rng = np.random.default_rng(78)
    blocks, _ = parity.fused_near_tie_blocks(rng, 1024, 7.0)
    gu = blocks.reshape(-1, 8 * 32)                       # I = 128
    for gs, compat in ((1.0, True), (0.8125, False), (2.5, True)):
        p, s = M.moe_swiglu_nvfp4_quantize_ex(dev(gu), 7.0, global_scale=gs, round_to_bf16=compat)
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(gu, 7.0, global_scale=gs, round_bf16=compat)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp)


@pytest.mark.parametrize("I", [64, 2048])
def test_padded_segments_bit_exact_and_gaps_untouched(I):
    w = W.ragged_routing(tokens=256, experts=16, topk=4, I=I, pad_rows=9)
    counts = np.diff(w.offsets)
    tile = 128
    padded = np.ceil(counts / tile).astype(np.int64) * tile
    out_off = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    out_rows = int(out_off[-1])
    for gs, compat in ((1.0, False), (1.7, True)):
        sent_p = np.full((out_rows, I // 2), 0xA5, np.uint8)
        sent_s = np.full((out_rows, I // 16), 0x5A, np.uint8)
        p, s = M.moe_swiglu_nvfp4_quantize_ex(
            dev(w.data), w.clamp_L, torch.from_numpy(w.offsets).cuda(), gs, compat,
            torch.from_numpy(out_off).cuda(), out_rows, torch.from_numpy(sent_p.copy()).cuda(),
            torch.from_numpy(sent_s.copy()).cuda())
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data, w.clamp_L, w.offsets, out_off, out_rows,
                                                 gs, compat, packed=sent_p, sf=sent_s)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp)
        assert np.any(rp == 0xA5)                          # gaps exist and stayed


@pytest.mark.parametrize("I", [16, 48, 2048])
def test_padded_segments_empty_single_row_and_offset_start(I):
    """Hand-made segments: a nonzero first offset, empty and single-row
    segments, a long one; output segments padded to 16 rows with gaps. I = 16
    and 48 put several rows (and segment ends) inside one 64-block chunk."""
    offsets = np.array([5, 5, 6, 6, 6, 40, 41, 300, 300, 301, 333], np.int32)
    w = W.fused_normal(rows=340, I=I, seed=12)
    counts = np.diff(offsets)
    out_off = np.concatenate([[3], 3 + np.cumsum((counts + 15) // 16 * 16 + 2)]).astype(np.int32)
    out_rows = int(out_off[-1]) + 7
    for gs, compat in ((1.0, False), (1.3, False), (0.9, True)):
        sent_p = np.full((out_rows, I // 2), 0xA5, np.uint8)
        sent_s = np.full((out_rows, I // 16), 0x5A, np.uint8)
        p, s = M.moe_swiglu_nvfp4_quantize_ex(
            dev(w.data), w.clamp_L, torch.from_numpy(offsets).cuda(), gs, compat,
            torch.from_numpy(out_off).cuda(), out_rows, torch.from_numpy(sent_p.copy()).cuda(),
            torch.from_numpy(sent_s.copy()).cuda())
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data, w.clamp_L, offsets, out_off, out_rows,
                                                 gs, compat, packed=sent_p, sf=sent_s)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp), (gs, compat)


@pytest.mark.parametrize("I", [48, 2048])
def test_padded_destinations_outside_the_output_are_skipped(I):
    """Segment 0 starts 4 rows before the output and the last one runs past
    out_rows: those rows are skipped, every other row lands, gaps stay."""
    offsets = np.array([0, 10, 25, 40], np.int32)
    out_off = np.array([-4, 12, 30, 45], np.int32)
    out_rows = 40
    w = W.fused_normal(rows=40, I=I, seed=13)
    for gs, compat in ((1.0, False), (1.3, False), (1.0, True)):
        sent_p = np.full((out_rows, I // 2), 0xA5, np.uint8)
        sent_s = np.full((out_rows, I // 16), 0x5A, np.uint8)
        p, s = M.moe_swiglu_nvfp4_quantize_ex(
            dev(w.data), w.clamp_L, torch.from_numpy(offsets).cuda(), gs, compat,
            torch.from_numpy(out_off).cuda(), out_rows, torch.from_numpy(sent_p.copy()).cuda(),
            torch.from_numpy(sent_s.copy()).cuda())
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data, w.clamp_L, offsets, out_off, out_rows,
                                                 gs, compat, packed=sent_p, sf=sent_s)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp), (gs, compat)
        assert np.all(rp[6:12] == 0xA5) and np.all(rp[27:30] == 0xA5)


@pytest.mark.parametrize("I", [64, 1024])
def test_padded_many_tiny_segments(I):
    """3000 segments of 0 to 4 rows (many empty): with I = 64 a 64-block
    chunk spans 16 rows and several segment ends, so threads step and bisect
    through the offsets all the time; output segments padded to 4 rows with
    random gaps."""
    rng = np.random.default_rng(41)
    counts = rng.integers(0, 5, 3000)
    offsets = np.concatenate([[7], 7 + np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1]) + 5
    gaps = rng.integers(0, 3, 3000)
    out_off = np.concatenate([[0], np.cumsum((counts + 3) // 4 * 4 + gaps)]).astype(np.int32)
    out_rows = int(out_off[-1])
    w = W.fused_normal(rows=rows, I=I, seed=42)
    for gs, compat in ((1.0, False), (0.8, True)):
        sent_p = np.full((out_rows, I // 2), 0xA5, np.uint8)
        sent_s = np.full((out_rows, I // 16), 0x5A, np.uint8)
        p, s = M.moe_swiglu_nvfp4_quantize_ex(
            dev(w.data), w.clamp_L, torch.from_numpy(offsets).cuda(), gs, compat,
            torch.from_numpy(out_off).cuda(), out_rows, torch.from_numpy(sent_p.copy()).cuda(),
            torch.from_numpy(sent_s.copy()).cuda())
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data, w.clamp_L, offsets, out_off, out_rows,
                                                 gs, compat, packed=sent_p, sf=sent_s)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp), (gs, compat)


@pytest.mark.parametrize("L", [7.3, 0.3, 1234.567])
def test_extensions_with_a_clamp_not_representable_in_bf16(L):
    """The extension kernels' fp32-clamp instantiations: two-level, BF16
    compat (gs = 1 and not) and the compact writer, bit for bit."""
    w = W.fused_normal(rows=96, I=1024, seed=32, L=L)
    for gs, compat in ((1.0, False), (1.25, False), (1.0, True), (0.7, True)):
        p, s = M.moe_swiglu_nvfp4_quantize_ex(dev(w.data), L, global_scale=gs, round_to_bf16=compat)
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data, L, global_scale=gs, round_bf16=compat)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp), (gs, compat)
    out = M.moe_swiglu_bf16(dev(w.data), L)
    assert np.array_equal(bits(out), oracle.swiglu_bf16(w.data, L))
    offsets = np.array([3, 40, 41, 90], np.int32)         # padded output, both quantize modes
    out_off = np.array([0, 48, 64, 128], np.int32)
    for gs, compat in ((1.25, False), (1.0, True)):
        sent_p = np.full((128, 512), 0xA5, np.uint8)
        sent_s = np.full((128, 64), 0x5A, np.uint8)
        p, s = M.moe_swiglu_nvfp4_quantize_ex(
            dev(w.data), L, torch.from_numpy(offsets).cuda(), gs, compat, torch.from_numpy(out_off).cuda(), 128,
            torch.from_numpy(sent_p.copy()).cuda(), torch.from_numpy(sent_s.copy()).cuda())
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data, L, offsets, out_off, 128, gs, compat,
                                                 packed=sent_p, sf=sent_s)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp), ("padded", gs, compat)


def test_compact_writer_bit_exact():
    for w in (W.fused_normal(rows=512, I=2048, seed=4), W.prefill_heavy_tail(rows=256, I=3072),
              W.edge_structured(rows=128, I=4096)):
        out = M.moe_swiglu_bf16(dev(w.data), w.clamp_L)
        assert np.array_equal(bits(out), oracle.swiglu_bf16(w.data, w.clamp_L))


def test_compact_writer_and_compat_near_bf16_midpoints():
    """Every output within 8 fp32 ulps of a BF16 rounding midpoint: the
    fast pass cannot decide these, so each goes through the definition."""
    rng = np.random.default_rng(91)
    blocks, dist = parity.near_bf16_midpoint_blocks(rng, 512, 7.0)
    assert dist.max() <= 8 and np.count_nonzero(dist <= 1) > 0
    gu = blocks.reshape(-1, 8 * 32)                       # I = 128
    out = M.moe_swiglu_bf16(dev(gu), 7.0)
    assert np.array_equal(bits(out), oracle.swiglu_bf16(gu, 7.0))
    for gs in (1.0, 1.7):
        p, s = M.moe_swiglu_nvfp4_quantize_ex(dev(gu), 7.0, global_scale=gs, round_to_bf16=True)
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(gu, 7.0, global_scale=gs, round_bf16=True)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp)


def test_compact_writer_and_compat_results_near_underflow():
    """Results below 2^-100 (tiny and subnormal BF16 ups or gates): whole
    blocks of them, and a few of them beside normal results, through the
    compact writer and compat at global scales 1, 1.7, 2^86 and 2^110 (where
    they reach values that matter). No mode re-decides them separately: the
    BF16 midpoint test decides them as it decides normal values."""
    rng = np.random.default_rng(93)
    nblk = 512
    g = rng.normal(0.0, 2.0, (nblk, 16)).astype(np.float32)
    u = rng.normal(0.0, 1.0, (nblk, 16)).astype(np.float32)
    tiny = np.ldexp(rng.uniform(1.0, 2.0, (nblk, 16)), rng.integers(-133, -100, (nblk, 16))).astype(np.float32)
    tiny *= np.where(rng.random((nblk, 16)) < 0.5, -1.0, 1.0).astype(np.float32)
    kind = np.arange(nblk) % 4
    u = np.where((kind == 0)[:, None], tiny, u)                         # whole blocks tiny
    few = (kind == 1)[:, None] & (rng.random((nblk, 16)) < 0.8)
    u = np.where(few, tiny, u)                                          # tiny beside normal
    g = np.where(((kind == 2)[:, None]) & (rng.random((nblk, 16)) < 0.5), tiny, g)   # tiny gates
    gb = W.bf16_bits(g)
    ub = W.bf16_bits(u)
    gu = W.interleave_gate_up(gb, ub).reshape(-1, 8 * 32)
    out = M.moe_swiglu_bf16(dev(gu), 7.0)
    assert np.array_equal(bits(out), oracle.swiglu_bf16(gu, 7.0))
    for gs in (1.0, 1.7, 2.0 ** 86, 2.0 ** 110):
        p, s = M.moe_swiglu_nvfp4_quantize_ex(dev(gu), 7.0, global_scale=gs, round_to_bf16=True)
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(gu, 7.0, global_scale=gs, round_bf16=True)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp), gs


def test_compact_writer_and_compat_subnormal_results_near_bf16_midpoints():
    """Results in the fp32 subnormal range and just above it (ups with
    exponent field 0..3, every BF16 gate with 1/8 <= |g| <= 16) whose fp32
    value lies within 48 ulps of a BF16 rounding midpoint, found with the
    oracle: the fast value's error there is the window's relative error plus
    half an ulp for the underflowing product, and the midpoint test alone
    must decide them (no separate re-decision of results near underflow)."""
    allg = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    gv = W.bf16_to_f32(allg)
    gates = allg[np.isfinite(gv) & (np.abs(gv) <= 16.0) & (np.abs(gv) >= 0.125)]
    ups = np.array([sg | (e << 7) | m for sg in (0, 0x8000) for e in range(4) for m in range(128)], np.uint16)
    ups = ups[(ups & 0x7FFF) != 0]
    g_all = np.repeat(gates, ups.size)
    u_all = np.tile(ups, gates.size)
    n = g_all.size - g_all.size % 16
    y = oracle.swiglu_values(W.interleave_gate_up(g_all[:n].reshape(-1, 16), u_all[:n].reshape(-1, 16)),
                             7.0).ravel()
    low = (y.astype(np.float32).view(np.uint32) & 0xFFFF).astype(np.int64)
    pick = np.flatnonzero((np.abs(low - 0x8000) <= 48) & (y != 0))
    assert pick.size > 1000 and np.count_nonzero(np.abs(y[pick]) < 2.0 ** -126) > 500
    pick = pick[:pick.size - pick.size % 16]
    gu = W.interleave_gate_up(g_all[pick].reshape(-1, 16), u_all[pick].reshape(-1, 16))
    gu = gu[:gu.shape[0] - gu.shape[0] % 8].reshape(-1, 8 * 32)                # I = 128
    out = M.moe_swiglu_bf16(dev(gu), 7.0)
    assert np.array_equal(bits(out), oracle.swiglu_bf16(gu, 7.0))
    for gs in (1.0, 2.0 ** 110):
        p, s = M.moe_swiglu_nvfp4_quantize_ex(dev(gu), 7.0, global_scale=gs, round_to_bf16=True)
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(gu, 7.0, global_scale=gs, round_bf16=True)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp), gs


def test_compact_writer_and_compat_near_bf16_midpoints_negative_gates():
    """The per-block tolerance grows with the most negative gate; here every
    gate is in [-16, -4] and every output sits next to a BF16 midpoint."""
    rng = np.random.default_rng(92)
    blocks, dist = parity.near_bf16_midpoint_blocks(rng, 256, 7.0, gate_range=(-16.0, -4.0))
    gu = blocks.reshape(-1, 8 * 32)
    out = M.moe_swiglu_bf16(dev(gu), 7.0)
    assert np.array_equal(bits(out), oracle.swiglu_bf16(gu, 7.0))
    for gs in (1.0, 0.6):
        p, s = M.moe_swiglu_nvfp4_quantize_ex(dev(gu), 7.0, global_scale=gs, round_to_bf16=True)
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(gu, 7.0, global_scale=gs, round_bf16=True)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp)


def test_per_gate_silu_bound_holds_for_every_bf16_gate():
    """The BF16 decisions' per-block tolerance rests on the fast silu's
    relative error being at most c0 + c1 max(-a, 0) units of 2^-24 for every
    BF16 gate a >= -16 (c0, c1 read from the kernel source). Measured
    exhaustively with up = 1 (an exact product) and L = 100."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "moe_swiglu_epilogue_gb300", "csrc", "moe_nvfp4.cu")).read()
    c0 = float(re.search(r"constexpr float kSiluErrUlps0 = ([0-9.]+)f;", src).group(1))
    c1 = float(re.search(r"constexpr float kSiluErrUlpsPerGate = ([0-9.]+)f;", src).group(1))
    allg = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    gv = W.bf16_to_f32(allg)
    gates = allg[np.isfinite(gv) & (gv >= -16.0)]
    n = gates.size - gates.size % 16
    up = W.bf16_bits(np.ones(n, np.float32))
    gu = W.interleave_gate_up(gates[:n].reshape(-1, 16), up.reshape(-1, 16))
    y_fast = M.moe_swiglu_fast_values(dev(gu), 100.0).cpu().numpy().ravel().astype(np.float64)
    y_ref = oracle.swiglu_values(gu, 100.0).ravel().astype(np.float64)
    a = W.bf16_to_f32(gates[:n]).astype(np.float64)
    nz = y_ref != 0
    rel = np.abs(y_fast[nz] - y_ref[nz]) / np.abs(y_ref[nz]) / 2.0 ** -24
    bound = c0 + c1 * np.maximum(-a[nz], 0.0)
    assert np.all(rel <= bound), float((rel - bound).max())


def test_compact_writer_ragged_rows_untouched():
    w = W.ragged_routing(tokens=128, experts=8, topk=4, I=256, pad_rows=13)
    sent = torch.full((w.rows, w.width), 3.0, dtype=torch.bfloat16, device="cuda")
    out = M.moe_swiglu_bf16(dev(w.data), w.clamp_L, torch.from_numpy(w.offsets).cuda(), sent)
    ref = oracle.swiglu_bf16(w.data, w.clamp_L, w.offsets,
                             out=np.full((w.rows, w.width), 0x4040, np.uint16))
    assert np.array_equal(bits(out), ref)


def test_compact_then_quantize_equals_compat():
    w = W.fused_normal(rows=256, I=1024, seed=8)
    compact = M.moe_swiglu_bf16(dev(w.data), w.clamp_L)
    p1, s1 = M.moe_nvfp4_quantize(compact)
    p2, s2 = M.moe_swiglu_nvfp4_quantize_ex(dev(w.data), w.clamp_L, round_to_bf16=True)
    assert torch.equal(p1, p2) and torch.equal(s1, s2)


@pytest.mark.parametrize("gs", [1.0, 2.7, 0.3])
def test_dequantize_bit_exact_and_round_trip(gs):
    w = W.quantize_normal(rows=128, K=2048, seed=2)
    p, s = M.moe_nvfp4_quantize_scaled(dev(w.data), gs)
    out = M.moe_nvfp4_dequantize(p, s, gs)
    ref = oracle.dequantize_nvfp4(host(p), host(s), gs)
    assert np.array_equal(bits(out), ref)
    # every (nibble, scale) pair
    codes = np.arange(0x7f, dtype=np.uint8)
    nibs = np.arange(16, dtype=np.uint8)
    packed = np.tile((nibs[0::2] | (nibs[1::2] << 4))[None, :], (codes.size + 1, 1))
    sf = np.concatenate([codes, np.zeros(1, np.uint8)])[:, None]
    out = M.moe_nvfp4_dequantize(torch.from_numpy(packed).cuda(), torch.from_numpy(sf).cuda(), gs)
    assert np.array_equal(bits(out), oracle.dequantize_nvfp4(packed, sf, gs))


def test_dequantize_every_pair_over_global_scales():
    """Every (nibble, scale code) pair under many global scales: the
    corrected-reciprocal division in [2^-90, 2^90], its edges, and the IEEE
    division outside; block counts that are not a multiple of four."""
    rng = np.random.default_rng(11)
    scales = [2.0 ** -90, 2.0 ** 90, np.nextafter(np.float32(2.0 ** -90), np.float32(0)),
              np.nextafter(np.float32(2.0 ** 90), np.float32(np.inf)), 2.0 ** -120, 3e37,
              1e-30, 7.0, 1.0 / 3.0]
    scales += list(np.exp(rng.uniform(np.log(1e-6), np.log(1e6), 24)))
    codes = np.arange(0x7f, dtype=np.uint8)
    nibs = np.arange(16, dtype=np.uint8)
    for gs in scales:
        gs = float(np.float32(gs))
        for extra_rows in (0, 1, 3):
            rows = codes.size + extra_rows
            packed = np.tile((nibs[0::2] | (nibs[1::2] << 4))[None, :], (rows, 1))
            sf = np.concatenate([codes, rng.integers(0, 0x7f, extra_rows).astype(np.uint8)])[:, None]
            out = M.moe_nvfp4_dequantize(torch.from_numpy(packed).cuda(),
                                         torch.from_numpy(np.ascontiguousarray(sf)).cuda(), gs)
            assert np.array_equal(bits(out), oracle.dequantize_nvfp4(packed, sf, gs)), (gs, rows)


@pytest.mark.parametrize("name", ["ragged", "prefill", "edge"])
def test_full_size_extensions_sampled(name):
    """Every fused extension at the full workload size, in the launch shape
    the benchmark times, checked on sampled rows: two-level, BF16 compat
    with and without a global scale, and the compact writer (the edge
    workload carries the adversarial blocks: ties, subnormal scales, zeros)."""
    w = W.make(name)
    off = None if w.offsets is None else torch.from_numpy(w.offsets).cuda()
    g = dev(w.data)
    rng = np.random.default_rng(1)
    r0 = 0 if w.offsets is None else int(w.offsets[0])
    r1 = w.rows if w.offsets is None else int(w.offsets[-1])
    rows = rng.integers(r0, r1, 24)
    sub = w.data[rows]
    for gs, compat in ((1.25, False), (1.25, True), (1.0, True)):
        p, s = M.moe_swiglu_nvfp4_quantize_ex(g, w.clamp_L, off, gs, compat)
        hp, hs = host(p), host(s)
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(sub, w.clamp_L, global_scale=gs, round_bf16=compat)
        assert np.array_equal(hs[rows], rs) and np.array_equal(hp[rows], rp), (gs, compat)
    out = M.moe_swiglu_bf16(g, w.clamp_L, off)
    assert np.array_equal(bits(out)[rows], oracle.swiglu_bf16(sub, w.clamp_L))


def test_edge_workload_extensions_every_block():
    """Two-level and BF16 compat on the whole edge workload (16384 rows x
    I = 4096, 10 % adversarial blocks on and next to rounding ties), every
    block against the oracle: the warp-wide re-decisions of the two-level
    step and the queued blocks of compat at their highest rates."""
    w = W.make("edge")
    g = dev(w.data)
    for gs, compat in ((1.25, False), (1.0, True), (1.25, True)):
        p, s = M.moe_swiglu_nvfp4_quantize_ex(g, w.clamp_L, None, gs, compat)
        rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data, w.clamp_L, global_scale=gs, round_bf16=compat)
        assert np.array_equal(host(s), rs) and np.array_equal(host(p), rp), (gs, compat)


def test_full_size_padded_sampled():
    """Padded output on the full ragged workload, as the benchmark times it
    (256 expert segments, each padded to 128 output rows): sampled input rows
    land at their shifted output rows with the oracle's values, and the
    padding rows after sampled segments keep their sentinel bytes."""
    w = W.make("ragged")
    off64 = w.offsets.astype(np.int64)
    counts = np.diff(off64)
    padded = (counts + 127) // 128 * 128
    out_off = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    out_rows = int(out_off[-1])
    pk = torch.full((out_rows, w.width // 2), 0xA5, dtype=torch.uint8, device="cuda")
    sf = torch.full((out_rows, w.width // 16), 0x5A, dtype=torch.uint8, device="cuda")
    p, s = M.moe_swiglu_nvfp4_quantize_ex(dev(w.data), w.clamp_L, torch.from_numpy(w.offsets).cuda(), 1.0,
                                         False, torch.from_numpy(out_off).cuda(), out_rows, pk, sf)
    hp, hs = host(p), host(s)
    rng = np.random.default_rng(2)
    rows = rng.integers(int(off64[0]), int(off64[-1]), 24)
    seg = np.searchsorted(off64, rows, side="right") - 1
    orow = out_off[seg] + (rows - off64[seg])
    rp, rs = oracle.swiglu_quantize_nvfp4_ex(w.data[rows], w.clamp_L)
    assert np.array_equal(hs[orow], rs) and np.array_equal(hp[orow], rp)
    gaps = [int(out_off[e] + counts[e]) for e in np.unique(seg) if padded[e] > counts[e]]
    assert gaps
    assert np.all(hp[gaps] == 0xA5) and np.all(hs[gaps] == 0x5A)
