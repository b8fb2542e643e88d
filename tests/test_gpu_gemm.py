"""GPU parity of the L1 GEMM with the step in its epilogue, through the C
ABI: (1) the kernel's fp32 accumulators against the float64 GEMM within the
bound of fp32 accumulation; (2) its NVFP4 outputs against the oracle applied
to those same accumulators, within the fast SwiGLU's tolerance; (3) against
the oracle on exact accumulators, statistically; rows outside the segments
untouched; the kernel's wait status stays zero."""
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


def acc_bound(H):
    """fp32 accumulation: one rounding per K-16 MMA step at most, each within
    2^-24 of the running sum, which is at most sum |x w|; x2 margin."""
    return (H / 16 + 2) * 2.0 ** -23


CASES = {
    "tiny": dict(tokens=96, experts=4, topk=2, H=256, I=128, seed=31),
    "ragged_pad": dict(tokens=512, experts=8, topk=2, H=512, I=256, pad_rows=37, seed=32),
    "dense": dict(tokens=200, experts=1, topk=1, H=1024, I=512, seed=33),
    # the most experts the kernels take (2048): most segments empty, the
    # others one or a few rows, so nearly every tile is a ragged tail
    "max_experts": dict(tokens=1024, experts=2048, topk=2, H=256, I=128, seed=34),
}


def _case(name):
    return W.gemm_ragged(**CASES[name])


def _run(w, acc_too=True):
    x, w1, off = dev(w.x), dev(w.w1), torch.from_numpy(w.offsets).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = w.rows
    sent_p = torch.full((rows, w.I // 2), 0xA5, dtype=torch.uint8, device="cuda")
    sent_s = torch.full((rows, w.I // 16), 0x5A, dtype=torch.uint8, device="cuda")
    p, s = M.moe_l1_gemm_swiglu_nvfp4(x, w1, w.clamp_L, off, sent_p, sent_s, status)
    acc = None
    if acc_too:
        acc = M.moe_l1_gemm_accumulators(x, w1, off, status=status)
    assert int(host(status)[0]) == 0
    return host(p), host(s), None if acc is None else host(acc)


@pytest.mark.parametrize("name", list(CASES))
def test_accumulators_within_fp32_accumulation_bound(name):
    w = _case(name)
    _, _, acc = _run(w)
    ref = oracle.l1_gemm_accumulators(w.x, w.w1, w.offsets)
    mag = oracle.l1_gemm_abs_accumulators(w.x, w.w1, w.offsets)
    r0, r1 = int(w.offsets[0]), int(w.offsets[-1])
    err = np.abs(acc[r0:r1].astype(np.float64) - ref[r0:r1])
    assert np.all(err <= acc_bound(w.H) * mag[r0:r1] + 1e-30), (err / mag[r0:r1]).max()


@pytest.mark.parametrize("name", list(CASES))
def test_fused_output_matches_the_oracle_on_the_kernels_accumulators(name):
    w = _case(name)
    p, s, acc = _run(w)
    r0, r1 = int(w.offsets[0]), int(w.offsets[-1])
    y_ref = oracle.gemm_swiglu_values(acc[r0:r1].astype(np.float64), w.clamp_L)
    sf_bad, nib_bad, n = parity.compare_gemm_fused(p[r0:r1], s[r0:r1], y_ref)
    assert sf_bad <= 2 and nib_bad <= max(2, n * 1e-4)
    # rows past the last segment were never written
    assert np.all(p[r1:] == 0xA5) and np.all(s[r1:] == 0x5A)


@pytest.mark.parametrize("name", list(CASES))
def test_fused_output_against_exact_accumulators(name):
    """The GEMM end to end: nearly every decision equals the oracle's on the
    exact (float64) accumulators; the rest sit next to a rounding boundary."""
    w = _case(name)
    p, s, _ = _run(w, acc_too=False)
    rp, rs = oracle.l1_gemm_swiglu_quantize_nvfp4(w.x, w.w1, w.offsets, w.clamp_L)
    r0, r1 = int(w.offsets[0]), int(w.offsets[-1])
    assert np.mean(s[r0:r1] == rs[r0:r1]) >= 0.999
    gn, rn = parity.unpack_nibbles(p[r0:r1]), parity.unpack_nibbles(rp[r0:r1])
    assert np.mean(gn == rn) >= 0.999
    assert np.all(np.abs(parity.signed_index(gn) - parity.signed_index(rn)) <= 1)


def test_segments_with_gaps_and_empty_experts():
    rng = np.random.default_rng(5)
    rows, H, I, E = 300, 256, 256, 5
    x = W.bf16_bits(rng.standard_normal((rows, H)).astype(np.float32))
    w1 = W.bf16_bits((rng.standard_normal((E, 2 * I, H)) / 10).astype(np.float32))
    offsets = np.array([7, 7, 140, 141, 141, 290], np.int32)       # gap, empties, one-row expert
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = torch.full((rows, I // 2), 0xA5, dtype=torch.uint8, device="cuda")
    ss = torch.full((rows, I // 16), 0x5A, dtype=torch.uint8, device="cuda")
    p, s = M.moe_l1_gemm_swiglu_nvfp4(dev(x), dev(w1).view(E, 2 * I, H), 7.0,
                                      torch.from_numpy(offsets).cuda(), sp, ss, status)
    acc = M.moe_l1_gemm_accumulators(dev(x), dev(w1).view(E, 2 * I, H), torch.from_numpy(offsets).cuda(),
                                     status=status)
    p, s, acc = host(p), host(s), host(acc)
    assert int(host(status)[0]) == 0
    y_ref = oracle.gemm_swiglu_values(acc[7:290].astype(np.float64), 7.0)
    parity.compare_gemm_fused(p[7:290], s[7:290], y_ref)
    assert np.all(p[:7] == 0xA5) and np.all(p[290:] == 0xA5)
    assert np.all(s[:7] == 0x5A) and np.all(s[290:] == 0x5A)
    ref = oracle.l1_gemm_accumulators(x, w1, offsets)
    mag = oracle.l1_gemm_abs_accumulators(x, w1, offsets)
    assert np.all(np.abs(acc[7:290] - ref[7:290]) <= acc_bound(H) * mag[7:290] + 1e-30)


def test_full_width_sampled_rows():
    """H = 7168, I = 2048 (the sizes the benchmark uses), 4 experts; rows
    sampled from every expert checked against the oracle."""
    w = W.gemm_ragged(tokens=256, experts=4, topk=2, H=7168, I=2048, seed=21)
    p, s, acc = _run(w)
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(np.arange(int(w.offsets[0]), int(w.offsets[-1])), 24, replace=False))
    sub_off = np.searchsorted(rows, w.offsets).astype(np.int32)       # segments of the sample
    ref = oracle.l1_gemm_accumulators(w.x[rows], w.w1, sub_off)
    mag = oracle.l1_gemm_abs_accumulators(w.x[rows], w.w1, sub_off)
    assert np.all(np.abs(acc[rows] - ref) <= acc_bound(w.H) * mag + 1e-30)
    y_ref = oracle.gemm_swiglu_values(acc[rows].astype(np.float64), w.clamp_L)
    parity.compare_gemm_fused(p[rows], s[rows], y_ref)


@pytest.mark.parametrize("name", ["tiny", "ragged_pad"])
def test_bf16_outputs_of_the_unfused_flows(name):
    """gu: the RN_bf16 of the kernel's accumulators (bit for bit, same MMA
    sequence) and within half a BF16 ulp plus the accumulation bound of the
    exact GEMM. SwiGLU: the oracle's SwiGLU of those accumulators rounded to
    BF16, except one-ulp differences where that value lies within the fast
    SwiGLU's tolerance of a BF16 midpoint. Rows outside the segments stay."""
    w = _case(name)
    x, w1, off = dev(w.x), dev(w.w1), torch.from_numpy(w.offsets).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows, I = w.rows, w.I
    sent = 0x4040
    gu = torch.full((rows, 2 * I), sent, dtype=torch.int16, device="cuda")
    sw = torch.full((rows, I), sent, dtype=torch.int16, device="cuda")
    M.moe_l1_gemm_bf16(x, w1, off, "gu", out=gu, status=status)
    M.moe_l1_gemm_bf16(x, w1, off, "swiglu", w.clamp_L, out=sw, status=status)
    acc = host(M.moe_l1_gemm_accumulators(x, w1, off, status=status))
    assert int(host(status)[0]) == 0
    gu, sw = host(gu).view(np.uint16), host(sw).view(np.uint16)
    r0, r1 = int(w.offsets[0]), int(w.offsets[-1])
    assert np.all(gu[:r0] == sent) and np.all(gu[r1:] == sent)
    assert np.all(sw[:r0] == sent) and np.all(sw[r1:] == sent)
    assert np.array_equal(gu[r0:r1], W.bf16_bits(acc[r0:r1]))
    ref = oracle.l1_gemm_accumulators(w.x, w.w1, w.offsets)[r0:r1]
    mag = oracle.l1_gemm_abs_accumulators(w.x, w.w1, w.offsets)[r0:r1]
    g = W.bf16_to_f32(gu[r0:r1]).reshape(r1 - r0, 2 * I).astype(np.float64)
    half_ulp = np.abs(g) * 2.0 ** -8
    assert np.all(np.abs(g - ref) <= half_ulp + acc_bound(w.H) * mag + 1e-30)
    y = oracle.gemm_swiglu_values(acc[r0:r1].astype(np.float64), w.clamp_L)
    want = W.bf16_bits(y)
    bad = np.argwhere(sw[r0:r1] != want)
    for r, c in bad:
        yv = np.float64(y[r, c])
        lo = W.bf16_bits(np.float32(yv * (1 - parity.GEMM_Y_REL_TOL)))
        hi = W.bf16_bits(np.float32(yv * (1 + parity.GEMM_Y_REL_TOL)))
        assert lo != hi and sw[r0 + r, c] in (lo, hi), (r, c, yv)
    assert bad.shape[0] <= max(2, 1e-4 * want.size)


def test_expired_wait_reports_its_status_and_the_device_stays_usable():
    """Failure path without a fault: with its loads withheld, the kernel's
    first MMA wait can never complete; after the given limit (~10 ms here)
    it records the code of the expired wait, every role stops, the TMEM is
    released, and packed / sf stay untouched. The next GEMM on the same
    device (which must allocate the TMEM again) is correct."""
    w = _case("tiny")
    x, w1, off = dev(w.x), dev(w.w1), torch.from_numpy(w.offsets).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = torch.full((w.rows, w.I // 2), 0xA5, dtype=torch.uint8, device="cuda")
    ss = torch.full((w.rows, w.I // 16), 0x5A, dtype=torch.uint8, device="cuda")
    M.moe_l1_gemm_wait_selftest(x, w1, off, status, 20_000_000, sp, ss, mode="no_loads")
    code = int(host(status)[0])
    assert code in (3, 4), code
    assert bool((sp == 0xA5).all()) and bool((ss == 0x5A).all())
    status.zero_()
    p, s, acc = _run(w)
    r0, r1 = int(w.offsets[0]), int(w.offsets[-1])
    y_ref = oracle.gemm_swiglu_values(acc[r0:r1].astype(np.float64), w.clamp_L)
    parity.compare_gemm_fused(p[r0:r1], s[r0:r1], y_ref)


def _w4_case(name):
    """The case's BF16 weights quantized to NVFP4 by the oracle, and the
    oracle's (exact) dequantization of them back to BF16."""
    w = _case(name)
    E, two_i, H = w.w1.shape
    qp, qs = oracle.quantize_nvfp4(w.w1.reshape(E * two_i, H))
    deq = oracle.dequantize_nvfp4(qp, qs)
    return w, qp.reshape(E, two_i, H // 2), qs.reshape(E, two_i, H // 16), deq.reshape(E, two_i, H)


def _run_w4(w, qp, qs):
    x, off = dev(w.x), torch.from_numpy(w.offsets).cuda()
    tq, ts = torch.from_numpy(qp).cuda(), torch.from_numpy(qs).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = torch.full((w.rows, w.I // 2), 0xA5, dtype=torch.uint8, device="cuda")
    ss = torch.full((w.rows, w.I // 16), 0x5A, dtype=torch.uint8, device="cuda")
    p, s = M.moe_l1_gemm_w4_swiglu_nvfp4(x, tq, ts, w.clamp_L, off, sp, ss, status)
    acc = M.moe_l1_gemm_w4_accumulators(x, tq, ts, off, status=status)
    assert int(host(status)[0]) == 0
    return host(p), host(s), host(acc)


@pytest.mark.parametrize("name", list(CASES))
def test_w4_gemm_equals_the_bf16_gemm_on_the_dequantized_weights(name):
    """NVFP4 weights expanded in the kernel: the outputs and accumulators
    equal, bit for bit, the BF16 GEMM's on the oracle's dequantization."""
    w, qp, qs, deq = _w4_case(name)
    p4, s4, a4 = _run_w4(w, qp, qs)
    wd = W.GemmWorkload(w.name, w.rows, w.H, w.I, w.x, deq, w.offsets, w.clamp_L)
    p, s, a = _run(wd)
    r0, r1 = int(w.offsets[0]), int(w.offsets[-1])
    assert np.array_equal(a4[r0:r1], a[r0:r1])
    assert np.array_equal(p4, p) and np.array_equal(s4, s)


@pytest.mark.parametrize("name", list(CASES))
def test_w4_gemm_against_the_oracle(name):
    w, qp, qs, deq = _w4_case(name)
    p, s, acc = _run_w4(w, qp, qs)
    r0, r1 = int(w.offsets[0]), int(w.offsets[-1])
    ref = oracle.l1_gemm_accumulators(w.x, deq, w.offsets)[r0:r1]
    mag = oracle.l1_gemm_abs_accumulators(w.x, deq, w.offsets)[r0:r1]
    assert np.all(np.abs(acc[r0:r1] - ref) <= acc_bound(w.H) * mag + 1e-30)
    y_ref = oracle.gemm_swiglu_values(acc[r0:r1].astype(np.float64), w.clamp_L)
    parity.compare_gemm_fused(p[r0:r1], s[r0:r1], y_ref)
    assert np.all(p[r1:] == 0xA5) and np.all(s[r1:] == 0x5A)


def test_w4_gemm_full_width():
    """H = 7168, I = 2048 over 4 experts: equal to the BF16 GEMM on the
    dequantized weights everywhere; sampled rows against the oracle."""
    w = W.gemm_ragged(tokens=256, experts=4, topk=2, H=7168, I=2048, seed=22)
    E, two_i, H = w.w1.shape
    qp, qs = oracle.quantize_nvfp4(w.w1.reshape(E * two_i, H))
    deq = oracle.dequantize_nvfp4(qp, qs).reshape(E, two_i, H)
    p4, s4, a4 = _run_w4(w, qp.reshape(E, two_i, H // 2), qs.reshape(E, two_i, H // 16))
    p, s, a = _run(W.GemmWorkload(w.name, w.rows, H, w.I, w.x, deq, w.offsets, w.clamp_L))
    assert np.array_equal(a4, a) and np.array_equal(p4, p) and np.array_equal(s4, s)
    rows = np.sort(np.random.default_rng(4).choice(np.arange(int(w.offsets[-1])), 16, replace=False))
    sub_off = np.searchsorted(rows, w.offsets).astype(np.int32)
    ref = oracle.l1_gemm_accumulators(w.x[rows], deq, sub_off)
    mag = oracle.l1_gemm_abs_accumulators(w.x[rows], deq, sub_off)
    assert np.all(np.abs(a4[rows] - ref) <= acc_bound(H) * mag + 1e-30)


def test_expired_wait_with_work_in_flight_drains_before_exit():
    """The abort path with loads and MMAs issued: the epilogue never frees
    an accumulator, and one CTA runs every tile, so after two tiles the MMA
    issuer's wait (or the producer's, for a stage of the third) expires
    while TMA loads for the next tile and the MMAs of the first two were
    issued. Both roles wait for that work before the TMEM is released: the
    status holds the expired wait's code (never the drain's 8), the outputs
    stay untouched, and the next GEMM on the device is correct."""
    w = _case("ragged_pad")
    x, w1, off = dev(w.x), dev(w.w1), torch.from_numpy(w.offsets).cuda()
    assert w.active_rows // 128 * (2 * w.I // 256) >= 3                   # at least three tiles
    for _ in range(2):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        sp = torch.full((w.rows, w.I // 2), 0xA5, dtype=torch.uint8, device="cuda")
        ss = torch.full((w.rows, w.I // 16), 0x5A, dtype=torch.uint8, device="cuda")
        M.moe_l1_gemm_wait_selftest(x, w1, off, status, 20_000_000, sp, ss, mode="no_release")
        code = int(host(status)[0])
        assert code in (1, 2), code
        assert bool((sp == 0xA5).all()) and bool((ss == 0x5A).all())
    p, s, acc = _run(w)
    r0, r1 = int(w.offsets[0]), int(w.offsets[-1])
    y_ref = oracle.gemm_swiglu_values(acc[r0:r1].astype(np.float64), w.clamp_L)
    parity.compare_gemm_fused(p[r0:r1], s[r0:r1], y_ref)
