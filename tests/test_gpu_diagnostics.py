"""The diagnostic entry points on the GPU, through the C ABI: the offsets
check (non-monotone, out-of-range and overlapping padded offsets set their
status bits; valid ones set none), the traffic-floor kernels (they touch
every block: their stores are the XOR of the words each block read), and the
fused and quantize-only steps on both sides of the size where the launch
shape changes from the small-problem kernels to the persistent grid, and
the small fused kernel's exact paths on near-tie blocks."""
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


def i32(a):
    return torch.tensor(np.asarray(a, np.int32), device="cuda")


def check(offsets, rows, out_offsets=None, out_rows=0):
    st = M.moe_nvfp4_check_offsets(i32(offsets), rows,
                                   None if out_offsets is None else i32(out_offsets), out_rows)
    torch.cuda.synchronize()
    return int(st.item())


B = M.CHECK_BITS


def test_offsets_check_accepts_valid_offsets():
    w = W.ragged_routing(tokens=512, experts=64, topk=4, I=64)
    assert check(w.offsets, w.rows) == 0
    counts = np.diff(w.offsets.astype(np.int64))
    out_off = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    assert check(w.offsets, w.rows, out_off, int(out_off[-1])) == 0
    assert check([0, 0, 0], 0) == 0                                   # empty segments
    assert check([5, 5], 10, [3, 3], 4) == 0


def test_offsets_check_flags_each_violation():
    assert check([0, 4, 3, 8], 8) == B["decreasing"]
    assert check([0, 4, 9], 8) == B["outside"]
    assert check([-1, 4, 8], 8) == B["outside"]
    assert check([0, 4, 2, 9], 8) == B["decreasing"] | B["outside"]
    # segment 0 -> rows [0, 4), segment 1 -> rows [3, 7): one row shared
    assert check([0, 4, 8], 8, [0, 3, 0], 16) == B["overlap"]
    # the same ranges in the other order, and far apart in the offsets array
    off = np.arange(0, 2 * 600 + 1, 2)                 # 600 segments of 2 rows
    dst = np.arange(0, 4 * 600 + 1, 4)                 # each padded to 4 rows
    assert check(off, 1200, dst, 2400) == 0
    dst_bad = dst.copy()
    dst_bad[599] = dst[3] + 1                          # the last segment lands on segment 3's rows
    assert check(off, 1200, dst_bad, 2400) == B["overlap"]
    # destination rows outside [0, out_rows) are skipped by the kernel, so
    # ranges that only meet there do not overlap
    assert check([0, 4, 8], 8, [-4, -4, 0], 16) == 0
    assert check([0, 4, 8], 8, [16, 14, 0], 16) == 0


def test_offsets_check_status_accumulates_and_step_stays_usable():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_nvfp4_check_offsets(i32([0, 4, 3]), 4, status=st)
    M.moe_nvfp4_check_offsets(i32([0, 5]), 4, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == B["decreasing"] | B["outside"]
    w = W.fused_normal(rows=64, I=256, seed=9)          # the step afterwards is unaffected
    gp, gs = M.moe_swiglu_nvfp4_quantize(torch.from_numpy(w.data.view(np.int16)).cuda(), w.clamp_L)
    rp, rs = oracle.swiglu_quantize_nvfp4(w.data, w.clamp_L)
    assert np.array_equal(gp.cpu().numpy(), rp) and np.array_equal(gs.cpu().numpy(), rs)


def xor_fold_blocks(data_u16: np.ndarray, words_per_block: int):
    w = np.ascontiguousarray(data_u16).view(np.uint32).reshape(-1, words_per_block)
    h = words_per_block // 2
    a = np.bitwise_xor.reduce(w[:, :h], axis=1)
    b = np.bitwise_xor.reduce(w[:, h:], axis=1)
    return a, b


@pytest.mark.parametrize("kind,rows,width", [("fused", 512, 2048), ("fused", 4099, 1024),
                                             ("quantize", 128, 2048), ("quantize", 16411, 512)])
def test_traffic_floor_touches_every_block(kind, rows, width):
    rng = np.random.default_rng(rows)
    in_w = 2 * width if kind == "fused" else width
    src = rng.integers(0, 2 ** 16, (rows, in_w), dtype=np.uint16)
    packed = torch.empty((rows, width // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, width // 16), dtype=torch.uint8, device="cuda")
    M.moe_nvfp4_traffic_floor(kind, torch.from_numpy(src.view(np.int16)).cuda(), width, packed, sf)
    torch.cuda.synchronize()
    a, b = xor_fold_blocks(src, 16 if kind == "fused" else 8)
    got = packed.cpu().numpy().reshape(-1, 8).view(np.uint32)
    assert np.array_equal(got[:, 0], a) and np.array_equal(got[:, 1], b)
    # the scale byte is a byte of the folded words (the persistent shape
    # folds both halves, the small fused shape's even lane its own)
    g = sf.cpu().numpy().ravel()
    assert np.all((g == ((a ^ b) & 0xFF)) | (g == (a & 0xFF)))


def test_traffic_floor_read_sweep_and_empty_launch():
    rng = np.random.default_rng(3)
    src = rng.integers(0, 2 ** 16, 3 * 2 ** 20 + 48, dtype=np.uint16)
    sink = torch.zeros(4, dtype=torch.uint8, device="cuda")
    M.moe_nvfp4_traffic_floor("read", torch.from_numpy(src.view(np.int16)).cuda(), packed=sink)
    M.moe_nvfp4_traffic_floor("empty")
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(src.view(np.uint32))
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(want)


def _shape_boundary_rows(width: int) -> list:
    """Row counts whose block counts span the sizes where the launch shape
    changes from the small-problem kernels (one block per thread for
    quantize-only, two threads per block for the fused step, up to one wave
    of their resident CTAs: about 0.7 to 1.2 x 10^5 blocks on 152 SMs,
    depending on their register counts) to the persistent grid, plus a
    ragged tail at each."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bpr = width // 16
    blocks = [sms * 128 * k // 2 for k in (7, 8, 10, 12)] + [sms * 128 * k for k in (5, 6, 7, 8)]
    return sorted({b // bpr + d for b in blocks for d in (0, 1)})


@pytest.mark.parametrize("I", [2048, 3072])
def test_fused_on_both_sides_of_the_launch_shape_boundary(I):
    for rows in _shape_boundary_rows(I):
        w = W.fused_normal(rows=rows, I=I, seed=rows)
        gp, gs = M.moe_swiglu_nvfp4_quantize(torch.from_numpy(w.data.view(np.int16)).cuda(), w.clamp_L)
        torch.cuda.synchronize()
        rp, rs = oracle.swiglu_quantize_nvfp4(w.data, w.clamp_L)
        rep = parity.compare_fused(gp.cpu().numpy(), gs.cpu().numpy(), rp, rs,
                                   lambda r, c: float(oracle.swiglu_values(w.data, w.clamp_L, r, r + 1)[0, c]))
        rep.assert_within_tolerance()
        assert rep.exact, (rows, rep)


def test_quantize_on_both_sides_of_the_launch_shape_boundary():
    for rows in _shape_boundary_rows(2048):
        w = W.quantize_normal(rows=rows, K=2048, seed=rows)
        gp, gs = M.moe_nvfp4_quantize(torch.from_numpy(w.data.view(np.int16)).cuda())
        torch.cuda.synchronize()
        rp, rs = oracle.quantize_nvfp4(w.data)
        assert np.array_equal(gp.cpu().numpy(), rp) and np.array_equal(gs.cpu().numpy(), rs), rows


def test_small_shape_ragged_offsets_with_sentinels():
    """The small-problem shape with device offsets: rows outside the
    segments keep their contents, including when the segments start past
    row 0."""
    w = W.ragged_routing(tokens=128, experts=16, topk=4, I=1024, pad_rows=33)
    off = w.offsets.astype(np.int64) + 17
    off = np.minimum(off, w.rows).astype(np.int32)
    sent_p = np.full((w.rows, w.width // 2), 0xA5, np.uint8)
    sent_s = np.full((w.rows, w.width // 16), 0x5A, np.uint8)
    p = torch.from_numpy(sent_p.copy()).cuda()
    s = torch.from_numpy(sent_s.copy()).cuda()
    M.moe_swiglu_nvfp4_quantize(torch.from_numpy(w.data.view(np.int16)).cuda(), w.clamp_L, i32(off), p, s)
    torch.cuda.synchronize()
    rp, rs = oracle.swiglu_quantize_nvfp4(w.data, w.clamp_L, off, packed=sent_p, sf=sent_s)
    assert np.array_equal(p.cpu().numpy(), rp) and np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("n_blocks,I", [(2048, 2048), (4096, 512)])
def test_small_shape_near_tie_blocks_exact(n_blocks, I):
    """Near-tie blocks (amax on 6 x E4M3 values and on 6 x midpoints, other
    outputs on half-step ties) at a size the small-problem kernel takes:
    both of its re-evaluation paths (the scale, shared by the two lanes of a
    block, and the nibbles) must give the definition's bytes."""
    rng = np.random.default_rng(n_blocks + I)
    blocks, stats = parity.fused_near_tie_blocks(rng, n_blocks, 7.0)
    gu = blocks.reshape(-1, 2 * I)
    gp, gs = M.moe_swiglu_nvfp4_quantize(torch.from_numpy(gu.view(np.int16)).cuda(), 7.0)
    cnt = torch.zeros(3, dtype=torch.int64, device="cuda")
    M.moe_swiglu_nvfp4_quantize_counted(torch.from_numpy(gu.view(np.int16)).cuda(), 7.0, cnt)
    torch.cuda.synchronize()
    rp, rs = oracle.swiglu_quantize_nvfp4(gu, 7.0)
    rep = parity.compare_fused(gp.cpu().numpy(), gs.cpu().numpy(), rp, rs,
                               lambda r, c: float(oracle.swiglu_values(gu, 7.0, r, r + 1)[0, c]))
    rep.assert_within_tolerance()
    assert rep.exact, rep
    blocks_done, scales, nibbles = (int(v) for v in cnt.cpu())
    assert blocks_done == n_blocks and scales > 0 and nibbles > 0      # both paths ran (counted variant)
