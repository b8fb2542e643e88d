"""The diagnostic entry points on the GPU, through the C ABI: the offsets
check (non-monotone, out-of-range and overlapping padded offsets set their
status bits; valid ones set none), the traffic-floor kernels (they touch
every block: their stores are the XOR of the words each block read), and the
fused and quantize-only steps on both sides of the size where the launch
shape changes from one block per thread to the persistent grid."""
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
    assert np.array_equal(sf.cpu().numpy().ravel(), ((a ^ b) & 0xFF).astype(np.uint8))


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
    """Row counts whose block count sits at the largest size the one-block-
    per-thread shape takes (152 SMs x 3 CTAs x 256 threads) and just past
    it, where the persistent grid takes over."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cap = sms * 3 * 256
    bpr = width // 16
    return sorted({cap // bpr, cap // bpr + 1, (cap + bpr - 1) // bpr + 7})


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
    """One block per thread with device offsets: rows outside the segments
    keep their contents, including when the segments start past row 0."""
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
