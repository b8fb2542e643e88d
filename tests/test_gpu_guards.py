"""Guard bytes around every output: each entry point writes into the middle
of a larger buffer whose head and tail hold a pattern, with odd shapes
(33 rows, widths that are not powers of two); afterwards the pattern must
be intact (a substitute for a memory checker, which is not available)."""
import numpy as np
import pytest
import torch

import oracle
import moe_swiglu_epilogue_gb300 as M
from moe_swiglu_epilogue_gb300 import FusedOptions, workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes before and after each output (keeps 256-byte alignment)
PATTERN = 0xC3


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


class Guarded:
    """A [shape] tensor of `dtype` living between two guard regions."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.n = n
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return bool((self.raw[:GUARD] == PATTERN).all()) and bool((self.raw[GUARD + self.n:] == PATTERN).all())


def test_activation_step_outputs_stay_inside_their_buffers():
    rows, I = 33, 1040
    w = W.ragged_routing(tokens=12, experts=4, topk=2, I=I, pad_rows=9)
    gu = dev(w.data)
    off = torch.from_numpy(w.offsets).cuda()
    rows = w.rows
    p, s = Guarded((rows, I // 2), torch.uint8), Guarded((rows, I // 16), torch.uint8)
    M.moe_swiglu_nvfp4_quantize(gu, w.clamp_L, off, p.t, s.t)
    assert p.intact() and s.intact()
    for gs, compat in ((1.0, False), (1.3, False), (1.0, True), (0.7, True)):
        p, s = Guarded((rows, I // 2), torch.uint8), Guarded((rows, I // 16), torch.uint8)
        M.moe_swiglu_nvfp4_quantize_ex(gu, w.clamp_L, off, gs, compat, packed=p.t, sf=s.t)
        assert p.intact() and s.intact(), (gs, compat)
    counts = np.diff(w.offsets)
    out_off = np.concatenate([[0], np.cumsum(np.ceil(counts / 16).astype(np.int64) * 16)]).astype(np.int32)
    orows = int(out_off[-1])
    p, s = Guarded((orows, I // 2), torch.uint8), Guarded((orows, I // 16), torch.uint8)
    M.moe_swiglu_nvfp4_quantize_ex(gu, w.clamp_L, off, 1.0, False, torch.from_numpy(out_off).cuda(), orows,
                                   p.t, s.t)
    assert p.intact() and s.intact()
    c = Guarded((rows, I), torch.bfloat16)
    M.moe_swiglu_bf16(gu, w.clamp_L, off, c.t)
    assert c.intact()
    q = W.quantize_normal(rows=33, K=272, seed=4)
    x = dev(q.data)
    for gs in (None, 2.5):
        p, s = Guarded((33, 136), torch.uint8), Guarded((33, 17), torch.uint8)
        if gs is None:
            M.moe_nvfp4_quantize(x, p.t, s.t)
        else:
            M.moe_nvfp4_quantize_scaled(x, gs, p.t, s.t)
        assert p.intact() and s.intact()
    pq, sq = M.moe_nvfp4_quantize(x)
    d = Guarded((33, 272), torch.bfloat16)
    M.moe_nvfp4_dequantize(pq, sq, 1.0, d.t)
    assert d.intact()


def test_gemm_outputs_stay_inside_their_buffers():
    g = W.gemm_ragged(tokens=33, experts=3, topk=2, H=192, I=384, seed=8, pad_rows=5)
    x, w1, off = dev(g.x), dev(g.w1), torch.from_numpy(g.offsets).cuda()
    rows, I = g.rows, g.I
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    p, s = Guarded((rows, I // 2), torch.uint8), Guarded((rows, I // 16), torch.uint8)
    M.moe_l1_gemm_swiglu_nvfp4(x, w1, g.clamp_L, off, p.t, s.t, status)
    assert p.intact() and s.intact()
    a = Guarded((rows, 2 * I), torch.float32)
    M.moe_l1_gemm_accumulators(x, w1, off, a.t, status)
    assert a.intact()
    for output, width in (("gu", 2 * I), ("swiglu", I)):
        o = Guarded((rows, width), torch.bfloat16)
        M.moe_l1_gemm_bf16(x, w1, off, output, g.clamp_L, o.t, status)
        assert o.intact(), output
    torch.cuda.synchronize()
    assert int(status.item()) == 0
