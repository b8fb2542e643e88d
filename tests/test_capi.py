"""The C ABI without a GPU: the library builds and loads, exports every
function include/moe_nvfp4.h declares, and rejects bad arguments on the host
before any CUDA call (none of these calls reach the device)."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


@pytest.fixture(scope="module")
def lib():
    from moe_swiglu_epilogue_gb300 import build, load_library
    build.build()
    return load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(
        r"^\s*MOE_NVFP4_API\s+(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(",
        text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_nvfp4_quantize", "moe_swiglu_nvfp4_quantize", "moe_nvfp4_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert [e for e in exported if e.startswith("moe_")] == declared_functions()


def test_abi_version_and_strerror(lib):
    assert lib.moe_nvfp4_abi_version() == 6
    for code in range(0, -10, -1):
        assert lib.moe_nvfp4_strerror(code)
    assert b"unknown" in lib.moe_nvfp4_strerror(-99)


# Fake device addresses with chosen alignment. Every call below must be
# rejected on the host (or have rows == 0) so that nothing is ever launched
# on them, even when this file runs on a machine with a GPU.
A32 = ctypes.c_void_p(0x7f0000000000)
A16 = ctypes.c_void_p(0x7f0000000010)
A2 = ctypes.c_void_p(0x7f0000000002)
NULL = ctypes.c_void_p(0)
S = ctypes.c_void_p(0)


def test_quantize_argument_errors(lib):
    q = lib.moe_nvfp4_quantize
    assert q(A32, -1, 32, A16, A16, S) == -4
    assert q(A32, 4, 24, A16, A16, S) == -2
    assert q(A32, 4, 0, A16, A16, S) == -2
    assert q(NULL, 4, 32, A16, A16, S) == -1
    assert q(A32, 4, 32, NULL, A16, S) == -1
    assert q(A16, 4, 32, A16, A16, S) == -3       # input only 16-byte aligned
    assert q(A32, 4, 32, A2, A16, S) == -3
    assert q(A32, 2 ** 62, 2 ** 10, A16, A16, S) == -4
    assert q(NULL, 0, 32, NULL, NULL, S) == 0     # nothing to do, nothing launched


def test_fused_argument_errors(lib):
    f = lib.moe_swiglu_nvfp4_quantize
    for bad_L in (0.0, -1.0, float("nan"), float("inf"), 1e30):
        assert f(A32, 0, 32, bad_L, NULL, 0, A16, A16, S) == -5
    assert f(A32, 0, 32, 7.0, NULL, -1, A16, A16, S) == -6
    assert f(A32, 0, 32, 7.0, NULL, 3, A16, A16, S) == -6
    assert f(A32, 4, 40, 7.0, NULL, 0, A16, A16, S) == -2
    assert f(A16, 4, 32, 7.0, NULL, 0, A16, A16, S) == -3
    assert f(A32, 0, 32, 7.0, NULL, 0, A16, A16, S) == 0
    assert f(A32, 4, 32, 7.0, A2, 3, A16, A16, S) == -3           # offsets must be 4-byte aligned


def test_e4m3_codes_argument_errors(lib):
    c = lib.moe_nvfp4_e4m3_codes
    assert c(A16, -1, A16, S) == -4
    assert c(NULL, 8, A16, S) == -1
    assert c(A16, 8, NULL, S) == -1
    assert c(A2, 8, A16, S) == -3                  # a float pointer must be 4-byte aligned
    assert c(NULL, 0, NULL, S) == 0


def test_window(lib):
    w7 = lib.moe_swiglu_nvfp4_window(7.0)
    w10 = lib.moe_swiglu_nvfp4_window(10.0)
    assert 2 ** -20 < w7 < 2 ** -16
    assert w7 <= w10 <= lib.moe_swiglu_nvfp4_window(1e6)
    assert lib.moe_swiglu_nvfp4_window(-1.0) < 0
    assert lib.moe_swiglu_nvfp4_window(float("nan")) < 0


def test_extension_argument_errors(lib):
    from moe_swiglu_epilogue_gb300 import FusedOptions
    import ctypes as C
    qs = lib.moe_nvfp4_quantize_scaled
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert qs(A32, 0, 32, bad, A16, A16, S) == -8
    assert qs(A32, 4, 24, 1.0, A16, A16, S) == -2
    assert qs(A32, 0, 32, 2.0, A16, A16, S) == 0
    ex = lib.moe_swiglu_nvfp4_quantize_ex
    opt = FusedOptions(0.0, 0, None, 0)
    assert ex(A32, 0, 32, 7.0, NULL, 0, C.byref(opt), A16, A16, S) == -8
    opt = FusedOptions(1.0, 1, 0x7f0000000100, 10)          # padded output without segments
    assert ex(A32, 0, 32, 7.0, NULL, 0, C.byref(opt), A16, A16, S) == -6
    opt = FusedOptions(1.0, 0, 0x7f0000000100, -1)
    assert ex(A32, 0, 32, 7.0, A16, 2, C.byref(opt), A16, A16, S) == -4
    assert ex(A32, 0, 32, 7.0, NULL, 0, None, A16, A16, S) == 0
    assert ex(A32, 4, 32, 0.0, NULL, 0, None, A16, A16, S) == -5
    assert ex(A32, 4, 32, 7.0, A2, 2, None, A16, A16, S) == -3     # offsets 4-byte aligned
    bad_out = FusedOptions(1.0, 0, A2.value, 8)
    assert ex(A32, 4, 32, 7.0, A16, 2, C.byref(bad_out), A16, A16, S) == -3
    compat = FusedOptions(1.0, 1, None, 0)
    # 2^32 blocks (256 GiB of input) and more are refused before any device call
    assert ex(A32, 1 << 28, 256, 7.0, NULL, 0, C.byref(compat), A16, A16, S) == -4
    assert ex(A32, 1 << 24, 1 << 16, 7.0, NULL, 0, C.byref(compat), A16, A16, S) == -4
    cw = lib.moe_swiglu_bf16
    assert cw(A32, 4, 32, 7.0, NULL, 0, NULL, S) == -1
    assert cw(A32, 4, 32, 7.0, NULL, 0, A2, S) == -3
    assert cw(A32, 1 << 28, 256, 7.0, NULL, 0, A32, S) == -4
    dq = lib.moe_nvfp4_dequantize
    assert dq(A16, A16, 4, 24, 1.0, A32, S) == -2
    assert dq(A16, A16, 4, 32, 0.0, A32, S) == -8
    assert dq(A16, A16, 4, 32, 1.0, A16, S) == -3      # output must be 32-byte aligned
    assert dq(NULL, A16, 4, 32, 1.0, A32, S) == -1
    assert dq(NULL, NULL, 0, 32, 1.0, NULL, S) == 0


def test_gemm_argument_errors(lib):
    g = lib.moe_l1_gemm_swiglu_nvfp4
    # (x, w1, rows, H, I, clamp_L, offsets, E, packed, sf, status, stream)
    assert g(A16, A16, -1, 64, 128, 7.0, A16, 1, A16, A16, NULL, S) == -4
    assert g(A16, A16, 4, 96, 128, 7.0, A16, 1, A16, A16, NULL, S) == -2      # H % 64
    assert g(A16, A16, 4, 64, 192, 7.0, A16, 1, A16, A16, NULL, S) == -2      # I % 128
    assert g(A16, A16, 4, 64, 128, 0.0, A16, 1, A16, A16, NULL, S) == -5
    assert g(A16, A16, 4, 64, 128, float("nan"), A16, 1, A16, A16, NULL, S) == -5
    assert g(A16, A16, 4, 64, 128, 7.0, NULL, 1, A16, A16, NULL, S) == -6     # offsets required
    assert g(A16, A16, 4, 64, 128, 7.0, A16, 0, A16, A16, NULL, S) == -6
    assert g(A16, A16, 4, 64, 128, 7.0, A16, 4096, A16, A16, NULL, S) == -6   # > 2048 experts
    assert g(A16, A16, 4, 64, 2 ** 30, 7.0, A16, 2, A16, A16, NULL, S) == -4  # E * 2I >= 2^31
    assert g(NULL, A16, 4, 64, 128, 7.0, A16, 1, A16, A16, NULL, S) == -1
    assert g(A16, A16, 4, 64, 128, 7.0, A16, 1, NULL, A16, NULL, S) == -1
    assert g(A2, A16, 4, 64, 128, 7.0, A16, 1, A16, A16, NULL, S) == -3
    assert g(A16, A16, 4, 64, 128, 7.0, A16, 1, A16, A2, NULL, S) == -3
    assert g(A16, A16, 4, 64, 128, 7.0, A2, 1, A16, A16, NULL, S) == -3      # offsets 4-byte aligned
    assert g(A16, A16, 4, 64, 128, 7.0, A16, 1, A16, A16, A2, S) == -3       # status 4-byte aligned
    assert g(NULL, NULL, 0, 64, 128, 7.0, A16, 1, NULL, NULL, NULL, S) == 0   # nothing to do
    a = lib.moe_l1_gemm_accumulators
    # (x, w1, rows, H, I, offsets, E, acc, status, stream)
    assert a(A16, A16, 4, 64, 128, A16, 1, NULL, NULL, S) == -1
    assert a(A16, A16, 4, 64, 128, A16, 1, A2, NULL, S) == -3
    assert a(A16, A16, 4, 100, 128, A16, 1, A16, NULL, S) == -2
    b = lib.moe_l1_gemm_bf16
    # (x, w1, rows, H, I, clamp_L, offsets, E, output, out, status, stream)
    assert b(A16, A16, 4, 64, 128, 7.0, A16, 1, 2, A16, NULL, S) == -9          # unknown output
    assert b(A16, A16, 4, 64, 128, 0.0, A16, 1, 1, A16, NULL, S) == -5          # SwiGLU needs L
    assert b(A16, A16, 4, 64, 128, 7.0, A16, 1, 0, NULL, NULL, S) == -1
    assert b(A16, A16, 4, 64, 128, 7.0, A16, 1, 0, A2, NULL, S) == -3
    assert b(A16, A16, 0, 64, 128, 0.0, A16, 1, 0, NULL, NULL, S) == 0         # gu ignores L
    t = lib.moe_l1_gemm_wait_selftest
    # (x, w1, rows, H, I, offsets, E, packed, sf, status, wait_cycles, mode, stream)
    assert t(A16, A16, 4, 64, 128, A16, 1, A16, A16, NULL, 10 ** 7, 1, S) == -1   # status required
    assert t(A16, A16, 4, 64, 128, A16, 1, A16, A16, A16, 10, 1, S) == -4         # limit out of range
    assert t(A16, A16, 4, 64, 128, A16, 1, A16, A16, A16, 10 ** 12, 2, S) == -4
    assert t(A16, A16, 4, 64, 128, A16, 1, A16, A16, A16, 10 ** 7, 0, S) == -9    # unknown mode
    assert t(A16, A16, 4, 64, 128, A16, 1, A16, A16, A16, 10 ** 7, 3, S) == -9
    w4 = lib.moe_l1_gemm_w4_swiglu_nvfp4
    # (x, w1_packed, w1_sf, rows, H, I, clamp_L, offsets, E, packed, sf, status, stream)
    assert w4(A16, A16, A16, 4, 128, 128, 7.0, A16, 1, A16, A16, NULL, S) == -2   # H % 256
    assert w4(A16, NULL, A16, 4, 256, 128, 7.0, A16, 1, A16, A16, NULL, S) == -1
    assert w4(A16, A16, A2, 4, 256, 128, 7.0, A16, 1, A16, A16, NULL, S) == -3
    assert w4(A16, A16, A16, 4, 256, 128, 0.0, A16, 1, A16, A16, NULL, S) == -5
    assert w4(NULL, NULL, NULL, 0, 256, 128, 7.0, A16, 1, NULL, NULL, NULL, S) == 0


def test_diagnostic_argument_errors(lib):
    tf = lib.moe_nvfp4_traffic_floor
    # (in, rows, width, kind, packed, sf, stream)
    assert tf(A32, 4, 32, 9, A16, A16, S) == -9                 # unknown kind
    assert tf(A32, 4, 32, -1, A16, A16, S) == -9
    assert tf(A32, 4, 24, 0, A16, A16, S) == -2
    assert tf(A16, 4, 32, 0, A16, A16, S) == -3                 # input 32-byte aligned
    assert tf(A32, 4, 32, 1, NULL, A16, S) == -1
    assert tf(A32, -1, 32, 3, A16, NULL, S) == -4
    assert tf(NULL, 4, 32, 3, A16, NULL, S) == -1
    assert tf(A32, 4, 32, 3, A2, NULL, S) == -3                 # sink 4-byte aligned
    assert tf(NULL, 0, 32, 0, NULL, NULL, S) == 0
    co = lib.moe_nvfp4_check_offsets
    # (offsets, E, rows, out_offsets, out_rows, status, stream)
    assert co(A16, -1, 4, NULL, 0, A16, S) == -4
    assert co(A16, 2, -4, NULL, 0, A16, S) == -4
    assert co(NULL, 2, 4, NULL, 0, A16, S) == -1
    assert co(A16, 2, 4, NULL, 0, NULL, S) == -1
    assert co(A2, 2, 4, NULL, 0, A16, S) == -3
    assert co(A16, 2, 4, A2, 8, A16, S) == -3
    assert co(A16, 2, 4, NULL, 0, A2, S) == -3
    assert co(A16, 2 ** 31 - 1, 4, A16, 8, A16, S) == -4       # too many segments for the overlap test
