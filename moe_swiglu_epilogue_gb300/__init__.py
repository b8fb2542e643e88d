"""GB300 (sm_103a) MoE expert activation step: deinterleave + clamped SwiGLU
+ NVFP4 quantize, behind the C ABI of ``libmoe_swiglu_nvfp4.so``
(``include/moe_nvfp4.h``).

This module only marshals arguments: it checks torch tensors, takes their
device pointers and the current CUDA stream, and calls the C entry point of
the same name. Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and importing the binding fails
loudly when the library has not been built (``python -m
moe_swiglu_epilogue_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = ["moe_nvfp4_quantize", "moe_swiglu_nvfp4_quantize", "moe_swiglu_fast_values",
           "moe_swiglu_precise_values", "moe_nvfp4_e4m3_codes", "moe_nvfp4_quantize_scaled",
           "moe_swiglu_nvfp4_quantize_ex", "moe_swiglu_bf16", "moe_nvfp4_dequantize",
           "moe_swiglu_nvfp4_quantize_counted", "moe_swiglu_nvfp4_window",
           "moe_l1_gemm_swiglu_nvfp4", "moe_l1_gemm_accumulators", "moe_l1_gemm_bf16",
           "moe_l1_gemm_wait_selftest", "moe_l1_gemm_w4_swiglu_nvfp4", "moe_l1_gemm_w4_accumulators",
           "moe_nvfp4_traffic_floor", "moe_nvfp4_check_offsets", "TRAFFIC_KINDS", "CHECK_BITS",
           "moe_nvfp4_strerror", "MoeNvfp4Error", "library_path", "load_library"]

# include/moe_nvfp4.h: MOE_NVFP4_TRAFFIC_* and MOE_NVFP4_CHECK_*
TRAFFIC_KINDS = {"fused": 0, "quantize": 1, "empty": 2, "read": 3}
CHECK_BITS = {"decreasing": 1, "outside": 2, "overlap": 4}

_lib = None


class FusedOptions(ctypes.Structure):
    """moe_nvfp4_fused_options of include/moe_nvfp4.h."""
    _fields_ = [("global_scale", ctypes.c_float), ("round_to_bf16", ctypes.c_int32),
                ("out_offsets", ctypes.c_void_p), ("out_rows", ctypes.c_int64)]


class MoeNvfp4Error(RuntimeError):
    def __init__(self, code: int, name: str):
        self.code = code
        super().__init__(f"{name}: {moe_nvfp4_strerror(code)} (code {code})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m moe_swiglu_epilogue_gb300.build` (no fallback exists)")
    lib = ctypes.CDLL(path)
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    lib.moe_nvfp4_quantize.argtypes = [P, I64, I64, P, P, P]
    lib.moe_nvfp4_quantize.restype = ctypes.c_int
    lib.moe_swiglu_nvfp4_quantize.argtypes = [P, I64, I64, F, P, I32, P, P, P]
    lib.moe_swiglu_nvfp4_quantize.restype = ctypes.c_int
    lib.moe_swiglu_fast_values.argtypes = [P, I64, I64, F, P, P]
    lib.moe_swiglu_fast_values.restype = ctypes.c_int
    lib.moe_swiglu_precise_values.argtypes = [P, I64, I64, F, P, P]
    lib.moe_nvfp4_e4m3_codes.argtypes = [P, I64, P, P]
    lib.moe_nvfp4_e4m3_codes.restype = ctypes.c_int
    lib.moe_swiglu_precise_values.restype = ctypes.c_int
    lib.moe_swiglu_nvfp4_quantize_counted.argtypes = [P, I64, I64, F, P, I32, P, P, P, P]
    lib.moe_swiglu_nvfp4_quantize_counted.restype = ctypes.c_int
    lib.moe_swiglu_nvfp4_window.argtypes = [F]
    lib.moe_swiglu_nvfp4_window.restype = ctypes.c_double
    lib.moe_nvfp4_strerror.argtypes = [ctypes.c_int]
    lib.moe_nvfp4_strerror.restype = ctypes.c_char_p
    lib.moe_nvfp4_quantize_scaled.argtypes = [P, I64, I64, F, P, P, P]
    lib.moe_nvfp4_quantize_scaled.restype = ctypes.c_int
    lib.moe_swiglu_nvfp4_quantize_ex.argtypes = [P, I64, I64, F, P, I32, ctypes.POINTER(FusedOptions),
                                                 P, P, P]
    lib.moe_swiglu_nvfp4_quantize_ex.restype = ctypes.c_int
    lib.moe_swiglu_bf16.argtypes = [P, I64, I64, F, P, I32, P, P]
    lib.moe_swiglu_bf16.restype = ctypes.c_int
    lib.moe_nvfp4_dequantize.argtypes = [P, P, I64, I64, F, P, P]
    lib.moe_nvfp4_dequantize.restype = ctypes.c_int
    lib.moe_l1_gemm_swiglu_nvfp4.argtypes = [P, P, I64, I64, I64, F, P, I32, P, P, P, P]
    lib.moe_l1_gemm_swiglu_nvfp4.restype = ctypes.c_int
    lib.moe_l1_gemm_accumulators.argtypes = [P, P, I64, I64, I64, P, I32, P, P, P]
    lib.moe_l1_gemm_accumulators.restype = ctypes.c_int
    lib.moe_l1_gemm_w4_swiglu_nvfp4.argtypes = [P, P, P, I64, I64, I64, F, P, I32, P, P, P, P]
    lib.moe_l1_gemm_w4_swiglu_nvfp4.restype = ctypes.c_int
    lib.moe_l1_gemm_w4_accumulators.argtypes = [P, P, P, I64, I64, I64, P, I32, P, P, P]
    lib.moe_l1_gemm_w4_accumulators.restype = ctypes.c_int
    lib.moe_l1_gemm_wait_selftest.argtypes = [P, P, I64, I64, I64, P, I32, P, P, P, I64, I32, P]
    lib.moe_l1_gemm_wait_selftest.restype = ctypes.c_int
    lib.moe_l1_gemm_bf16.argtypes = [P, P, I64, I64, I64, F, P, I32, I32, P, P, P]
    lib.moe_l1_gemm_bf16.restype = ctypes.c_int
    lib.moe_nvfp4_traffic_floor.argtypes = [P, I64, I64, I32, P, P, P]
    lib.moe_nvfp4_traffic_floor.restype = ctypes.c_int
    lib.moe_nvfp4_check_offsets.argtypes = [P, I32, I64, P, I64, P, P]
    lib.moe_nvfp4_check_offsets.restype = ctypes.c_int
    lib.moe_nvfp4_abi_version.argtypes = []
    lib.moe_nvfp4_abi_version.restype = ctypes.c_int
    _lib = lib
    return lib


def moe_nvfp4_strerror(code: int) -> str:
    return load_library().moe_nvfp4_strerror(int(code)).decode()


def moe_swiglu_nvfp4_window(clamp_L: float) -> float:
    return float(load_library().moe_swiglu_nvfp4_window(float(clamp_L)))


# ---------------------------------------------------------------------------
# torch-tensor front end
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _bf16_bits(t, name: str, width_mult: int):
    torch = _torch()
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in (torch.bfloat16, torch.uint16, torch.int16):
        raise ValueError(f"{name} must hold BF16 (bfloat16, or its bits as uint16/int16)")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")
    if t.shape[1] % width_mult:
        raise ValueError(f"{name}.shape[1] must be a multiple of {width_mult}")
    return t


def _out(t, shape, device, name: str):
    torch = _torch()
    if t is None:
        return torch.empty(shape, dtype=torch.uint8, device=device)
    if t.dtype != torch.uint8 or tuple(t.shape) != tuple(shape) or not t.is_contiguous() \
            or t.device != device:
        raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor of shape {shape}")
    return t


def _stream_ptr(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, name: str):
    if rc != 0:
        raise MoeNvfp4Error(rc, name)


def moe_nvfp4_quantize(x, packed=None, sf=None, stream=None):
    """Quantize-only: x BF16 [rows, K] -> (packed uint8 [rows, K/2],
    sf uint8 [rows, K/16]; view sf as torch.float8_e4m3fn for the values)."""
    x = _bf16_bits(x, "x", 16)
    rows, K = x.shape
    packed = _out(packed, (rows, K // 2), x.device, "packed")
    sf = _out(sf, (rows, K // 16), x.device, "sf")
    with _torch().cuda.device(x.device):
        rc = load_library().moe_nvfp4_quantize(
            ctypes.c_void_p(x.data_ptr()), rows, K, ctypes.c_void_p(packed.data_ptr()),
            ctypes.c_void_p(sf.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_nvfp4_quantize")
    return packed, sf


def _offsets_arg(offsets, device):
    torch = _torch()
    if offsets is None:
        return ctypes.c_void_p(0), 0
    if not offsets.is_cuda or offsets.dtype != torch.int32 or offsets.dim() != 1 \
            or not offsets.is_contiguous() or offsets.device != device:
        raise ValueError("expert_offsets must be a contiguous int32 CUDA tensor [E+1] "
                         "on the input's device")
    return ctypes.c_void_p(offsets.data_ptr()), offsets.shape[0] - 1


def moe_swiglu_nvfp4_quantize(gu, clamp_L: float, expert_offsets=None, packed=None, sf=None,
                              stream=None):
    """Fused: gu BF16 [rows, 2I] in [gate x8, up x8, ...] groups ->
    (packed uint8 [rows, I/2], sf uint8 [rows, I/16]). With expert_offsets
    (int32 [E+1] on the device) rows outside [offsets[0], offsets[E]) are
    left untouched; pass preallocated `packed`/`sf` to keep them."""
    gu = _bf16_bits(gu, "gu", 32)
    rows, two_i = gu.shape
    I = two_i // 2
    packed = _out(packed, (rows, I // 2), gu.device, "packed")
    sf = _out(sf, (rows, I // 16), gu.device, "sf")
    off_p, E = _offsets_arg(expert_offsets, gu.device)
    with _torch().cuda.device(gu.device):
        rc = load_library().moe_swiglu_nvfp4_quantize(
            ctypes.c_void_p(gu.data_ptr()), rows, I, float(clamp_L), off_p, E,
            ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(sf.data_ptr()),
            _stream_ptr(stream))
    _check(rc, "moe_swiglu_nvfp4_quantize")
    return packed, sf


def moe_swiglu_nvfp4_quantize_counted(gu, clamp_L: float, counters, expert_offsets=None,
                                      packed=None, sf=None, stream=None):
    """As moe_swiglu_nvfp4_quantize, adding to `counters` (int64 CUDA [3]):
    blocks processed, scale re-evaluations, nibble re-evaluations."""
    torch = _torch()
    gu = _bf16_bits(gu, "gu", 32)
    rows, two_i = gu.shape
    I = two_i // 2
    if counters.dtype != torch.int64 or counters.numel() != 3 or not counters.is_cuda:
        raise ValueError("counters must be an int64 CUDA tensor of 3 elements")
    packed = _out(packed, (rows, I // 2), gu.device, "packed")
    sf = _out(sf, (rows, I // 16), gu.device, "sf")
    off_p, E = _offsets_arg(expert_offsets, gu.device)
    with torch.cuda.device(gu.device):
        rc = load_library().moe_swiglu_nvfp4_quantize_counted(
            ctypes.c_void_p(gu.data_ptr()), rows, I, float(clamp_L), off_p, E,
            ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(sf.data_ptr()),
            ctypes.c_void_p(counters.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_swiglu_nvfp4_quantize_counted")
    return packed, sf


def moe_swiglu_fast_values(gu, clamp_L: float, stream=None):
    """Diagnostic: the fused kernel's fast-path fp32 SwiGLU values [rows, I]."""
    torch = _torch()
    gu = _bf16_bits(gu, "gu", 32)
    rows, two_i = gu.shape
    y = torch.empty((rows, two_i // 2), dtype=torch.float32, device=gu.device)
    with torch.cuda.device(gu.device):
        rc = load_library().moe_swiglu_fast_values(
            ctypes.c_void_p(gu.data_ptr()), rows, two_i // 2, float(clamp_L),
            ctypes.c_void_p(y.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_swiglu_fast_values")
    return y


def moe_swiglu_precise_values(gu, clamp_L: float, stream=None):
    """Diagnostic: the definition-path fp32 SwiGLU values [rows, I] (what the
    fused kernel uses inside its decision window)."""
    torch = _torch()
    gu = _bf16_bits(gu, "gu", 32)
    rows, two_i = gu.shape
    y = torch.empty((rows, two_i // 2), dtype=torch.float32, device=gu.device)
    with torch.cuda.device(gu.device):
        rc = load_library().moe_swiglu_precise_values(
            ctypes.c_void_p(gu.data_ptr()), rows, two_i // 2, float(clamp_L),
            ctypes.c_void_p(y.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_swiglu_precise_values")
    return y


def moe_nvfp4_e4m3_codes(x, stream=None):
    """Diagnostic: the kernels' E4M3 scale conversion of every value of a
    float32 CUDA tensor (uint8 codes, same shape)."""
    torch = _torch()
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32):
        raise TypeError("x must be a float32 CUDA tensor")
    x = x.contiguous()
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        rc = load_library().moe_nvfp4_e4m3_codes(ctypes.c_void_p(x.data_ptr()), x.numel(),
                                                 ctypes.c_void_p(codes.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_nvfp4_e4m3_codes")
    return codes


def moe_nvfp4_quantize_scaled(x, global_scale: float, packed=None, sf=None, stream=None):
    """Two-level quantize-only: NVFP4 of v = fl(x * global_scale)."""
    x = _bf16_bits(x, "x", 16)
    rows, K = x.shape
    packed = _out(packed, (rows, K // 2), x.device, "packed")
    sf = _out(sf, (rows, K // 16), x.device, "sf")
    with _torch().cuda.device(x.device):
        rc = load_library().moe_nvfp4_quantize_scaled(
            ctypes.c_void_p(x.data_ptr()), rows, K, float(global_scale),
            ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(sf.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_nvfp4_quantize_scaled")
    return packed, sf


def moe_swiglu_nvfp4_quantize_ex(gu, clamp_L: float, expert_offsets=None, global_scale=1.0,
                                 round_to_bf16=False, out_offsets=None, out_rows=None,
                                 packed=None, sf=None, stream=None):
    """The fused step with a global scale, the BF16-compat mode and padded
    per-expert output rows (out_offsets: int32 CUDA [E+1], out_rows rows)."""
    torch = _torch()
    gu = _bf16_bits(gu, "gu", 32)
    rows, two_i = gu.shape
    I = two_i // 2
    orows = rows
    ooff_p = None
    if out_offsets is not None:
        if out_rows is None:
            raise ValueError("out_rows is required with out_offsets")
        if (not out_offsets.is_cuda or out_offsets.dtype != torch.int32
                or not out_offsets.is_contiguous()):
            raise ValueError("out_offsets must be a contiguous int32 CUDA tensor")
        orows = int(out_rows)
        ooff_p = out_offsets.data_ptr()
    packed = _out(packed, (orows, I // 2), gu.device, "packed")
    sf = _out(sf, (orows, I // 16), gu.device, "sf")
    off_p, E = _offsets_arg(expert_offsets, gu.device)
    opt = FusedOptions(float(global_scale), 1 if round_to_bf16 else 0, ooff_p, orows)
    with torch.cuda.device(gu.device):
        rc = load_library().moe_swiglu_nvfp4_quantize_ex(
            ctypes.c_void_p(gu.data_ptr()), rows, I, float(clamp_L), off_p, E, ctypes.byref(opt),
            ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(sf.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_swiglu_nvfp4_quantize_ex")
    return packed, sf


def moe_swiglu_bf16(gu, clamp_L: float, expert_offsets=None, out=None, stream=None):
    """Compact writer: the BF16-rounded SwiGLU [rows, I] (torch.bfloat16)."""
    torch = _torch()
    gu = _bf16_bits(gu, "gu", 32)
    rows, two_i = gu.shape
    I = two_i // 2
    if out is None:
        out = torch.empty((rows, I), dtype=torch.bfloat16, device=gu.device)
    elif out.dtype != torch.bfloat16 or tuple(out.shape) != (rows, I) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous bfloat16 tensor of shape {(rows, I)}")
    off_p, E = _offsets_arg(expert_offsets, gu.device)
    with torch.cuda.device(gu.device):
        rc = load_library().moe_swiglu_bf16(
            ctypes.c_void_p(gu.data_ptr()), rows, I, float(clamp_L), off_p, E,
            ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_swiglu_bf16")
    return out


def moe_nvfp4_dequantize(packed, sf, global_scale=1.0, out=None, stream=None):
    """NVFP4 -> BF16 [rows, K]: RN_bf16(e2m1 * e4m3 / global_scale)."""
    torch = _torch()
    if packed.dtype != torch.uint8 or sf.dtype != torch.uint8 or packed.dim() != 2 \
            or not packed.is_cuda or not packed.is_contiguous() or not sf.is_contiguous():
        raise ValueError("packed and sf must be contiguous uint8 CUDA tensors")
    rows, half = packed.shape
    K = 2 * half
    if tuple(sf.shape) != (rows, K // 16):
        raise ValueError(f"sf must have shape {(rows, K // 16)}")
    if out is None:
        out = torch.empty((rows, K), dtype=torch.bfloat16, device=packed.device)
    with torch.cuda.device(packed.device):
        rc = load_library().moe_nvfp4_dequantize(
            ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(sf.data_ptr()), rows, K,
            float(global_scale), ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_nvfp4_dequantize")
    return out


# ---------------------------------------------------------------------------
# The step in the L1 GEMM's epilogue
# ---------------------------------------------------------------------------

def _gemm_operands(x, w1, expert_offsets):
    torch = _torch()
    x = _bf16_bits(x, "x", 64)
    if not w1.is_cuda or w1.dtype not in (torch.bfloat16, torch.uint16, torch.int16) \
            or w1.dim() != 3 or not w1.is_contiguous():
        raise ValueError("w1 must be a contiguous BF16 CUDA tensor [experts, 2I, H]")
    E, two_i, H = w1.shape
    if H != x.shape[1]:
        raise ValueError("w1.shape[2] must equal x.shape[1]")
    if two_i % 256:
        raise ValueError("w1.shape[1] (2I) must be a multiple of 256")
    if expert_offsets is None or expert_offsets.dtype != torch.int32 or not expert_offsets.is_cuda \
            or tuple(expert_offsets.shape) != (E + 1,):
        raise ValueError(f"expert_offsets must be an int32 CUDA tensor of shape ({E + 1},)")
    return x, w1, E, two_i // 2, H


def moe_l1_gemm_swiglu_nvfp4(x, w1, clamp_L: float, expert_offsets, packed=None, sf=None, status=None,
                             stream=None):
    """The fused L1 GEMM: for every expert segment, gu = x_e @ w1[e]^T in
    fp32, and straight from the accumulators the clamped SwiGLU of its
    [gate x8, up x8] groups and its NVFP4 quantization.
    x BF16 [rows, H]; w1 BF16 [E, 2I, H]; expert_offsets int32 [E+1] (device).
    Returns (packed uint8 [rows, I/2], sf uint8 [rows, I/16]); `status`, an
    optional int32 CUDA tensor [1], receives a nonzero code if a wait expired."""
    x, w1, E, I, H = _gemm_operands(x, w1, expert_offsets)
    rows = x.shape[0]
    packed = _out(packed, (rows, I // 2), x.device, "packed")
    sf = _out(sf, (rows, I // 16), x.device, "sf")
    with _torch().cuda.device(x.device):
        rc = load_library().moe_l1_gemm_swiglu_nvfp4(
            ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w1.data_ptr()), rows, H, I, float(clamp_L),
            ctypes.c_void_p(expert_offsets.data_ptr()), E, ctypes.c_void_p(packed.data_ptr()),
            ctypes.c_void_p(sf.data_ptr()), ctypes.c_void_p(0 if status is None else status.data_ptr()),
            _stream_ptr(stream))
    _check(rc, "moe_l1_gemm_swiglu_nvfp4")
    return packed, sf


def moe_l1_gemm_accumulators(x, w1, expert_offsets, acc=None, status=None, stream=None):
    """Diagnostic: the same GEMM's fp32 accumulators [rows, 2I] (rows of
    the segments written, others untouched)."""
    torch = _torch()
    x, w1, E, I, H = _gemm_operands(x, w1, expert_offsets)
    rows = x.shape[0]
    if acc is None:
        acc = torch.zeros((rows, 2 * I), dtype=torch.float32, device=x.device)
    elif acc.dtype != torch.float32 or tuple(acc.shape) != (rows, 2 * I) or not acc.is_contiguous():
        raise ValueError(f"acc must be a contiguous float32 CUDA tensor of shape {(rows, 2 * I)}")
    with torch.cuda.device(x.device):
        rc = load_library().moe_l1_gemm_accumulators(
            ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w1.data_ptr()), rows, H, I,
            ctypes.c_void_p(expert_offsets.data_ptr()), E, ctypes.c_void_p(acc.data_ptr()),
            ctypes.c_void_p(0 if status is None else status.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_l1_gemm_accumulators")
    return acc


def moe_l1_gemm_bf16(x, w1, expert_offsets, output: str = "gu", clamp_L: float = 7.0, out=None,
                     status=None, stream=None):
    """The same GEMM writing the BF16 tensors of the unfused flows:
    output="gu" -> gu [rows, 2I] ([gate x8, up x8] columns), output="swiglu"
    -> the SwiGLU [rows, I] (clamp_L used only there). Rows outside the
    segments are left untouched."""
    torch = _torch()
    x, w1, E, I, H = _gemm_operands(x, w1, expert_offsets)
    rows = x.shape[0]
    sel = {"gu": 0, "swiglu": 1}[output]
    width = 2 * I if sel == 0 else I
    if out is None:
        out = torch.zeros((rows, width), dtype=torch.bfloat16, device=x.device)
    elif out.dtype not in (torch.bfloat16, torch.int16, torch.uint16) or tuple(out.shape) != (rows, width) \
            or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous BF16 CUDA tensor of shape {(rows, width)}")
    with torch.cuda.device(x.device):
        rc = load_library().moe_l1_gemm_bf16(
            ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w1.data_ptr()), rows, H, I, float(clamp_L),
            ctypes.c_void_p(expert_offsets.data_ptr()), E, sel, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(0 if status is None else status.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_l1_gemm_bf16")
    return out


SELFTEST_MODES = {"no_loads": 1, "no_release": 2}


def moe_l1_gemm_wait_selftest(x, w1, expert_offsets, status, wait_cycles: int, packed=None, sf=None,
                              stream=None, mode: str = "no_loads"):
    """Diagnostic of the failure path: the fused GEMM with every wait limited
    to wait_cycles and a wait that can never complete (mode "no_loads": the
    producer issues nothing; "no_release": the epilogue never frees an
    accumulator, one CTA runs every tile); `status` (int32 CUDA tensor [1])
    receives the code of the wait that expired."""
    x, w1, E, I, H = _gemm_operands(x, w1, expert_offsets)
    rows = x.shape[0]
    packed = _out(packed, (rows, I // 2), x.device, "packed")
    sf = _out(sf, (rows, I // 16), x.device, "sf")
    with _torch().cuda.device(x.device):
        rc = load_library().moe_l1_gemm_wait_selftest(
            ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w1.data_ptr()), rows, H, I,
            ctypes.c_void_p(expert_offsets.data_ptr()), E, ctypes.c_void_p(packed.data_ptr()),
            ctypes.c_void_p(sf.data_ptr()), ctypes.c_void_p(status.data_ptr()), int(wait_cycles),
            SELFTEST_MODES[mode], _stream_ptr(stream))
    _check(rc, "moe_l1_gemm_wait_selftest")
    return packed, sf


def _w4_operands(x, w1_packed, w1_sf, expert_offsets):
    torch = _torch()
    x = _bf16_bits(x, "x", 256)
    rows, H = x.shape
    for t, name in ((w1_packed, "w1_packed"), (w1_sf, "w1_sf")):
        if not t.is_cuda or t.dtype != torch.uint8 or t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor [experts, 2I, ...]")
    E, two_i, half = w1_packed.shape
    if half * 2 != H or tuple(w1_sf.shape) != (E, two_i, H // 16) or two_i % 256:
        raise ValueError("w1_packed must be [E, 2I, H/2] and w1_sf [E, 2I, H/16], 2I % 256 == 0")
    if expert_offsets is None or expert_offsets.dtype != torch.int32 or not expert_offsets.is_cuda \
            or tuple(expert_offsets.shape) != (E + 1,):
        raise ValueError(f"expert_offsets must be an int32 CUDA tensor of shape ({E + 1},)")
    return x, E, two_i // 2, H


def moe_l1_gemm_w4_swiglu_nvfp4(x, w1_packed, w1_sf, clamp_L: float, expert_offsets, packed=None, sf=None,
                                status=None, stream=None):
    """The fused L1 GEMM with NVFP4 weights (packed nibbles [E, 2I, H/2] and
    E4M3 scales [E, 2I, H/16], as moe_nvfp4_quantize lays them out)."""
    x, E, I, H = _w4_operands(x, w1_packed, w1_sf, expert_offsets)
    rows = x.shape[0]
    packed = _out(packed, (rows, I // 2), x.device, "packed")
    sf = _out(sf, (rows, I // 16), x.device, "sf")
    with _torch().cuda.device(x.device):
        rc = load_library().moe_l1_gemm_w4_swiglu_nvfp4(
            ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w1_packed.data_ptr()),
            ctypes.c_void_p(w1_sf.data_ptr()), rows, H, I, float(clamp_L),
            ctypes.c_void_p(expert_offsets.data_ptr()), E, ctypes.c_void_p(packed.data_ptr()),
            ctypes.c_void_p(sf.data_ptr()), ctypes.c_void_p(0 if status is None else status.data_ptr()),
            _stream_ptr(stream))
    _check(rc, "moe_l1_gemm_w4_swiglu_nvfp4")
    return packed, sf


def moe_l1_gemm_w4_accumulators(x, w1_packed, w1_sf, expert_offsets, acc=None, status=None, stream=None):
    torch = _torch()
    x, E, I, H = _w4_operands(x, w1_packed, w1_sf, expert_offsets)
    rows = x.shape[0]
    if acc is None:
        acc = torch.zeros((rows, 2 * I), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        rc = load_library().moe_l1_gemm_w4_accumulators(
            ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w1_packed.data_ptr()),
            ctypes.c_void_p(w1_sf.data_ptr()), rows, H, I, ctypes.c_void_p(expert_offsets.data_ptr()), E,
            ctypes.c_void_p(acc.data_ptr()), ctypes.c_void_p(0 if status is None else status.data_ptr()),
            _stream_ptr(stream))
    _check(rc, "moe_l1_gemm_w4_accumulators")
    return acc


# ---------------------------------------------------------------------------
# Diagnostics
# ---------------------------------------------------------------------------

def moe_nvfp4_traffic_floor(kind: str, src=None, width: int = 0, packed=None, sf=None, stream=None):
    """The memory traffic of a step without its arithmetic, in the step's
    launch shape: kind "fused" (src BF16 [rows, 2*width]) or "quantize" (src
    BF16 [rows, width]) writes packed [rows, width/2] and sf [rows, width/16];
    "empty" launches one idle CTA; "read" sweeps src (read only) and XORs it
    into packed (uint8 CUDA, >= 4 bytes)."""
    torch = _torch()
    code = TRAFFIC_KINDS[kind]
    z = ctypes.c_void_p(0)
    dev = src.device if src is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        if kind == "empty":
            rc = load_library().moe_nvfp4_traffic_floor(z, 0, 0, code, z, z, _stream_ptr(stream))
        elif kind == "read":
            n = src.numel() * src.element_size() // 2
            rc = load_library().moe_nvfp4_traffic_floor(
                ctypes.c_void_p(src.data_ptr()), n // 16, 16, code, ctypes.c_void_p(packed.data_ptr()), z,
                _stream_ptr(stream))
        else:
            rows = src.shape[0]
            rc = load_library().moe_nvfp4_traffic_floor(
                ctypes.c_void_p(src.data_ptr()), rows, int(width), code, ctypes.c_void_p(packed.data_ptr()),
                ctypes.c_void_p(sf.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_nvfp4_traffic_floor")


def moe_nvfp4_check_offsets(expert_offsets, rows: int, out_offsets=None, out_rows: int = 0, status=None,
                            stream=None):
    """Checks the offsets' preconditions on the device; returns the int32
    CUDA status word [1] with CHECK_BITS OR-ed in (0 = none violated). Pass
    a zeroed `status` to accumulate several checks."""
    torch = _torch()
    off_p, E = _offsets_arg(expert_offsets, expert_offsets.device)
    ooff = ctypes.c_void_p(0)
    if out_offsets is not None:
        o_p, E2 = _offsets_arg(out_offsets, expert_offsets.device)
        if E2 != E:
            raise ValueError("out_offsets must have as many entries as expert_offsets")
        ooff = o_p
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=expert_offsets.device)
    with torch.cuda.device(expert_offsets.device):
        rc = load_library().moe_nvfp4_check_offsets(off_p, E, int(rows), ooff, int(out_rows),
                                                    ctypes.c_void_p(status.data_ptr()), _stream_ptr(stream))
    _check(rc, "moe_nvfp4_check_offsets")
    return status
