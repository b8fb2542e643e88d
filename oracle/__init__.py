"""NVFP4 oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.

A ctypes wrapper around ``nvfp4_oracle.c``: a plain, single-threaded C99
restatement of the deinterleave + clamped-SwiGLU + NVFP4-quantize step, built
with gcc. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may import this package; the CUDA library and its Python binding
never do.

Every function is pinned in ``tests/test_oracle_pins.py`` against facts that
do not come from this code (the pages' printed values, torch's own
``float8_e4m3fn`` cast, brute-force nearest-even searches, exact rational
arithmetic and a decimal high-precision SwiGLU).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libnvfp4_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict ISO C99, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fvisibility=hidden", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    sig = {
        "bf16_to_float32": (ctypes.c_float, [ctypes.c_uint16]),
        "fp8_e4m3_from_float32": (ctypes.c_uint8, [ctypes.c_float]),
        "fp8_e4m3_to_float32": (ctypes.c_float, [ctypes.c_uint8]),
        "half_step_to_e2m1_idx": (ctypes.c_int, [ctypes.c_int]),
        "e2m1_nibble_to_float32": (ctypes.c_float, [ctypes.c_uint8]),
        "quantize_e2m1_nibble": (ctypes.c_uint8, [ctypes.c_float]),
        "swiglu_clamped": (ctypes.c_float, [ctypes.c_float, ctypes.c_float, ctypes.c_float]),
        "quantize_nvfp4_block": (None, [_P, _P, _P]),
        "quantize_nvfp4": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
        "swiglu_quantize_nvfp4": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_float, _P,
                                                 ctypes.c_int32, _P, _P]),
        "swiglu_quantize_nvfp4_blocks": (None, [_P, _I64, ctypes.c_float, _P, _P, _I64, _P, _P]),
        "quantize_nvfp4_blocks": (None, [_P, _I64, _P, _P, _I64, _P, _P]),
        "swiglu_values": (None, [_P, _I64, ctypes.c_float, _I64, _I64, _P]),
        "swiglu_clamped_array": (None, [_P, _P, _I64, ctypes.c_float, _P]),
        "quantize_element_with_scale": (ctypes.c_uint8, [ctypes.c_float, ctypes.c_uint8]),
        "fp8_e4m3_from_float32_array": (None, [_P, _I64, _P]),
        "quantize_e2m1_nibble_array": (None, [_P, _I64, _P]),
        "bf16_round": (ctypes.c_float, [ctypes.c_float]),
        "quantize_nvfp4_scaled": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_float, _P, _P]),
        "swiglu_quantize_nvfp4_ex": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_float, _P,
                                                    ctypes.c_int32, _P, _I64, ctypes.c_float,
                                                    ctypes.c_int, _P, _P]),
        "swiglu_bf16": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_float, _P, ctypes.c_int32, _P]),
        "dequantize_nvfp4": (ctypes.c_int, [_P, _P, _I64, _I64, ctypes.c_float, _P]),
        "swiglu_clamped_f64": (ctypes.c_float, [ctypes.c_double, ctypes.c_double, ctypes.c_float]),
        "swiglu_clamped_f64_array": (None, [_P, _P, _I64, ctypes.c_float, _P]),
        "quantize_nvfp4_f32": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---- scalar primitives (the pages' named functions) -------------------------

def fp8_e4m3_from_float32(v: float) -> int:
    return int(_load().fp8_e4m3_from_float32(float(np.float32(v))))


def fp8_e4m3_to_float32(code: int) -> float:
    return float(_load().fp8_e4m3_to_float32(int(code)))


def half_step_to_e2m1_idx(h: int) -> int:
    return int(_load().half_step_to_e2m1_idx(int(h)))


def e2m1_nibble_to_float32(nib: int) -> float:
    return float(_load().e2m1_nibble_to_float32(int(nib)))


def quantize_e2m1_nibble(s: float) -> int:
    return int(_load().quantize_e2m1_nibble(float(np.float32(s))))


def swiglu_clamped(g: float, u: float, L: float) -> float:
    return float(_load().swiglu_clamped(float(np.float32(g)), float(np.float32(u)),
                                        float(np.float32(L))))


def fp8_e4m3_from_float32_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.zeros(v.shape[0], np.uint8)
    _load().fp8_e4m3_from_float32_array(_ptr(v), v.shape[0], _ptr(out))
    return out


def quantize_e2m1_nibble_array(s) -> np.ndarray:
    s = np.ascontiguousarray(s, dtype=np.float32).ravel()
    out = np.zeros(s.shape[0], np.uint8)
    _load().quantize_e2m1_nibble_array(_ptr(s), s.shape[0], _ptr(out))
    return out


def quantize_element_with_scale(y: float, sf: int) -> int:
    return int(_load().quantize_element_with_scale(float(np.float32(y)), int(sf)))


def bf16_to_float32(h: int) -> float:
    return float(_load().bf16_to_float32(int(h)))


# ---- block / tensor level ----------------------------------------------------

def quantize_nvfp4_block(y) -> tuple[np.ndarray, int]:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    assert y.shape == (16,)
    packed = np.zeros(8, np.uint8)
    sf = np.zeros(1, np.uint8)
    _load().quantize_nvfp4_block(_ptr(y), _ptr(packed), _ptr(sf))
    return packed, int(sf[0])


def quantize_nvfp4(x_bf16: np.ndarray):
    """x BF16 bits uint16 [rows, K] -> (packed uint8 [rows, K/2], sf uint8 [rows, K/16])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    packed = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    rc = _load().quantize_nvfp4(_ptr(x), rows, K, _ptr(packed), _ptr(sf))
    if rc != 0:
        raise ValueError(f"oracle quantize_nvfp4 rejected shape {x.shape}")
    return packed, sf


def swiglu_quantize_nvfp4(gu_bf16: np.ndarray, clamp_L: float, offsets=None,
                          packed: np.ndarray | None = None, sf: np.ndarray | None = None):
    """gu BF16 bits uint16 [rows, 2I] -> (packed [rows, I/2], sf [rows, I/16]).

    With ``offsets`` (int32 [E+1]) only rows of some segment are written; pass
    ``packed``/``sf`` to see that the other rows are left untouched.
    """
    gu = np.ascontiguousarray(gu_bf16, dtype=np.uint16)
    rows, two_i = gu.shape
    I = two_i // 2
    if packed is None:
        packed = np.zeros((rows, I // 2), np.uint8)
    if sf is None:
        sf = np.zeros((rows, I // 16), np.uint8)
    if offsets is None:
        off_p, E = None, 0
    else:
        off = np.ascontiguousarray(offsets, dtype=np.int32)
        off_p, E = _ptr(off), off.shape[0] - 1
    rc = _load().swiglu_quantize_nvfp4(_ptr(gu), rows, I, float(clamp_L), off_p, E,
                                      _ptr(packed), _ptr(sf))
    if rc != 0:
        raise ValueError(f"oracle swiglu_quantize_nvfp4 rejected shape {gu.shape}")
    return packed, sf


def swiglu_quantize_nvfp4_blocks(gu_bf16: np.ndarray, clamp_L: float, rows_idx, blk_idx):
    """Oracle output of selected (row, block) pairs: (packed [n, 8], sf [n])."""
    gu = np.ascontiguousarray(gu_bf16, dtype=np.uint16)
    I = gu.shape[1] // 2
    r = np.ascontiguousarray(rows_idx, dtype=np.int64)
    b = np.ascontiguousarray(blk_idx, dtype=np.int64)
    n = r.shape[0]
    packed = np.zeros((n, 8), np.uint8)
    sf = np.zeros(n, np.uint8)
    _load().swiglu_quantize_nvfp4_blocks(_ptr(gu), I, float(clamp_L), _ptr(r), _ptr(b), n,
                                         _ptr(packed), _ptr(sf))
    return packed, sf


def quantize_nvfp4_blocks(x_bf16: np.ndarray, rows_idx, blk_idx):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    K = x.shape[1]
    r = np.ascontiguousarray(rows_idx, dtype=np.int64)
    b = np.ascontiguousarray(blk_idx, dtype=np.int64)
    n = r.shape[0]
    packed = np.zeros((n, 8), np.uint8)
    sf = np.zeros(n, np.uint8)
    _load().quantize_nvfp4_blocks(_ptr(x), K, _ptr(r), _ptr(b), n, _ptr(packed), _ptr(sf))
    return packed, sf


def swiglu_values(gu_bf16: np.ndarray, clamp_L: float, r0: int = 0, r1: int | None = None):
    """fp32 SwiGLU values of rows [r0, r1) in output-column order: [r1-r0, I]."""
    gu = np.ascontiguousarray(gu_bf16, dtype=np.uint16)
    rows, two_i = gu.shape
    I = two_i // 2
    r1 = rows if r1 is None else r1
    y = np.zeros((r1 - r0, I), np.float32)
    _load().swiglu_values(_ptr(gu), I, float(clamp_L), r0, r1, _ptr(y))
    return y


def swiglu_clamped_array(g, u, clamp_L: float) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float32).ravel()
    u = np.ascontiguousarray(u, dtype=np.float32).ravel()
    assert g.shape == u.shape
    y = np.zeros_like(g)
    _load().swiglu_clamped_array(_ptr(g), _ptr(u), g.shape[0], float(clamp_L), _ptr(y))
    return y


# ---- extensions: two-level scale, BF16 compat / compact, padded segments,
#      dequantization (each a reading of the pages; see nvfp4_oracle.c) ----

def bf16_round(v: float) -> float:
    return float(_load().bf16_round(float(np.float32(v))))


def quantize_nvfp4_scaled(x_bf16: np.ndarray, gs: float):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    packed = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    if _load().quantize_nvfp4_scaled(_ptr(x), rows, K, float(np.float32(gs)), _ptr(packed), _ptr(sf)):
        raise ValueError("oracle quantize_nvfp4_scaled rejected its arguments")
    return packed, sf


def swiglu_quantize_nvfp4_ex(gu_bf16: np.ndarray, clamp_L: float, offsets=None, out_offsets=None,
                             out_rows=None, global_scale=1.0, round_bf16=False,
                             packed=None, sf=None):
    """The fused step with the extensions; outputs have out_rows rows (the
    input's row count unless out_offsets is given)."""
    gu = np.ascontiguousarray(gu_bf16, dtype=np.uint16)
    rows, two_i = gu.shape
    I = two_i // 2
    orows = rows if out_rows is None else int(out_rows)
    if packed is None:
        packed = np.zeros((orows, I // 2), np.uint8)
    if sf is None:
        sf = np.zeros((orows, I // 16), np.uint8)
    off = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int32)
    ooff = None if out_offsets is None else np.ascontiguousarray(out_offsets, dtype=np.int32)
    E = 0 if off is None else off.shape[0] - 1
    rc = _load().swiglu_quantize_nvfp4_ex(
        _ptr(gu), rows, I, float(clamp_L), None if off is None else _ptr(off), E,
        None if ooff is None else _ptr(ooff), orows, float(np.float32(global_scale)),
        1 if round_bf16 else 0, _ptr(packed), _ptr(sf))
    if rc != 0:
        raise ValueError("oracle swiglu_quantize_nvfp4_ex rejected its arguments")
    return packed, sf


def swiglu_bf16(gu_bf16: np.ndarray, clamp_L: float, offsets=None, out=None):
    gu = np.ascontiguousarray(gu_bf16, dtype=np.uint16)
    rows, two_i = gu.shape
    I = two_i // 2
    if out is None:
        out = np.zeros((rows, I), np.uint16)
    off = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int32)
    E = 0 if off is None else off.shape[0] - 1
    if _load().swiglu_bf16(_ptr(gu), rows, I, float(clamp_L), None if off is None else _ptr(off),
                           E, _ptr(out)):
        raise ValueError("oracle swiglu_bf16 rejected its arguments")
    return out


def dequantize_nvfp4(packed: np.ndarray, sf: np.ndarray, global_scale=1.0) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    s = np.ascontiguousarray(sf, dtype=np.uint8)
    rows, half = p.shape
    K = 2 * half
    out = np.zeros((rows, K), np.uint16)
    if _load().dequantize_nvfp4(_ptr(p), _ptr(s), rows, K, float(np.float32(global_scale)), _ptr(out)):
        raise ValueError("oracle dequantize_nvfp4 rejected its arguments")
    return out


# ---- the step in the L1 GEMM's epilogue ("2026-05-28 Status", priority 3) ----

def swiglu_clamped_f64(g: float, u: float, clamp_L: float) -> float:
    return float(_load().swiglu_clamped_f64(float(g), float(u), float(np.float32(clamp_L))))


def swiglu_clamped_f64_array(g, u, clamp_L: float) -> np.ndarray:
    """Clamped SwiGLU of double inputs, each rounded once to fp32."""
    g = np.ascontiguousarray(g, dtype=np.float64).ravel()
    u = np.ascontiguousarray(u, dtype=np.float64).ravel()
    assert g.shape == u.shape
    y = np.zeros(g.shape[0], np.float32)
    _load().swiglu_clamped_f64_array(_ptr(g), _ptr(u), g.shape[0], float(clamp_L), _ptr(y))
    return y


def quantize_nvfp4_f32(y: np.ndarray):
    """fp32 values [rows, K] -> (packed [rows, K/2], sf [rows, K/16])."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    rows, K = y.shape
    packed = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    if _load().quantize_nvfp4_f32(_ptr(y), rows, K, _ptr(packed), _ptr(sf)):
        raise ValueError("oracle quantize_nvfp4_f32 rejected its arguments")
    return packed, sf


def _bf16_as_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def l1_gemm_accumulators(x_bf16, w1_bf16, offsets) -> np.ndarray:
    """gu [rows, 2I] in float64: for expert e, rows [offsets[e], offsets[e+1])
    of x times w1[e]^T. The products of BF16 values are exact in double and a
    library matmul sums them, so each value is within ~2^-40 of sum |x w| of
    the exact one. Rows outside every segment are NaN."""
    x = _bf16_as_f64(x_bf16)
    E, two_i, H = w1_bf16.shape
    rows = x.shape[0]
    off = np.clip(np.asarray(offsets, np.int64), 0, rows)
    acc = np.full((rows, two_i), np.nan)
    for e in range(E):
        r0, r1 = int(off[e]), max(int(off[e]), int(off[e + 1]))
        if r1 > r0:
            acc[r0:r1] = x[r0:r1] @ _bf16_as_f64(w1_bf16[e]).T
    return acc


def l1_gemm_abs_accumulators(x_bf16, w1_bf16, offsets) -> np.ndarray:
    """sum_k |x[r, k] w1[e, c, k]| per accumulator (the scale of its rounding)."""
    x = np.abs(_bf16_as_f64(x_bf16))
    E, two_i, H = w1_bf16.shape
    rows = x.shape[0]
    off = np.clip(np.asarray(offsets, np.int64), 0, rows)
    out = np.full((rows, two_i), np.nan)
    for e in range(E):
        r0, r1 = int(off[e]), max(int(off[e]), int(off[e + 1]))
        if r1 > r0:
            out[r0:r1] = x[r0:r1] @ np.abs(_bf16_as_f64(w1_bf16[e])).T
    return out


def gemm_swiglu_values(acc: np.ndarray, clamp_L: float) -> np.ndarray:
    """Deinterleave gu's [gate x8, up x8] column groups ("NVFP4-1.1 Approach
    Update") and apply the clamped SwiGLU to the (double) accumulators:
    output column c takes gate gu[:, 16*(c//8) + c%8], up 8 columns on."""
    rows, two_i = acc.shape
    I = two_i // 2
    c = np.arange(I)
    gate_col = 16 * (c // 8) + c % 8
    g = np.ascontiguousarray(acc[:, gate_col])
    u = np.ascontiguousarray(acc[:, gate_col + 8])
    return swiglu_clamped_f64_array(g, u, clamp_L).reshape(rows, I)


def l1_gemm_swiglu_quantize_nvfp4(x_bf16, w1_bf16, offsets, clamp_L: float, packed=None, sf=None,
                                  acc=None):
    """The fused L1 GEMM output: NVFP4 of SwiGLU(gu) for the rows of the
    segments; other rows of packed / sf are left as given. `acc` (float64
    [rows, 2I]) replaces the exact accumulators when given."""
    if acc is None:
        acc = l1_gemm_accumulators(x_bf16, w1_bf16, offsets)
    rows, two_i = acc.shape
    I = two_i // 2
    packed = np.zeros((rows, I // 2), np.uint8) if packed is None else packed.copy()
    sf = np.zeros((rows, I // 16), np.uint8) if sf is None else sf.copy()
    off = np.clip(np.asarray(offsets, np.int64), 0, rows)
    for e in range(len(off) - 1):
        r0, r1 = int(off[e]), max(int(off[e]), int(off[e + 1]))
        if r1 > r0:
            p, s = quantize_nvfp4_f32(gemm_swiglu_values(acc[r0:r1], clamp_L))
            packed[r0:r1] = p
            sf[r0:r1] = s
    return packed, sf
