// Device helpers shared by the activation-step kernels and the L1 GEMM
// epilogue: PTX wrappers (streaming loads and stores, programmatic dependent
// launch, the E4M3 / E2M1 / BF16 conversions), the exact NVFP4 quantization
// of 16 fp32 values, and the packed fp32x2 SwiGLU and half-step arithmetic.
// Format rules as on the nvfp4-megamoe-kernel pages ("2026-05-28 Status",
// commit "NVFP4-1.1: FP4 quantization primitives"; "NVFP4-1.1 Approach,
// Part 2"). Every function is inline; each translation unit gets its own.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>

namespace nvfp4dev {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kHalfStepBias = 6291456.0f;        // 1.5 * 2^22: fp32 spacing 0.5 there
constexpr float kNegLog2e = -1.44269504088896341f;
constexpr float kInv6 = 0.16666667163372039794921875f;   // RN(1/6)

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 32 bytes, read once: bypass L1, evict first from L2.
__device__ __forceinline__ void load_stream_32B(const void* p, uint64_t pol, uint32_t* r) {
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]),
          "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "l"(p), "l"(pol));
}

// 32 bytes through the read-only path, bypassing L1, default L2 policy.
__device__ __forceinline__ void load_nc_32B(const void* p, uint32_t* r) {
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]),
          "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "l"(p));
}

__device__ __forceinline__ void load_stream_16B(const void* p, uint64_t pol, uint32_t* r) {
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "l"(p), "l"(pol));
}

__device__ __forceinline__ void store_32B(void* p, const uint32_t* r) {
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]),
                    "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]) : "memory");
}

// The same with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void store_32B_hint(void* p, const uint32_t* r, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]),
                    "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "l"(pol) : "memory");
}

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible (a no-op without a programmatic
// dependency), then let the next grid start launching.
__device__ __forceinline__ void wait_for_preceding_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_next_grid_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Per 16-bit half, the smaller unsigned value.
__device__ __forceinline__ uint32_t u16x2_min(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two fp32 -> two E4M3 codes, RNE, saturating: `hi` in bits 8-15, `lo` in 0-7.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// E4M3 code (low byte) -> its value, exactly (via f16, which holds every E4M3).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code)));
    return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
}

// Eight signed half steps (exact multiples of 0.5; magnitudes above 6
// saturate to 6) -> eight E2M1 nibbles, element 0 in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
    uint32_t r;
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Two fp32 -> BF16x2 (RNE): `hi` in bits 16-31, `lo` in 0-15.
__device__ __forceinline__ uint32_t bf16x2_rn(float hi, float lo) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Byte `k` (0..3) of w, two E2M1 nibbles -> their values as f16x2 (low
// nibble in the low half).
template <int k>
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t w) {
    uint32_t h;
    if (k == 0) asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b0; }" : "=r"(h) : "r"(w));
    if (k == 1) asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b1; }" : "=r"(h) : "r"(w));
    if (k == 2) asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b2; }" : "=r"(h) : "r"(w));
    if (k == 3) asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b3; }" : "=r"(h) : "r"(w));
    return h;
}

// ---------------------------------------------------------------------------
// Scalar pieces
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float with_sign_of(float mag, float s) {
    return __uint_as_float(__float_as_uint(mag) | (__float_as_uint(s) & 0x80000000u));
}

// max |v_i| over 16 values, as a tree of 3-input maxima.
__device__ __forceinline__ float abs_max16(const float* v) {
    const float m0 = max3(fabsf(v[0]), fabsf(v[1]), fabsf(v[2]));
    const float m1 = max3(fabsf(v[3]), fabsf(v[4]), fabsf(v[5]));
    const float m2 = max3(fabsf(v[6]), fabsf(v[7]), fabsf(v[8]));
    const float m3 = max3(fabsf(v[9]), fabsf(v[10]), fabsf(v[11]));
    const float m4 = max3(fabsf(v[12]), fabsf(v[13]), fabsf(v[14]));
    return max3(max3(m0, m1, m2), max3(m3, m4, fabsf(v[15])), 0.0f);
}

// a / 6, correctly rounded: q0 = a * RN(1/6) is within an ulp, the residual
// a - 6 q0 is exact in one fma, and one correction step rounds correctly
// (Markstein's theorem for a reciprocal rounded to nearest).
__device__ __forceinline__ float div6(float a) {
    const float q0 = a * kInv6;
    const float r = fmaf(-q0, 6.0f, a);
    return fmaf(r, kInv6, q0);
}

// Exact NVFP4 quantization of 16 fp32 values (the definition's decisions):
// amax / 6 correctly rounded (Markstein correction with RN(1/6)), the
// hardware's RNE + saturating E4M3 cast, the correctly rounded quotient
// |v| / d by the same correction, the exact half-step rounding, and the
// hardware E2M1 cast of the signed half step. With kIeeeRcp the reciprocal
// of d is correctly rounded, which the correction needs for arbitrary fp32
// v; for BF16-valued v any reciprocal within an ulp works, because the
// corrected quotient is exact at a tie and elsewhere |v| / d sits at least
// 2^-13 (relative) away from every half-step boundary. Returns the code.
template <bool kIeeeRcp, bool kPacked>
__device__ __forceinline__ uint32_t quantize16_exact(const float* v_in, uint32_t& lo, uint32_t& hi) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = v_in[i];
    float amax = abs_max16(v);
    if (kIeeeRcp && amax > FLT_MAX) {
        // an infinity (a scaled value past FLT_MAX): clamped to +-FLT_MAX,
        // the scale and every infinite element saturate as the definition's
#pragma unroll
        for (int i = 0; i < 16; i++) v[i] = fminf(fmaxf(v[i], -FLT_MAX), FLT_MAX);
        amax = FLT_MAX;
    }
    const float q = div6(amax);
    const uint32_t code = e4m3x2_rn_sat(0.0f, q) & 0xFFu;
    const float d = e4m3_value(code);
    const float inv = (code == 0u) ? 0.0f : (kIeeeRcp ? __frcp_rn(d) : rcp_approx(d));
    float hs[16];
    if (kPacked) {
        // signed quotient v / d corrected as above (every step is odd in v,
        // so its magnitude is the one |v| / d would give), then the signed
        // half step: the bias is an even number of half steps, so RN(q +
        // bias) - bias rounds q to half steps with ties to even on both
        // sides of zero; the sign of a zero half step is taken from v
        const float2 inv2 = make_float2(inv, inv), nd2 = make_float2(-d, -d);
        const float2 bias2 = make_float2(kHalfStepBias, kHalfStepBias);
        const float2 nbias2 = make_float2(-kHalfStepBias, -kHalfStepBias);
#pragma unroll
        for (int p = 0; p < 8; p++) {
            const float2 vv = make_float2(v[2 * p], v[2 * p + 1]);
            const float2 q0 = __fmul2_rn(vv, inv2);
            const float2 q1 = __ffma2_rn(__ffma2_rn(q0, nd2, vv), inv2, q0);
            const float2 h = __fadd2_rn(__fadd2_rn(q1, bias2), nbias2);
            hs[2 * p] = copysignf(h.x, v[2 * p]);
            hs[2 * p + 1] = copysignf(h.y, v[2 * p + 1]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const float ax = fabsf(v[i]);
            const float q0 = ax * inv;
            const float q1 = fmaf(fmaf(-q0, d, ax), inv, q0);     // |v| / d, corrected
            hs[i] = with_sign_of((q1 + kHalfStepBias) - kHalfStepBias, v[i]);
        }
    }
    lo = e2m1x8(hs);
    hi = e2m1x8(hs + 8);
    return code;
}

// silu(a) * b for two elements at once: the multiplies and the add are
// packed fp32x2 instructions, each lane rounding as the scalar form does.
__device__ __forceinline__ float2 silu_times_fast2(float2 a, float2 b) {
    const float2 x = __fmul2_rn(a, make_float2(kNegLog2e, kNegLog2e));      // -a log2 e
    const float2 den = __fadd2_rn(make_float2(ex2_approx(x.x), ex2_approx(x.y)),
                                  make_float2(1.0f, 1.0f));
    return __fmul2_rn(__fmul2_rn(a, make_float2(rcp_approx(den.x), rcp_approx(den.y))), b);
}

// Half steps of t = y * inv for 16 values, two per packed instruction: hs
// (signed, ready for the E2M1 cast) and the largest |t - h|. RN(t + bias) -
// bias rounds t to half steps with ties to even on both sides of zero (the
// bias 1.5 * 2^22 is an even number of half steps and the spacing there is
// one half step); it is formed as -h = RN(-t - bias) + bias, which rounds
// identically, so that t - h is one fma. The sign of a zero half step is
// taken from y.
__device__ __forceinline__ float half_steps16(const float* y, float inv, float* hs) {
    const float2 inv2 = make_float2(inv, inv), ninv2 = make_float2(-inv, -inv);
    const float2 bias2 = make_float2(kHalfStepBias, kHalfStepBias);
    const float2 nbias2 = make_float2(-kHalfStepBias, -kHalfStepBias);
    float r[16];
#pragma unroll
    for (int p = 0; p < 8; p++) {
        const float2 yv = make_float2(y[2 * p], y[2 * p + 1]);
        const float2 nh = __fadd2_rn(__ffma2_rn(yv, ninv2, nbias2), bias2);
        const float2 rv = __ffma2_rn(yv, inv2, nh);
        hs[2 * p] = copysignf(nh.x, y[2 * p]);
        hs[2 * p + 1] = copysignf(nh.y, y[2 * p + 1]);
        r[2 * p] = rv.x;
        r[2 * p + 1] = rv.y;
    }
    return abs_max16(r);
}

}  // namespace nvfp4dev
