// GB300 (sm_103a) kernels for the MoE expert activation step: deinterleave
// the L1 GEMM's BF16 [gate x8, up x8, ...] column groups, clamped SwiGLU,
// NVFP4 quantize (E2M1 nibbles + one FP8 E4M3 scale per 16 outputs).
//
// Operations as defined on the nvfp4-megamoe-kernel pages:
//   "2026-05-28 Status", commit "NVFP4-1.1: FP4 quantization primitives":
//     E4M3 bias 7, exponents 0-15 with exp 15 / mant 7 NaN (max 448),
//     subnormals m * 2^-9, round-to-nearest-even with carry; the half-step
//     index -> E2M1 index map; quantize + sign + pack.
//   "NVFP4-1.1 Approach, Part 2": round-half-even half steps (5.25 -> 6);
//     16 values -> 8 packed bytes + 1 scale byte.
//   "NVFP4-1.1 Approach Update", "Revised approach: Compact SwiGLU output":
//     the interleaved layout, the (tokens, I/2) and (tokens, I/16) outputs,
//     and quantize-only on a compact BF16 tensor.
//
// Design (memory-bound streaming; no tensor-core work exists on this path):
//   * The problem is a 1-D stream of independent 16-output blocks: block b of
//     row r reads the 64 contiguous input bytes gu[r, 32b .. 32b+31] (or the
//     32 bytes x[r, 16b .. 16b+15]) and writes 8 packed bytes + 1 scale
//     byte, all at index r * (I/16) + b. Row boundaries never split a block,
//     so the active blocks [first, last) are split into equal contiguous
//     ranges, one per resident CTA, whose warps claim 64-block chunks from a
//     shared counter; loads are 256-bit, L1-bypassing and marked evict-first
//     in L2 (the stream is read once; the compact BF16 writer alone streams
//     faster without the hint), two blocks in flight per lane.
//   * Each thread owns whole blocks, so the amax needs no shuffles.
//   * E4M3 scale: cvt.rn.satfinite.e4m3x2.f32 (RNE, saturating at 448);
//     E2M1 nibbles: the half step is rounded with the exact fp32 trick
//     (t + 1.5*2^22) - 1.5*2^22, then cvt.rn.satfinite.e2m1x2.f32 maps the
//     signed half step to its nibble (RNE onto the E2M1 grid is exactly the
//     pages' step_to_idx table for half-step inputs).
//   * Fused path: SwiGLU in fast fp32 (ex2.approx + rcp.approx). A scale or
//     nibble decision whose input lies within a relative window W of a
//     rounding boundary (W bounds the fast path's error, with margin) is
//     redone from the definition's value, evaluated in double-float
//     arithmetic (~46 bits) on the FP32 pipes.
//     Quantize-only: exact division by a Markstein correction
//     (q = x*rcp_rn(d), r = fma(-q, d, x), q' = fma(r, rcp_rn(d), q)).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include "moe_nvfp4.h"
#include "nvfp4_device.cuh"

namespace {

using namespace nvfp4dev;

constexpr int kThreads = 256;
constexpr int kUnroll = 2;                 // blocks in flight per lane (fused)
constexpr int kUnrollQuant = 4;            // blocks in flight per lane (quantize-only)
constexpr int kMinBlocksFused = 3;         // resident CTAs per SM the register budget targets
constexpr int kMinBlocksQuant = 3;         // quantize-only: 80 registers hold 4 blocks in flight and the packed quotients
constexpr int kMaxDevices = 64;

// The definition's value: the formula in double precision, rounded once.
__device__ __noinline__ float swiglu_double(float g, float u, float L) {
    const double a = static_cast<double>(fminf(g, L));
    const double b = static_cast<double>(fminf(fmaxf(u, -L), L));
    const double y = a / (1.0 + exp(-a)) * b;
    return __double2float_rn(y);
}

// ---------------------------------------------------------------------------
// The definition's value in double-float arithmetic
// ---------------------------------------------------------------------------
// A value is carried as the unevaluated sum hi + lo of two fp32 numbers
// (|lo| <= ulp(hi) / 2), about 46 significant bits: rounding the result to
// fp32 then agrees with a double-precision evaluation unless the exact value
// lies within ~2^-44 (relative) of an fp32 rounding midpoint. It runs on the
// FP32 pipes with a short dependency chain; GB300's FP64 pipe is narrow and
// slow, and one double-precision evaluation on a warp's critical path
// lengthens the whole launch by its latency (the last such element ends the
// kernel late). The explicit _rn intrinsics keep the compiler from fusing
// the error-free transformations into FMAs.

struct DFloat {
    float hi, lo;
};

__device__ __forceinline__ DFloat df_two_sum(float a, float b) {          // exact a + b
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

__device__ __forceinline__ DFloat df_fast_two_sum(float a, float b) {     // |a| >= |b|
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ DFloat df_two_prod(float a, float b) {         // exact a * b
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ DFloat df_add(DFloat a, DFloat b) {
    const DFloat s = df_two_sum(a.hi, b.hi);
    return df_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ DFloat df_mul(DFloat a, DFloat b) {
    const float p = __fmul_rn(a.hi, b.hi);
    float e = __fmaf_rn(a.hi, b.hi, -p);
    e = __fmaf_rn(a.hi, b.lo, e);
    e = __fmaf_rn(a.lo, b.hi, e);
    return df_fast_two_sum(p, e);
}

// ln 2 / 64 = kLn2x64Hi + kLn2x64Mid + kLn2x64Lo; the head has 9 significant
// bits, so n * head is exact for |n| < 2^15.
constexpr float kInvLn2x64 = 0x1.715476p+6f;       // 64 / ln 2
constexpr float kLn2x64Hi = 0x1.63p-7f;
constexpr float kLn2x64Mid = -0x1.bd0106p-19f;
constexpr float kLn2x64Lo = 0x1.cf79acp-46f;

// 2^(j/64) = hi + lo for j = 0..63.
__constant__ float2 kExp2Table[64] = {
    {0x1.0p+0f, 0.0f}, {0x1.02c9a4p+0f, -0x1.887fap-28f},
    {0x1.059b0ep+0f, -0x1.9d4f52p-25f}, {0x1.087452p+0f, -0x1.e2990ep-26f},
    {0x1.0b5586p+0f, 0x1.9f3122p-25f}, {0x1.0e3ec4p+0f, -0x1.a585ccp-25f},
    {0x1.11301ep+0f, -0x1.fdb496p-25f}, {0x1.1429aap+0f, 0x1.d525bcp-25f},
    {0x1.172b84p+0f, -0x1.c15742p-27f}, {0x1.1a35bep+0f, 0x1.6df96ep-25f},
    {0x1.1d4874p+0f, -0x1.d2e8cap-25f}, {0x1.2063b8p+0f, 0x1.0c519ap-25f},
    {0x1.2387a6p+0f, 0x1.ceac48p-25f}, {0x1.26b456p+0f, 0x1.789f38p-26f},
    {0x1.29e9ep+0f, -0x1.5c0424p-25f}, {0x1.2d285ap+0f, 0x1.b900c2p-26f},
    {0x1.306fep+0f, 0x1.4636e2p-25f}, {0x1.33c08cp+0f, -0x1.b37d2p-25f},
    {0x1.371a74p+0f, -0x1.18aac6p-25f}, {0x1.3a7db4p+0f, -0x1.634c02p-25f},
    {0x1.3dea64p+0f, 0x1.824684p-25f}, {0x1.4160a2p+0f, 0x1.f72e2ap-28f},
    {0x1.44e086p+0f, 0x1.8624b4p-30f}, {0x1.486a2cp+0f, -0x1.47d866p-25f},
    {0x1.4bfdaep+0f, -0x1.593abcp-25f}, {0x1.4f9b28p+0f, -0x1.2c5a6cp-25f},
    {0x1.5342b6p+0f, -0x1.2c561p-25f}, {0x1.56f474p+0f, -0x1.295b04p-25f},
    {0x1.5ab07ep+0f, -0x1.5bd5ecp-27f}, {0x1.5e76f2p+0f, -0x1.4a5bd6p-25f},
    {0x1.6247ecp+0f, -0x1.f8b55p-25f}, {0x1.662388p+0f, 0x1.2a9112p-27f},
    {0x1.6a09e6p+0f, 0x1.9fcef4p-26f}, {0x1.6dfb24p+0f, -0x1.cd72e8p-27f},
    {0x1.71f75ep+0f, 0x1.1d8beep-25f}, {0x1.75feb6p+0f, -0x1.37b306p-25f},
    {0x1.7a1148p+0f, -0x1.829fdp-25f}, {0x1.7e2f34p+0f, -0x1.261634p-25f},
    {0x1.82589ap+0f, -0x1.accc7cp-26f}, {0x1.868d9ap+0f, -0x1.2edb44p-26f},
    {0x1.8ace54p+0f, 0x1.15506ep-27f}, {0x1.8f1aeap+0f, -0x1.baa232p-26f},
    {0x1.93737cp+0f, -0x1.e64744p-25f}, {0x1.97d82ap+0f, -0x1.0d8d84p-31f},
    {0x1.9c4918p+0f, 0x1.51f848p-27f}, {0x1.a0c668p+0f, -0x1.2886a6p-26f},
    {0x1.a5503cp+0f, -0x1.b83b54p-25f}, {0x1.a9e6b6p+0f, -0x1.50c048p-25f},
    {0x1.ae89fap+0f, -0x1.a94b14p-26f}, {0x1.b33a2cp+0f, -0x1.ec3a82p-26f},
    {0x1.b7f77p+0f, -0x1.a09438p-25f}, {0x1.bcc1eap+0f, -0x1.f687c6p-25f},
    {0x1.c199bep+0f, -0x1.3d56b2p-27f}, {0x1.c67f12p+0f, 0x1.cafa2ap-25f},
    {0x1.cb720ep+0f, -0x1.8837ccp-27f}, {0x1.d072d4p+0f, 0x1.40f13p-25f},
    {0x1.d5818ep+0f, -0x1.822dbcp-27f}, {0x1.da9e6p+0f, 0x1.ed9942p-27f},
    {0x1.dfc974p+0f, -0x1.908c94p-25f}, {0x1.e502eep+0f, 0x1.e2cffep-26f},
    {0x1.ea4afap+0f, 0x1.52486cp-27f}, {0x1.efa1bep+0f, 0x1.cc2b44p-25f},
    {0x1.f50766p+0f, -0x1.246ebp-26f}, {0x1.fa7c18p+0f, 0x1.9e90d8p-28f},
};

// e^x for -100 <= x <= 80 as a double-float: x = n ln2/64 + r with
// |r| <= ln2/128, e^x = 2^(n/64) e^r, e^r by its Taylor series to r^5 (the
// r^3.. terms in fp32, the rest in double-float).
__device__ __forceinline__ DFloat exp_df(float x) {
    const float nf = rintf(__fmul_rn(x, kInvLn2x64));
    const int n = __float2int_rn(nf);
    const float r1 = __fmaf_rn(-nf, kLn2x64Hi, x);          // exact
    const DFloat t = df_two_prod(nf, kLn2x64Mid);
    DFloat r = df_two_sum(r1, -t.hi);
    r = df_fast_two_sum(r.hi, __fadd_rn(r.lo, __fmaf_rn(-nf, kLn2x64Lo, -t.lo)));
    const float rh = r.hi;
    const float tail = __fmul_rn(__fmul_rn(rh, __fmul_rn(rh, rh)),
                                 __fmaf_rn(rh, __fmaf_rn(rh, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f));
    DFloat sq = df_two_prod(rh, rh);
    sq.lo = __fmaf_rn(__fmul_rn(2.0f, rh), r.lo, sq.lo);
    const DFloat half_sq = {__fmul_rn(sq.hi, 0.5f), __fmul_rn(sq.lo, 0.5f)};
    DFloat s = df_add(half_sq, DFloat{tail, 0.0f});
    s = df_add(r, s);
    s = df_add(DFloat{1.0f, 0.0f}, s);
    const float2 tj = kExp2Table[n & 63];
    DFloat e = df_mul(DFloat{tj.x, tj.y}, s);
    const int k = n >> 6;                                      // floor(n / 64)
    e.hi = ldexpf(e.hi, k);
    e.lo = ldexpf(e.lo, k);
    return e;
}

// The definition's value: silu(min(g, L)) * clamp(u, -L, L) rounded once to
// fp32, from a double-float evaluation (a gate below -80 and results below
// 2^-100 fall back to double precision: no NVFP4 decision depends on such
// values, but a BF16 rounding can).
__device__ __noinline__ float swiglu_precise(float g, float u, float L) {
    const float a = fminf(g, L);
    const float b = fminf(fmaxf(u, -L), L);
    if (a < -80.0f) return swiglu_double(g, u, L);
    DFloat sig = {1.0f, 0.0f};                                 // e^-a underflows
    if (a <= 100.0f) {
        const DFloat den = df_add(DFloat{1.0f, 0.0f}, exp_df(-a));
        const float y0 = __frcp_rn(den.hi);
        float eps = __fmaf_rn(-den.hi, y0, 1.0f);              // exact residual
        eps = __fmaf_rn(-den.lo, y0, eps);
        sig = df_fast_two_sum(y0, __fmul_rn(y0, eps));         // 1 / (1 + e^-a)
    }
    const DFloat ab = df_two_prod(a, b);
    const DFloat y = df_mul(ab, sig);
    // near and below the fp32 subnormal range the low parts lose bits:
    // take the double-precision evaluation there
    if (fabsf(y.hi) < 0x1p-100f) return swiglu_double(g, u, L);
    return copysignf(y.hi, ab.hi);
}

// gate / up of output i (0..15) of the block starting at `blk_in`.
__device__ __forceinline__ void gate_up_at(const uint16_t* blk_in, int i, float& g, float& u) {
    const int grp = i >> 3, j = i & 7;
    g = __uint_as_float(static_cast<uint32_t>(blk_in[16 * grp + j]) << 16);
    u = __uint_as_float(static_cast<uint32_t>(blk_in[16 * grp + 8 + j]) << 16);
}

// One nibble by the definition: s = y / d (IEEE), h = RNE(2 min(|s|, 6)),
// index from the half-step table {0,1,2,3,4,4,5,6,6,6,6,7,7} (packed as
// hex digits), sign from s.
__device__ __forceinline__ uint32_t nibble_by_definition(float y, float d, uint32_t code) {
    const float s = (code == 0u) ? with_sign_of(0.0f, y) : __fdiv_rn(y, d);
    const int h = __float2int_rn(fminf(fabsf(s), 6.0f) * 2.0f);
    const uint32_t idx = static_cast<uint32_t>(0x7766665443210ull >> (4 * h)) & 0xFu;
    return idx | ((__float_as_uint(s) >> 28) & 8u);
}

// Half-step index pairs (k, k+1) whose table entries differ, as a bit mask
// over k: 0-1, 1-2, 2-3, 3-4, 5-6, 6-7, 10-11. A value near the boundary
// between any other pair gets the same nibble on both sides.
constexpr uint32_t kNibbleChangingBoundaries = 0x46Fu;

// ---------------------------------------------------------------------------
// Fused deinterleave + clamped SwiGLU + NVFP4 quantize
// ---------------------------------------------------------------------------

struct FusedArgs {
    const uint16_t* gu;        // [rows, 2I]
    int64_t rows;
    int64_t bpr;               // blocks per row = I / 16
    float L;
    uint32_t L2, negL2;        // (L, L) and (-L, -L) as BF16x2 (when L is a BF16 value)
    float W;                   // relative decision window
    float Wp1, Wm1;            // 1 + W, 1 - W
    float near_thr;            // 0.25 (1 - W)
    float near_fast;           // 0.25 (1 - W) - 7 W, rounded down: the block test
    const int32_t* offsets;    // [E+1] or null
    int E;
    uint8_t* packed;           // [rows, I/2]
    uint8_t* sf;               // [rows, I/16]
    unsigned long long* counters;   // [3] or null (counted variant)
    float* values;             // [rows, I] (fast-values variant)
};

struct Tally {
    unsigned long long blocks = 0, scales = 0, nibbles = 0;
};

__device__ __forceinline__ void active_block_range(const int32_t* offsets, int E, int64_t rows,
                                                   int64_t bpr, int64_t& b0, int64_t& b1) {
    int64_t r0 = 0, r1 = rows;
    if (offsets != nullptr) {
        const int64_t o0 = __ldg(offsets), oe = __ldg(offsets + E);
        r0 = o0 < 0 ? 0 : (o0 > rows ? rows : o0);
        r1 = oe < r0 ? r0 : (oe > rows ? rows : oe);
    }
    b0 = r0 * bpr;
    b1 = r1 * bpr;
}

// Scale code of a block whose fast amax lies within the window of an E4M3
// rounding boundary: every element that could be the true maximum is
// re-evaluated by the definition (and replaced in y), then the code is taken
// from the exact amax.
__device__ __forceinline__ uint32_t scale_by_definition(const uint16_t* blk_in, float L, float W,
                                                        float amax, float* y) {
    const float lim = amax * (1.0f - 2.0f * W);
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        if (fabsf(y[i]) >= lim) {
            float g, u;
            gate_up_at(blk_in, i, g, u);
            y[i] = swiglu_precise(g, u, L);
        }
        am = fmaxf(am, fabsf(y[i]));
    }
    return e4m3x2_rn_sat(0.0f, __fdiv_rn(am, 6.0f)) & 0xFFu;
}

// Fast SwiGLU of one block's 16 outputs from its two loaded 32-byte groups
// ([gate x8, up x8] twice): deinterleave, clamp, silu(g) u.
template <bool kBf16Clamp>
__device__ __forceinline__ void fast_swiglu16(const FusedArgs& A, const uint32_t* w, float* y) {
    const float L = A.L;
#pragma unroll
    for (int grp = 0; grp < 2; grp++) {
#pragma unroll
        for (int p = 0; p < 4; p++) {
            uint32_t gw = w[8 * grp + p], uw = w[8 * grp + 4 + p];
            float2 g, u;
            if (kBf16Clamp) {                        // clamp two values per instruction
                gw = bf16x2_min(gw, A.L2);
                uw = bf16x2_min(bf16x2_max(uw, A.negL2), A.L2);
                g = make_float2(bf16_lo(gw), bf16_hi(gw));
                u = make_float2(bf16_lo(uw), bf16_hi(uw));
            } else {
                g = make_float2(fminf(bf16_lo(gw), L), fminf(bf16_hi(gw), L));
                u = make_float2(fminf(fmaxf(bf16_lo(uw), -L), L), fminf(fmaxf(bf16_hi(uw), -L), L));
            }
            const float2 yv = silu_times_fast2(g, u);
            y[8 * grp + 2 * p] = yv.x;
            y[8 * grp + 2 * p + 1] = yv.y;
        }
    }
}

// Every lane of the warp calls this together (uniform control flow), with
// `valid` false for lanes past the end of the stream.
template <bool kCount, bool kValues, bool kBf16Clamp>
__device__ __forceinline__ void fused_block(const FusedArgs& A, int64_t blk, bool valid,
                                            const uint32_t* w, Tally& tally) {
    const float L = A.L;
    float y[16];
    fast_swiglu16<kBf16Clamp>(A, w, y);
    if (kValues) {
        if (valid) {
            float4* out = reinterpret_cast<float4*>(A.values + blk * 16);
#pragma unroll
            for (int k = 0; k < 4; k++)
                out[k] = make_float4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
        }
        return;
    }
    const uint16_t* blk_in = A.gu + blk * 32;

    // scale: safe when both ends of the window round to the same code (the
    // product by RN(1/6) is within an ulp of amax / 6, inside the window)
    const float amax = abs_max16(y);
    const float q = amax * kInv6;
    const uint32_t ends = e4m3x2_rn_sat(q * A.Wp1, q * A.Wm1);
    uint32_t code = ends & 0xFFu;
    if (valid && (ends >> 8) != code) {
        code = scale_by_definition(blk_in, L, A.W, amax, y);
        if (kCount) tally.scales++;
    }

    // nibbles: half steps of t = y / d. A t whose true value could lie
    // across a half-step boundary has |t - h| + W h > 0.25 (1 - W); past
    // the last nibble-changing boundary (t = 5.25) nothing matters, so h <= 7
    // there and max |t - h| > 0.25 (1 - W) - 7 W flags every such block
    const float d = e4m3_value(code);
    const float inv = (code == 0u) ? 0.0f : rcp_approx(d);
    float hs[16];
    const float closeness = half_steps16(y, inv, hs);
    uint32_t lo = e2m1x8(hs), hi = e2m1x8(hs + 8);

    const bool near = valid && closeness > A.near_fast;
    if (__any_sync(kFullMask, near)) {
        uint32_t todo = 0;
        if (near) {
            for (int i = 0; i < 16; i++) {
                const float ay = fabsf(y[i]);
                const float h = fmaf(ay, inv, kHalfStepBias) - kHalfStepBias;
                const float rr = fmaf(ay, inv, -h);
                if (fmaf(A.W, h, fabsf(rr)) > A.near_thr) {
                    // the boundary in question sits between half steps k and k+1
                    const int k = __float2int_rn(2.0f * h) - (rr < 0.0f ? 1 : 0);
                    if (k >= 0 && k < 12 && ((kNibbleChangingBoundaries >> k) & 1u)) todo |= 1u << i;
                }
            }
        }
        // one definition-path SwiGLU per lane per pass, all lanes together
        while (__any_sync(kFullMask, todo != 0u)) {
            if (todo != 0u) {
                const int i = __ffs(todo) - 1;
                todo &= todo - 1u;
                float g, u;
                gate_up_at(blk_in, i, g, u);
                const uint32_t nib = nibble_by_definition(swiglu_precise(g, u, L), d, code);
                const int sh = 4 * (i & 7);
                if (i < 8) lo = (lo & ~(0xFu << sh)) | (nib << sh);
                else       hi = (hi & ~(0xFu << sh)) | (nib << sh);
                if (kCount) tally.nibbles++;
            }
        }
    }
    if (valid) {
        *reinterpret_cast<uint2*>(A.packed + blk * 8) = make_uint2(lo, hi);
        A.sf[blk] = static_cast<uint8_t>(code);
        if (kCount) tally.blocks++;
    }
}

template <bool kCount, bool kValues, bool kBf16Clamp>
__global__ void __launch_bounds__(kThreads, kMinBlocksFused)
swiglu_nvfp4_kernel(const FusedArgs A) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    int64_t b0, b1;
    active_block_range(A.offsets, A.E, A.rows, A.bpr, b0, b1);
    const uint64_t pol = l2_evict_first_policy();
    const int lane = threadIdx.x & 31;
    // Each CTA owns an equal contiguous range of blocks; its warps claim
    // chunks of 32 * kUnroll blocks from a shared counter, so a warp held up
    // by a rare exact re-evaluation (or slow memory) takes fewer chunks and
    // the CTA's other warps absorb the delay.
    constexpr int64_t kChunk = 32 * kUnroll;
    const int64_t total = b1 - b0;
    int64_t per_cta = (total + gridDim.x - 1) / gridDim.x;
    per_cta = (per_cta + kChunk - 1) / kChunk * kChunk;
    const int64_t cta_begin = b0 + static_cast<int64_t>(blockIdx.x) * per_cta;
    const int64_t cta_end = cta_begin + per_cta < b1 ? cta_begin + per_cta : b1;
    __shared__ int next_chunk;
    if (threadIdx.x == 0) next_chunk = 0;
    __syncthreads();
    Tally tally;
    for (;;) {                                              // warp-uniform
        int c = 0;
        if (lane == 0) c = atomicAdd(&next_chunk, 1);
        c = __shfl_sync(kFullMask, c, 0);
        const int64_t base = cta_begin + static_cast<int64_t>(c) * kChunk;
        if (base >= cta_end) break;
        uint32_t w[kUnroll][16];
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t blk = base + 32 * k + lane;
            if (blk < cta_end) {
                const uint16_t* p = A.gu + blk * 32;
                load_stream_32B(p, pol, w[k]);
                load_stream_32B(p + 16, pol, w[k] + 8);
            } else {
#pragma unroll
                for (int j = 0; j < 16; j++) w[k][j] = 0u;
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t blk = base + 32 * k + lane;
            fused_block<kCount, kValues, kBf16Clamp>(A, blk, blk < cta_end, w[k], tally);
        }
    }
    if (kCount) {
        atomicAdd(A.counters + 0, tally.blocks);
        if (tally.scales) atomicAdd(A.counters + 1, tally.scales);
        if (tally.nibbles) atomicAdd(A.counters + 2, tally.nibbles);
    }
}

// ---------------------------------------------------------------------------
// Extensions of the fused step: two-level (global) scale, the pages' BF16
// pipeline (compat quantize and compact writer), padded per-expert output.
// A separate kernel, so the plain step above keeps its code as measured.
// ---------------------------------------------------------------------------

// kExCompatUnit: the compat mode with global scale 1, where the values to
// quantize are the BF16 numbers themselves
enum ExMode : int { kExQuantize = 0, kExCompat = 1, kExCompact = 2, kExCompatUnit = 3 };

// Fast silu's relative error against the definition's fp32 value, in units
// of 2^-24, at most kSiluErrUlps0 + kSiluErrUlpsPerGate * max(-a, 0) for
// every BF16 gate a >= -16 (measured exhaustively by the test suite: 3.0
// for positive gates at any size, up to 13.7 at a = -16).
constexpr float kSiluErrUlps0 = 4.5f;
constexpr float kSiluErrUlpsPerGate = 0.8f;

struct ExArgs {
    FusedArgs f;                    // f.W and its derived fields include the global-scale product
    float gs;                       // global scale (1: single-level)
    const int32_t* out_offsets;     // [E+1] or null: padded output rows
    int64_t out_rows;               // rows of packed / sf
    uint16_t* out_bf16;             // compact writer output [rows, I]
    float gate_floor;               // most negative gate the window's bound covers
    uint32_t mid_tol;               // fp32 ulps a BF16 rounding midpoint must be away
    int mid_tol_per_block;          // 1: derive it per block from the most negative gate
};

// BF16 values of the 16 outputs by the definition (RN_bf16 of the fp32
// SwiGLU) as 8 BF16x2 words, element 2p in the low half of word p. A BF16
// rounding midpoint is the fp32 value whose low 16 bits are 0x8000; the
// window W keeps the definition's fp32 value within W |y| <= W 2^24 ulps
// of the fast value y, so when y's low half is more than mid_tol ulps from
// 0x8000 both round alike (a binade edge is 2^15 ulps from any midpoint).
// The fast pass returns the mask of elements it cannot decide; those are
// re-evaluated by resolve_bf16_elements.
__device__ __forceinline__ bool outside_window_range(float g, float u, float y, float gate_floor) {
    // the window bounds the fast path's relative error for gates >=
    // gate_floor and normal results; a BF16 rounding is scale-free, so any
    // other nonzero value is redone (a zero gate or up gives an exact +-0)
    const bool nonzero = (__float_as_uint(g) & 0x7FFFFFFFu) != 0u && (__float_as_uint(u) & 0x7FFFFFFFu) != 0u;
    return g < gate_floor || (nonzero && fabsf(y) < 0x1p-100f);
}

__device__ __forceinline__ uint32_t near_bf16_midpoint(float y, uint32_t c16, uint32_t t16) {
    return (__float_as_uint(y) * 0x10000u + c16 <= t16) ? 1u : 0u;
}

__device__ __forceinline__ uint32_t bf16_fast_of_block(const ExArgs& X, bool valid, const uint32_t* w,
                                                       const float* y, uint32_t* yb) {
    const uint32_t gmin2 = bf16x2_min(bf16x2_min(bf16x2_min(w[0], w[1]), bf16x2_min(w[2], w[3])),
                                      bf16x2_min(bf16x2_min(w[8], w[9]), bf16x2_min(w[10], w[11])));
    const float gmin = fminf(bf16_lo(gmin2), bf16_hi(gmin2));
    // the tolerance for this block: 1.5 x (the silu bound at its most
    // negative gate + 2 for the product and the definition's rounding),
    // plus one for the threshold and one for a value on it; blocks with a
    // gate below -16 keep the clamp's global tolerance
    uint32_t tol = X.mid_tol;
    if (X.mid_tol_per_block && gmin >= -16.0f) {
        const float e = fmaf(kSiluErrUlpsPerGate, fmaxf(-gmin, 0.0f), kSiluErrUlps0 + 2.0f);
        const uint32_t t = static_cast<uint32_t>(ceilf(1.5f * e)) + 2u;
        tol = t < tol ? t : tol;
    }
    // ((bits + tol - 0x8000) mod 2^16) <= 2 tol, computed in the top half
    const uint32_t c16 = (tol - 0x8000u) << 16, t16 = ((2u * tol) << 16) | 0xFFFFu;
    uint32_t amb = 0;
#pragma unroll
    for (int q = 0; q < 8; q++) {
        yb[q] = bf16x2_rn(y[2 * q + 1], y[2 * q]);
        amb |= (near_bf16_midpoint(y[2 * q], c16, t16) << (2 * q)) |
               (near_bf16_midpoint(y[2 * q + 1], c16, t16) << (2 * q + 1));
    }
    // block pre-test for the window's range (gates below the floor, results
    // near underflow); element by element only when it fires
    float ymin = fabsf(y[0]);
#pragma unroll
    for (int i = 1; i < 16; i++) ymin = fminf(ymin, fabsf(y[i]));
    if (gmin < X.gate_floor || ymin < 0x1p-100f) {
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const int grp = i >> 3, pw = (i & 7) >> 1;
            const uint32_t gw = w[8 * grp + pw], uw = w[8 * grp + 4 + pw];
            const float g = (i & 1) ? bf16_hi(gw) : bf16_lo(gw);
            const float u = (i & 1) ? bf16_hi(uw) : bf16_lo(uw);
            amb |= (outside_window_range(g, u, y[i], X.gate_floor) ? 1u : 0u) << i;
        }
    }
    return valid ? amb : 0u;
}

// Re-evaluates the undecided elements of kN / 16 blocks (block k of this
// lane at blk0 + 32 k, element i as bit 16 k + i of `elems`) by the
// definition path. The warp works through them together: every lane takes
// its next element each round, so the rounds are the largest count on one
// lane.
template <int kN>
__device__ __forceinline__ void resolve_bf16_elements(const FusedArgs& A, int64_t blk0, uint32_t elems,
                                                      uint32_t* yb) {
    static_assert(kN <= 32, "one bit per element");
    while (__any_sync(kFullMask, elems != 0u)) {
        if (elems != 0u) {
            const int j = __ffs(elems) - 1;
            elems &= elems - 1u;
            float g, u;
            gate_up_at(A.gu + (blk0 + 32 * (j >> 4)) * 32, j & 15, g, u);
            const uint32_t h = bf16x2_rn(0.0f, swiglu_precise(g, u, A.L));   // low half
            const uint32_t keep = (j & 1) ? 0x0000FFFFu : 0xFFFF0000u;
            const uint32_t put = (j & 1) ? (h << 16) : h;
            // the word is picked by a one-hot mask: a chain of `t == j / 2`
            // tests is folded into one indexed store, which moves the whole
            // array to local memory
            const uint32_t onehot = 1u << (j >> 1);
#pragma unroll
            for (int t = 0; t < kN / 2; t++)
                if (onehot & (1u << t)) yb[t] = (yb[t] & keep) | put;
        }
    }
}

// The two-level fused step for one block: v = y * gs, then the plain step's
// fast decisions and exact path on v.
__device__ __forceinline__ void scaled_block(const ExArgs& X, const uint16_t* blk_in, bool valid,
                                             const float* y, uint32_t& lo, uint32_t& hi,
                                             uint32_t& code) {
    const FusedArgs& A = X.f;
    const float L = A.L, gs = X.gs;
    float v[16];
#pragma unroll
    for (int p = 0; p < 8; p++) {
        const float2 vv = __fmul2_rn(make_float2(y[2 * p], y[2 * p + 1]), make_float2(gs, gs));
        v[2 * p] = vv.x;
        v[2 * p + 1] = vv.y;
    }
    const float amax = abs_max16(v);
    const float q = amax * kInv6;
    const uint32_t ends = e4m3x2_rn_sat(q * A.Wp1, q * A.Wm1);
    code = ends & 0xFFu;
    if (valid && (ends >> 8) != code) {
        const float lim = amax * (1.0f - 2.0f * A.W);
        float am = 0.0f;
        for (int i = 0; i < 16; i++) {
            if (fabsf(v[i]) >= lim) {
                float g, u;
                gate_up_at(blk_in, i, g, u);
                am = fmaxf(am, fabsf(__fmul_rn(swiglu_precise(g, u, L), gs)));
            }
        }
        code = e4m3x2_rn_sat(0.0f, __fdiv_rn(am, 6.0f)) & 0xFFu;
    }
    const float d = e4m3_value(code);
    const float inv = (code == 0u) ? 0.0f : rcp_approx(d);
    float hs[16];
    const float closeness = half_steps16(v, inv, hs);      // flags as in the plain step
    lo = e2m1x8(hs);
    hi = e2m1x8(hs + 8);
    const bool near = valid && closeness > A.near_fast;
    if (__any_sync(kFullMask, near)) {
        uint32_t todo = 0;
        if (near) {
            for (int i = 0; i < 16; i++) {
                const float av = fabsf(v[i]);
                const float h = fmaf(av, inv, kHalfStepBias) - kHalfStepBias;
                const float rr = fmaf(av, inv, -h);
                if (fmaf(A.W, h, fabsf(rr)) > A.near_thr) {
                    const int k = __float2int_rn(2.0f * h) - (rr < 0.0f ? 1 : 0);
                    if (k >= 0 && k < 12 && ((kNibbleChangingBoundaries >> k) & 1u)) todo |= 1u << i;
                }
            }
        }
        while (__any_sync(kFullMask, todo != 0u)) {
            if (todo != 0u) {
                const int i = __ffs(todo) - 1;
                todo &= todo - 1u;
                float g, u;
                gate_up_at(blk_in, i, g, u);
                const uint32_t nib =
                    nibble_by_definition(__fmul_rn(swiglu_precise(g, u, L), gs), d, code);
                const int sh = 4 * (i & 7);
                if (i < 8) lo = (lo & ~(0xFu << sh)) | (nib << sh);
                else       hi = (hi & ~(0xFu << sh)) | (nib << sh);
            }
        }
    }
}

// Segment of row r: the largest e with offsets[e] <= r (offsets
// non-decreasing, r inside [offsets[0], offsets[E])).
__device__ __forceinline__ int segment_of(const int32_t* offsets, int E, int64_t r) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(__ldg(offsets + mid)) <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// A thread's current segment for padded output, in blocks (row r starts at
// block r * bpr, so row >= R exactly when block >= R * bpr): the first
// block past the segment, the blocks [lo, hi) whose output row lies inside
// [0, out_rows), and the output block minus the input block.
struct alignas(32) PadSegment {
    int64_t end_blk, lo_blk, hi_blk, shift_blk;
};

template <int kMode, bool kBf16Clamp, bool kPadded>
__global__ void __launch_bounds__(kThreads, kMinBlocksFused)
swiglu_ex_kernel(const ExArgs X) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const FusedArgs& A = X.f;
    int64_t b0, b1;
    active_block_range(A.offsets, A.E, A.rows, A.bpr, b0, b1);
    const uint64_t pol = l2_evict_first_policy();
    const int lane = threadIdx.x & 31;
    constexpr int64_t kChunk = 32 * kUnroll;
    const int64_t total = b1 - b0;
    int64_t per_cta = (total + gridDim.x - 1) / gridDim.x;
    per_cta = (per_cta + kChunk - 1) / kChunk * kChunk;
    const int64_t cta_begin = b0 + static_cast<int64_t>(blockIdx.x) * per_cta;
    const int64_t cta_end = cta_begin + per_cta < b1 ? cta_begin + per_cta : b1;
    const bool padded = kPadded && X.out_offsets != nullptr && A.offsets != nullptr;
    // padded output: each thread's current segment (and its index) lives in
    // shared memory and is read at the store, so nothing of it is live
    // across the arithmetic
    __shared__ int next_chunk;
    __shared__ PadSegment pad_seg[kThreads];
    __shared__ int32_t pad_e[kThreads];
    if (threadIdx.x == 0) next_chunk = 0;
    if (padded) {
        pad_seg[threadIdx.x] = PadSegment{-1, 0, 0, 0};
        pad_e[threadIdx.x] = -1;
    }
    __syncthreads();
    for (;;) {                                              // warp-uniform
        int c = 0;
        if (lane == 0) c = atomicAdd(&next_chunk, 1);
        c = __shfl_sync(kFullMask, c, 0);
        const int64_t base = cta_begin + static_cast<int64_t>(c) * kChunk;
        if (base >= cta_end) break;
        uint32_t w[kUnroll][16];
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t blk = base + 32 * k + lane;
            if (blk < cta_end) {
                const uint16_t* p = A.gu + blk * 32;
                if (kMode == kExCompact) {
                    // the compact writer (2 output bytes per 4 input bytes)
                    // streams 8 % faster with plain loads; the quantizing
                    // modes are faster with the evict-first hint
                    load_nc_32B(p, w[k]);
                    load_nc_32B(p + 16, w[k] + 8);
                } else {
                    load_stream_32B(p, pol, w[k]);
                    load_stream_32B(p + 16, pol, w[k] + 8);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; j++) w[k][j] = 0u;
            }
        }
        // output block of block blk: its padded position and whether it is
        // stored (called by the whole warp after the block's arithmetic)
        auto out_block = [&](int64_t blk, bool valid, int64_t& oblk, bool& store) {
            oblk = blk;
            store = valid;
            if (!padded) return;
            PadSegment sg = pad_seg[threadIdx.x];
            if (valid && blk >= sg.end_blk) {               // once per segment
                // a thread's blocks only move forward: step on from its
                // segment, else bisect
                int e = pad_e[threadIdx.x];
                const int64_t row = blk / A.bpr;
                for (int t = 0; e >= 0 && t < 4 && e + 1 < A.E && row >= __ldg(A.offsets + e + 1); t++)
                    e++;
                if (e < 0 || (e + 1 < A.E && row >= __ldg(A.offsets + e + 1)))
                    e = segment_of(A.offsets, A.E, row);
                // rows are int32, so the stored-row range is clamped to [0, 2^31]
                const int64_t shift = static_cast<int64_t>(__ldg(X.out_offsets + e)) - __ldg(A.offsets + e);
                const int64_t lo = -shift, hi = X.out_rows - shift, top = int64_t(1) << 31;
                sg.end_blk = static_cast<int64_t>(__ldg(A.offsets + e + 1)) * A.bpr;
                sg.lo_blk = (lo < 0 ? 0 : (lo > top ? top : lo)) * A.bpr;
                sg.hi_blk = (hi < 0 ? 0 : (hi > top ? top : hi)) * A.bpr;
                sg.shift_blk = shift * A.bpr;
                pad_seg[threadIdx.x] = sg;
                pad_e[threadIdx.x] = e;
            }
            store = valid && blk >= sg.lo_blk && blk < sg.hi_blk;
            oblk = blk + sg.shift_blk;
        };
        if (kMode == kExQuantize) {
#pragma unroll
            for (int k = 0; k < kUnroll; k++) {
                const int64_t blk = base + 32 * k + lane;
                const bool valid = blk < cta_end;
                float y[16];
                fast_swiglu16<kBf16Clamp>(A, w[k], y);
                uint32_t lo, hi, code;
                scaled_block(X, A.gu + blk * 32, valid, y, lo, hi, code);
                int64_t oblk;
                bool store;
                out_block(blk, valid, oblk, store);
                if (store) {
                    *reinterpret_cast<uint2*>(A.packed + oblk * 8) = make_uint2(lo, hi);
                    A.sf[oblk] = static_cast<uint8_t>(code);
                }
            }
        } else {
            // BF16 values: fast pass over all blocks, one joint re-evaluation
            // of the undecided pairs, then store or quantize
            uint32_t yb[8 * kUnroll];
            uint32_t elems = 0;
#pragma unroll
            for (int k = 0; k < kUnroll; k++) {
                float y[16];
                fast_swiglu16<kBf16Clamp>(A, w[k], y);
                elems |= bf16_fast_of_block(X, base + 32 * k + lane < cta_end, w[k], y, yb + 8 * k)
                         << (16 * k);
            }
            resolve_bf16_elements<16 * kUnroll>(A, base + lane, elems, yb);
#pragma unroll
            for (int k = 0; k < kUnroll; k++) {
                const int64_t blk = base + 32 * k + lane;
                const bool valid = blk < cta_end;
                const uint32_t* b = yb + 8 * k;
                if (kMode == kExCompact) {
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(X.out_bf16 + blk * 16);
                        dst[0] = make_uint4(b[0], b[1], b[2], b[3]);
                        dst[1] = make_uint4(b[4], b[5], b[6], b[7]);
                    }
                } else {                                // compat: quantize the BF16 values
                    float v[16];
                    uint32_t lo, hi, code;
                    if (kMode == kExCompatUnit) {               // BF16 values: the cheap exact form
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            v[2 * q] = bf16_lo(b[q]);
                            v[2 * q + 1] = bf16_hi(b[q]);
                        }
                        code = quantize16_exact<false, true>(v, lo, hi);
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            const float2 vv = __fmul2_rn(make_float2(bf16_lo(b[q]), bf16_hi(b[q])),
                                                         make_float2(X.gs, X.gs));
                            v[2 * q] = vv.x;
                            v[2 * q + 1] = vv.y;
                        }
                        code = quantize16_exact<true, true>(v, lo, hi);
                    }
                    int64_t oblk;
                    bool store;
                    out_block(blk, valid, oblk, store);
                    if (store) {
                        *reinterpret_cast<uint2*>(A.packed + oblk * 8) = make_uint2(lo, hi);
                        A.sf[oblk] = static_cast<uint8_t>(code);
                    }
                }
            }
        }
    }
}

// Diagnostic: the kernels' E4M3 conversion (cvt.rn.satfinite.e4m3x2.f32,
// the scale step) applied to n fp32 values, two per instruction.
__global__ void e4m3_codes_kernel(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ codes) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const int64_t pairs = (n + 1) / 2;
    for (int64_t p = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; p < pairs;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = 2 * p;
        const float lo = x[i], hi = (i + 1 < n) ? x[i + 1] : 0.0f;
        const uint32_t r = e4m3x2_rn_sat(hi, lo);
        codes[i] = static_cast<uint8_t>(r & 0xFFu);
        if (i + 1 < n) codes[i + 1] = static_cast<uint8_t>(r >> 8);
    }
}

// Diagnostic: the definition-path SwiGLU value of every output element.
__global__ void swiglu_precise_values_kernel(const uint16_t* __restrict__ gu, int64_t rows,
                                             int64_t I, float L, float* __restrict__ y) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const int64_t n = rows * I;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = idx / I, c = idx % I;
        const uint16_t* row = gu + r * 2 * I;
        const int64_t gc = 16 * (c / 8) + (c % 8);
        const float g = __uint_as_float(static_cast<uint32_t>(row[gc]) << 16);
        const float u = __uint_as_float(static_cast<uint32_t>(row[gc + 8]) << 16);
        y[idx] = swiglu_precise(g, u, L);
    }
}

// ---------------------------------------------------------------------------
// Quantize-only
// ---------------------------------------------------------------------------

template <bool kScaled>
__global__ void __launch_bounds__(kThreads, kMinBlocksQuant)
nvfp4_quantize_kernel(const uint16_t* __restrict__ x, int64_t nblk, float gs,
                      uint8_t* __restrict__ packed, uint8_t* __restrict__ sf) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const uint64_t pol = l2_evict_first_policy();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t step = (static_cast<int64_t>(gridDim.x) * kThreads >> 5) * 32 * kUnrollQuant;
    for (int64_t base = warp * 32 * kUnrollQuant; base < nblk; base += step) {
        uint32_t w[kUnrollQuant][8];
#pragma unroll
        for (int k = 0; k < kUnrollQuant; k++) {
            const int64_t blk = base + 32 * k + lane;
            if (blk < nblk) load_stream_32B(x + blk * 16, pol, w[k]);
        }
#pragma unroll
        for (int k = 0; k < kUnrollQuant; k++) {
            const int64_t blk = base + 32 * k + lane;
            if (blk >= nblk) continue;
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; i++) {
                v[i] = (i & 1) ? bf16_hi(w[k][i >> 1]) : bf16_lo(w[k][i >> 1]);
                if (kScaled) v[i] = __fmul_rn(v[i], gs);          // two-level: v = fl(x * gs)
            }
            uint32_t lo, hi;
            // packed quotient steps (the register budget of 3 CTAs per SM
            // holds them and the 4 blocks in flight without spilling)
            const uint32_t code = quantize16_exact<kScaled, true>(v, lo, hi);
            *reinterpret_cast<uint2*>(packed + blk * 8) = make_uint2(lo, hi);
            sf[blk] = static_cast<uint8_t>(code);
        }
    }
}

// ---------------------------------------------------------------------------
// Dequantization: NVFP4 -> BF16, value = e2m1 * e4m3 / gs
// ---------------------------------------------------------------------------

enum DequantDivision { kDivNone = 0, kDivMarkstein = 1, kDivIeee = 2 };

// One 16-element block: 8 packed bytes (p), scale value d -> 16 BF16 values.
template <int kDiv>
__device__ __forceinline__ void dequantize_block(uint2 p, float d, float gs, float inv_gs,
                                                 uint16_t* dst16) {
    uint32_t o[8];
#pragma unroll
    for (int half = 0; half < 2; half++) {
        const uint32_t w = half ? p.y : p.x;
        const uint32_t h2[4] = {e2m1x2_to_f16x2<0>(w), e2m1x2_to_f16x2<1>(w),
                                e2m1x2_to_f16x2<2>(w), e2m1x2_to_f16x2<3>(w)};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            // e2m1 * e4m3 is exact in fp32 (at most 6 significant bits)
            float v[2] = {__half2float(__ushort_as_half(static_cast<uint16_t>(h2[k] & 0xFFFFu))) * d,
                          __half2float(__ushort_as_half(static_cast<uint16_t>(h2[k] >> 16))) * d};
#pragma unroll
            for (int t = 0; t < 2; t++) {
                if (kDiv == kDivMarkstein) {
                    // Markstein: with inv = RN(1/gs) and q0 = RN(a * inv) within
                    // one ulp of a/gs, r = a - q0*gs is exact and RN(q0 + r*inv)
                    // is RN(a/gs) while every quantity stays normal (the host
                    // takes this path only for such gs). The sign of a zero is
                    // restored explicitly.
                    const float q0 = v[t] * inv_gs;
                    v[t] = copysignf(fmaf(fmaf(-q0, gs, v[t]), inv_gs, q0), v[t]);
                } else if (kDiv == kDivIeee) {
                    v[t] = __fdiv_rn(v[t], gs);
                }
            }
            o[4 * half + k] = bf16x2_rn(v[1], v[0]);
        }
    }
    store_32B(dst16, o);
}

// Lanes take consecutive pairs of blocks, so every load and store of a warp
// covers whole 32-byte sectors: 16 packed bytes and 2 scale bytes in, two
// 32-byte stores out. Two pairs per lane are in flight in each iteration; an
// odd last block is done at the end.
template <int kDiv>
__global__ void __launch_bounds__(kThreads)
nvfp4_dequantize_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ sf,
                        int64_t nblk, float gs, uint16_t* __restrict__ out) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const float inv_gs = kDiv == kDivMarkstein ? __frcp_rn(gs) : 1.0f;
    const uint64_t pol = l2_evict_first_policy();
    const int64_t npair = nblk / 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    constexpr int kPairs = 2;
    for (int64_t p0 = tid; p0 < npair; p0 += kPairs * stride) {
        uint32_t w[kPairs][4];
        uint32_t s2[kPairs];
#pragma unroll
        for (int k = 0; k < kPairs; k++) {
            const int64_t pi = p0 + k * stride;
            if (pi < npair) {
                load_stream_16B(packed + pi * 16, pol, w[k]);
                s2[k] = __ldg(reinterpret_cast<const uint16_t*>(sf + 2 * pi));
            }
        }
#pragma unroll
        for (int k = 0; k < kPairs; k++) {
            const int64_t pi = p0 + k * stride;
            if (pi < npair) {
                dequantize_block<kDiv>(make_uint2(w[k][0], w[k][1]), e4m3_value(s2[k] & 0xFFu), gs,
                                       inv_gs, out + pi * 32);
                dequantize_block<kDiv>(make_uint2(w[k][2], w[k][3]), e4m3_value(s2[k] >> 8), gs,
                                       inv_gs, out + pi * 32 + 16);
            }
        }
    }
    if ((nblk & 1) && tid == 0) {
        const int64_t blk = nblk - 1;
        dequantize_block<kDiv>(*reinterpret_cast<const uint2*>(packed + blk * 8), e4m3_value(sf[blk]),
                               gs, inv_gs, out + blk * 16);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int occ[2][3] = {{0, 0, 0}, {0, 0, 0}};   // [bf16 clamp][plain, counted, values]
    int occ_ex[2][7] = {};          // [bf16 clamp][ExMode, then padded kExQuantize, kExCompat, kExCompatUnit]
    int occ_quant[2] = {0, 0};                  // [scaled]
    int occ_dequant = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

template <bool kBf16Clamp>
bool fused_occupancy(int* occ) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[0], swiglu_nvfp4_kernel<false, false, kBf16Clamp>, kThreads, 0) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[1], swiglu_nvfp4_kernel<true, false, kBf16Clamp>, kThreads, 0) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[2], swiglu_nvfp4_kernel<false, true, kBf16Clamp>, kThreads, 0) == cudaSuccess;
}

template <bool kBf16Clamp>
bool ex_occupancy(int* occ) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[0], swiglu_ex_kernel<kExQuantize, kBf16Clamp, false>, kThreads, 0) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[1], swiglu_ex_kernel<kExCompat, kBf16Clamp, false>, kThreads, 0) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[2], swiglu_ex_kernel<kExCompact, kBf16Clamp, false>, kThreads, 0) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[3], swiglu_ex_kernel<kExCompatUnit, kBf16Clamp, false>, kThreads, 0) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[4], swiglu_ex_kernel<kExQuantize, kBf16Clamp, true>, kThreads, 0) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[5], swiglu_ex_kernel<kExCompat, kBf16Clamp, true>, kThreads, 0) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(
               &occ[6], swiglu_ex_kernel<kExCompatUnit, kBf16Clamp, true>, kThreads, 0) == cudaSuccess;
}

int device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_NVFP4_ELAUNCH;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_NVFP4_ELAUNCH;
        if (!fused_occupancy<false>(di.occ[0]) || !fused_occupancy<true>(di.occ[1]) ||
            !ex_occupancy<false>(di.occ_ex[0]) || !ex_occupancy<true>(di.occ_ex[1]) ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_quant[0], nvfp4_quantize_kernel<false>, kThreads, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_quant[1], nvfp4_quantize_kernel<true>, kThreads, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_dequant, nvfp4_dequantize_kernel<kDivMarkstein>, kThreads, 0) != cudaSuccess)
            return MOE_NVFP4_ELAUNCH;
        di.ready = true;
    }
    out = di;
    return MOE_NVFP4_OK;
}

// Persistent grid: enough warps for the work, at most the resident CTAs.
int grid_for(int64_t nblk, int sms, int occ, int unroll = kUnroll) {
    const int64_t per_cta = static_cast<int64_t>(kThreads) * unroll;
    const int64_t want = (nblk + per_cta - 1) / per_cta;
    const int64_t cap = static_cast<int64_t>(sms) * (occ > 0 ? occ : 1);
    return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_common(const void* in, int64_t rows, int64_t width, int64_t in_bytes_per_elem,
                 const void* out0, const void* out1) {
    if (rows < 0) return MOE_NVFP4_ESIZE;
    if (width <= 0 || width % 16 != 0) return MOE_NVFP4_EWIDTH;
    // rows * width * in_bytes_per_elem must fit in int64
    if (rows > 0 && width > INT64_MAX / in_bytes_per_elem / rows) return MOE_NVFP4_ESIZE;
    if (rows == 0) return MOE_NVFP4_OK;
    if (in == nullptr || out0 == nullptr || out1 == nullptr) return MOE_NVFP4_ENULL;
    if (!aligned(in, 32) || !aligned(out0, 16) || !aligned(out1, 16)) return MOE_NVFP4_EALIGN;
    return MOE_NVFP4_OK;
}

// Largest relative error of the fast fp32 silu(a) = a * rcp(1 + ex2(-a log2 e))
// against the definition's fp32 value, over every BF16 gate a >= -16 (the
// test suite measures it exhaustively on the GPU and checks this bound).
constexpr double kFastSiluMaxRelErr = 8.5e-7;
constexpr double kFastSiluGateFloor = -16.0;

// The most negative gate for which window_for(L) bounds the fast error.
double window_gate_floor(float L) {
    const double target = std::ldexp(1.0, -12) / static_cast<double>(L);
    double z = 1.0;
    if (target < std::exp(-1.0)) {
        double lo = 1.0, hi = 200.0;
        for (int it = 0; it < 200; it++) {
            const double mid = 0.5 * (lo + hi);
            if (mid * std::exp(-mid) >= target) lo = mid; else hi = mid;
        }
        z = hi;
    }
    return -z >= kFastSiluGateFloor ? kFastSiluGateFloor : -z;
}

double window_for(float L) {
    if (!std::isfinite(L) || !(L > 0.0f) || static_cast<double>(L) > 18446744073709551616.0) return -1.0;
    // Largest z = -a for which a gate a < 0 can still give |y| >= 2^-12, the
    // smallest magnitude that reaches the first nibble boundary (0.25 * 2^-9,
    // the smallest nonzero scale) with margin: |y| <= z e^-z * L.
    const double target = std::ldexp(1.0, -12) / static_cast<double>(L);
    double z = 1.0;
    if (target < std::exp(-1.0)) {
        double lo = 1.0, hi = 200.0;
        for (int it = 0; it < 200; it++) {
            const double mid = 0.5 * (lo + hi);
            if (mid * std::exp(-mid) >= target) lo = mid; else hi = mid;
        }
        z = hi;
    }
    const double u24 = std::ldexp(1.0, -24);
    if (-z >= kFastSiluGateFloor) {
        // every gate that matters lies in the measured range: the measured
        // silu error, plus the product with the up value, the definition's
        // own rounding of y, the approximate reciprocal of the scale (one
        // ulp) -- with a 1.5x margin
        return 1.5 * (kFastSiluMaxRelErr + 5.0 * u24);
    }
    // otherwise an analytic bound: exponent-argument rounding (|x| 1.22 2^-24
    // in x = -a log2 e, times ln 2 in exp), ex2.approx (<= 2^-21), and nine
    // fp32 roundings / approximate reciprocals on the way from y to t,
    // doubled for margin
    const double x_max = z * 1.4426950408889634;
    return 2.0 * (x_max * 0.85 * u24 + std::ldexp(1.0, -21) + 9.0 * u24);
}

// BF16 bits of L when L is exactly a BF16 value, else -1.
int64_t bf16_bits_of(float L) {
    uint32_t b;
    std::memcpy(&b, &L, 4);
    if ((b & 0xFFFFu) != 0u) return -1;
    return static_cast<int64_t>(b >> 16);
}

// Launch with programmatic stream serialization, so this grid's launch
// overlaps the tail of the preceding one (each kernel above waits for it
// before touching memory).
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), int grid, cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <bool kBf16Clamp>
void launch_fused_kernel(const FusedArgs& A, int64_t nblk, const DeviceInfo& di, bool counted,
                         bool values, cudaStream_t stream) {
    const int* occ = di.occ[kBf16Clamp ? 1 : 0];
    if (values) {
        launch(swiglu_nvfp4_kernel<false, true, kBf16Clamp>, grid_for(nblk, di.sms, occ[2]), stream, A);
    } else if (counted) {
        launch(swiglu_nvfp4_kernel<true, false, kBf16Clamp>, grid_for(nblk, di.sms, occ[1]), stream, A);
    } else {
        launch(swiglu_nvfp4_kernel<false, false, kBf16Clamp>, grid_for(nblk, di.sms, occ[0]), stream, A);
    }
}

bool valid_scale(float gs) { return std::isfinite(gs) && gs > 0.0f; }

// Fills the fused-step arguments for clamp L and window W.
FusedArgs fused_args(const uint16_t* gu, int64_t rows, int64_t I, float L, double W,
                     const int32_t* offsets, int32_t E, uint8_t* packed, uint8_t* sf) {
    FusedArgs A;
    A.gu = gu; A.rows = rows; A.bpr = I / 16; A.L = L;
    const int64_t lb = bf16_bits_of(L);
    const int64_t nlb = bf16_bits_of(-L);
    A.L2 = lb < 0 ? 0u : static_cast<uint32_t>(lb) * 0x00010001u;
    A.negL2 = nlb < 0 ? 0u : static_cast<uint32_t>(nlb) * 0x00010001u;
    A.W = static_cast<float>(W);
    A.Wp1 = static_cast<float>(1.0 + W);
    A.Wm1 = static_cast<float>(1.0 - W);
    A.near_thr = static_cast<float>(0.25 * (1.0 - W));
    A.near_fast = std::nextafter(static_cast<float>(0.25 * (1.0 - W) - 7.0 * W), 0.0f);
    A.offsets = (E > 0) ? offsets : nullptr; A.E = E;
    A.packed = packed; A.sf = sf;
    A.counters = nullptr; A.values = nullptr;
    return A;
}

template <bool kBf16Clamp>
void launch_ex_kernel(const ExArgs& X, int mode, int64_t nblk, const DeviceInfo& di,
                      cudaStream_t stream) {
    const int* occ = di.occ_ex[kBf16Clamp ? 1 : 0];
    const bool padded = X.out_offsets != nullptr && X.f.offsets != nullptr;
    if (mode == kExQuantize && padded)
        launch(swiglu_ex_kernel<kExQuantize, kBf16Clamp, true>, grid_for(nblk, di.sms, occ[4]), stream, X);
    else if (mode == kExQuantize)
        launch(swiglu_ex_kernel<kExQuantize, kBf16Clamp, false>, grid_for(nblk, di.sms, occ[0]), stream, X);
    else if (mode == kExCompat && X.gs == 1.0f && padded)
        launch(swiglu_ex_kernel<kExCompatUnit, kBf16Clamp, true>, grid_for(nblk, di.sms, occ[6]), stream, X);
    else if (mode == kExCompat && X.gs == 1.0f)
        launch(swiglu_ex_kernel<kExCompatUnit, kBf16Clamp, false>, grid_for(nblk, di.sms, occ[3]), stream, X);
    else if (mode == kExCompat && padded)
        launch(swiglu_ex_kernel<kExCompat, kBf16Clamp, true>, grid_for(nblk, di.sms, occ[5]), stream, X);
    else if (mode == kExCompat)
        launch(swiglu_ex_kernel<kExCompat, kBf16Clamp, false>, grid_for(nblk, di.sms, occ[1]), stream, X);
    else
        launch(swiglu_ex_kernel<kExCompact, kBf16Clamp, false>, grid_for(nblk, di.sms, occ[2]), stream, X);
}

int launch_ex(const uint16_t* gu, int64_t rows, int64_t I, float L, const int32_t* offsets,
              int32_t E, float gs, int mode, const int32_t* out_offsets, int64_t out_rows,
              uint8_t* packed, uint8_t* sf, uint16_t* out_bf16, cudaStream_t stream) {
    int rc;
    if (mode == kExCompact) rc = check_common(gu, rows, I, 4, out_bf16, out_bf16);
    else rc = check_common(gu, rows, I, 4, packed, sf);
    if (rc != MOE_NVFP4_OK) return rc;
    double W = window_for(L);
    if (W < 0.0) return MOE_NVFP4_ECLAMP;
    if (!valid_scale(gs)) return MOE_NVFP4_ESCALE;
    if (E < 0 || (E > 0 && offsets == nullptr)) return MOE_NVFP4_EOFFSETS;
    if (out_offsets != nullptr && E == 0) return MOE_NVFP4_EOFFSETS;
    if (out_offsets != nullptr && out_rows < 0) return MOE_NVFP4_ESIZE;
    if ((E > 0 && !aligned(offsets, 4)) || (out_offsets != nullptr && !aligned(out_offsets, 4)))
        return MOE_NVFP4_EALIGN;
    if (rows == 0) return MOE_NVFP4_OK;
    DeviceInfo di;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    // BF16 roundings compare the fast value itself: W |y| <= W 2^24 ulps,
    // plus one for the threshold and one for a value on it
    const double mid_tol = std::ceil(W * 16777216.0) + 2.0;
    // the product with gs rounds once on each side of the comparison
    W += 1.5 * 2.0 * std::ldexp(1.0, -24);
    ExArgs X;
    X.f = fused_args(gu, rows, I, L, W, offsets, E, packed, sf);
    X.gs = gs;
    X.out_offsets = (mode == kExCompact) ? nullptr : out_offsets;
    X.out_rows = out_offsets != nullptr ? out_rows : rows;
    X.out_bf16 = out_bf16;
    X.gate_floor = static_cast<float>(window_gate_floor(L));
    X.mid_tol = mid_tol > 32767.0 ? 32767u : static_cast<uint32_t>(mid_tol);
    // the per-gate silu bound was measured with gates clamped at 100
    X.mid_tol_per_block = L <= 100.0f ? 1 : 0;
    const int64_t nblk = rows * (I / 16);
    if (bf16_bits_of(L) >= 0) launch_ex_kernel<true>(X, mode, nblk, di, stream);
    else launch_ex_kernel<false>(X, mode, nblk, di, stream);
    return cudaGetLastError() == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

int launch_fused(const uint16_t* gu, int64_t rows, int64_t I, float L, const int32_t* offsets,
                 int32_t E, uint8_t* packed, uint8_t* sf, uint64_t* counters, float* values,
                 cudaStream_t stream) {
    int rc;
    if (values != nullptr) rc = check_common(gu, rows, I, 4, values, values);
    else rc = check_common(gu, rows, I, 4, packed, sf);
    if (rc != MOE_NVFP4_OK) return rc;
    const double W = window_for(L);
    if (W < 0.0) return MOE_NVFP4_ECLAMP;
    if (E < 0 || (E > 0 && offsets == nullptr)) return MOE_NVFP4_EOFFSETS;
    if (E > 0 && !aligned(offsets, 4)) return MOE_NVFP4_EALIGN;
    if (rows == 0) return MOE_NVFP4_OK;
    DeviceInfo di;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    FusedArgs A;
    A.gu = gu; A.rows = rows; A.bpr = I / 16; A.L = L;
    const int64_t lb = bf16_bits_of(L);
    const int64_t nlb = bf16_bits_of(-L);
    A.L2 = lb < 0 ? 0u : static_cast<uint32_t>(lb) * 0x00010001u;
    A.negL2 = nlb < 0 ? 0u : static_cast<uint32_t>(nlb) * 0x00010001u;
    A.W = static_cast<float>(W);
    A.Wp1 = static_cast<float>(1.0 + W);
    A.Wm1 = static_cast<float>(1.0 - W);
    A.near_thr = static_cast<float>(0.25 * (1.0 - W));
    A.near_fast = std::nextafter(static_cast<float>(0.25 * (1.0 - W) - 7.0 * W), 0.0f);
    A.offsets = (E > 0) ? offsets : nullptr; A.E = E;
    A.packed = packed; A.sf = sf;
    A.counters = reinterpret_cast<unsigned long long*>(counters); A.values = values;
    const int64_t nblk = rows * (I / 16);
    if (lb >= 0) launch_fused_kernel<true>(A, nblk, di, counters != nullptr, values != nullptr, stream);
    else launch_fused_kernel<false>(A, nblk, di, counters != nullptr, values != nullptr, stream);
    return cudaGetLastError() == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

}  // namespace

extern "C" {

int moe_nvfp4_quantize(const uint16_t* x, int64_t rows, int64_t K, uint8_t* packed, uint8_t* sf,
                       moe_nvfp4_stream_t stream) {
    int rc = check_common(x, rows, K, 2, packed, sf);
    if (rc != MOE_NVFP4_OK || rows == 0) return rc;
    DeviceInfo di;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    const int64_t nblk = rows * (K / 16);
    launch(nvfp4_quantize_kernel<false>, grid_for(nblk, di.sms, di.occ_quant[0], kUnrollQuant),
           reinterpret_cast<cudaStream_t>(stream), x, nblk, 1.0f, packed, sf);
    return cudaGetLastError() == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

int moe_swiglu_nvfp4_quantize(const uint16_t* gu, int64_t rows, int64_t I, float clamp_L,
                              const int32_t* expert_offsets, int32_t num_experts,
                              uint8_t* packed, uint8_t* sf, moe_nvfp4_stream_t stream) {
    return launch_fused(gu, rows, I, clamp_L, expert_offsets, num_experts, packed, sf, nullptr,
                        nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int moe_swiglu_fast_values(const uint16_t* gu, int64_t rows, int64_t I, float clamp_L, float* y,
                           moe_nvfp4_stream_t stream) {
    if (rows > 0 && y == nullptr) return MOE_NVFP4_ENULL;
    return launch_fused(gu, rows, I, clamp_L, nullptr, 0, nullptr, nullptr, nullptr, y,
                        reinterpret_cast<cudaStream_t>(stream));
}

int moe_swiglu_precise_values(const uint16_t* gu, int64_t rows, int64_t I, float clamp_L,
                               float* y, moe_nvfp4_stream_t stream) {
    int rc = check_common(gu, rows, I, 4, y, y);
    if (rc != MOE_NVFP4_OK) return rc;
    if (window_for(clamp_L) < 0.0) return MOE_NVFP4_ECLAMP;
    if (rows == 0) return MOE_NVFP4_OK;
    DeviceInfo di;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    launch(swiglu_precise_values_kernel, di.sms * 8, reinterpret_cast<cudaStream_t>(stream), gu, rows,
           I, clamp_L, y);
    return cudaGetLastError() == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

int moe_nvfp4_e4m3_codes(const float* x, int64_t n, uint8_t* codes, moe_nvfp4_stream_t stream) {
    if (n < 0) return MOE_NVFP4_ESIZE;
    if (n > 0 && (x == nullptr || codes == nullptr)) return MOE_NVFP4_ENULL;
    if (n > 0 && !aligned(x, 4)) return MOE_NVFP4_EALIGN;
    if (n == 0) return MOE_NVFP4_OK;
    DeviceInfo di;
    int rc;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    launch(e4m3_codes_kernel, di.sms * 8, reinterpret_cast<cudaStream_t>(stream), x, n, codes);
    return cudaGetLastError() == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

int moe_swiglu_nvfp4_quantize_counted(const uint16_t* gu, int64_t rows, int64_t I, float clamp_L,
                                      const int32_t* expert_offsets, int32_t num_experts,
                                      uint8_t* packed, uint8_t* sf, uint64_t* counters,
                                      moe_nvfp4_stream_t stream) {
    if (rows > 0 && counters == nullptr) return MOE_NVFP4_ENULL;
    if (counters != nullptr && !aligned(counters, 8)) return MOE_NVFP4_EALIGN;
    return launch_fused(gu, rows, I, clamp_L, expert_offsets, num_experts, packed, sf, counters,
                        nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int moe_nvfp4_quantize_scaled(const uint16_t* x, int64_t rows, int64_t K, float global_scale,
                              uint8_t* packed, uint8_t* sf, moe_nvfp4_stream_t stream) {
    int rc = check_common(x, rows, K, 2, packed, sf);
    if (rc != MOE_NVFP4_OK) return rc;
    if (!valid_scale(global_scale)) return MOE_NVFP4_ESCALE;
    if (rows == 0) return MOE_NVFP4_OK;
    DeviceInfo di;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    const int64_t nblk = rows * (K / 16);
    launch(nvfp4_quantize_kernel<true>, grid_for(nblk, di.sms, di.occ_quant[1], kUnrollQuant),
           reinterpret_cast<cudaStream_t>(stream), x, nblk, global_scale, packed, sf);
    return cudaGetLastError() == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

int moe_swiglu_nvfp4_quantize_ex(const uint16_t* gu, int64_t rows, int64_t I, float clamp_L,
                                 const int32_t* expert_offsets, int32_t num_experts,
                                 const moe_nvfp4_fused_options* options, uint8_t* packed,
                                 uint8_t* sf, moe_nvfp4_stream_t stream) {
    moe_nvfp4_fused_options opt = {1.0f, 0, nullptr, 0};
    if (options != nullptr) opt = *options;
    return launch_ex(gu, rows, I, clamp_L, expert_offsets, num_experts, opt.global_scale,
                     opt.round_to_bf16 ? kExCompat : kExQuantize, opt.out_offsets, opt.out_rows,
                     packed, sf, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int moe_swiglu_bf16(const uint16_t* gu, int64_t rows, int64_t I, float clamp_L,
                    const int32_t* expert_offsets, int32_t num_experts, uint16_t* out,
                    moe_nvfp4_stream_t stream) {
    return launch_ex(gu, rows, I, clamp_L, expert_offsets, num_experts, 1.0f, kExCompact, nullptr,
                     0, nullptr, nullptr, out, reinterpret_cast<cudaStream_t>(stream));
}

int moe_nvfp4_dequantize(const uint8_t* packed, const uint8_t* sf, int64_t rows, int64_t K,
                         float global_scale, uint16_t* out, moe_nvfp4_stream_t stream) {
    if (rows < 0) return MOE_NVFP4_ESIZE;
    if (K <= 0 || K % 16 != 0) return MOE_NVFP4_EWIDTH;
    if (rows > 0 && K > INT64_MAX / 2 / rows) return MOE_NVFP4_ESIZE;
    if (!valid_scale(global_scale)) return MOE_NVFP4_ESCALE;
    if (rows == 0) return MOE_NVFP4_OK;
    if (packed == nullptr || sf == nullptr || out == nullptr) return MOE_NVFP4_ENULL;
    if (!aligned(packed, 16) || !aligned(sf, 16) || !aligned(out, 32)) return MOE_NVFP4_EALIGN;
    DeviceInfo di;
    int rc = device_info(di);
    if (rc != MOE_NVFP4_OK) return rc;
    const int64_t nblk = rows * (K / 16);
    int64_t grid = (nblk / 4 + kThreads - 1) / kThreads;     // two pairs per thread
    if (grid < 1) grid = 1;
    const int64_t cap = static_cast<int64_t>(di.sms) * di.occ_dequant;
    if (grid > cap) grid = cap;
    // e2m1 * e4m3 magnitudes lie in [2^-10, 2688]: for gs in [2^-90, 2^90]
    // every quotient, residual and RN(1/gs) is a normal fp32 number
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (global_scale == 1.0f)
        launch(nvfp4_dequantize_kernel<kDivNone>, static_cast<int>(grid), st, packed, sf, nblk,
               global_scale, out);
    else if (global_scale >= 0x1p-90f && global_scale <= 0x1p90f)
        launch(nvfp4_dequantize_kernel<kDivMarkstein>, static_cast<int>(grid), st, packed, sf,
               nblk, global_scale, out);
    else
        launch(nvfp4_dequantize_kernel<kDivIeee>, static_cast<int>(grid), st, packed, sf, nblk,
               global_scale, out);
    return cudaGetLastError() == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

double moe_swiglu_nvfp4_window(float clamp_L) { return window_for(clamp_L); }

const char* moe_nvfp4_strerror(int code) {
    switch (code) {
        case MOE_NVFP4_OK: return "ok";
        case MOE_NVFP4_ENULL: return "a required pointer is NULL";
        case MOE_NVFP4_EWIDTH: return "width (K or I) must be a positive multiple of 16";
        case MOE_NVFP4_EALIGN: return "input must be 32-byte aligned, outputs 16-byte aligned";
        case MOE_NVFP4_ESIZE: return "rows < 0 or the tensor size overflows int64";
        case MOE_NVFP4_ECLAMP: return "clamp_L must be finite and in (0, 2^64]";
        case MOE_NVFP4_EOFFSETS: return "num_experts < 0, or expert offsets missing";
        case MOE_NVFP4_ELAUNCH: return "CUDA launch or device query failed";
        case MOE_NVFP4_ESCALE: return "global_scale must be finite and > 0";
        case MOE_NVFP4_EMODE: return "unknown output selector";
        default: return "unknown error code";
    }
}

int moe_nvfp4_abi_version(void) { return 5; }

}  // extern "C"
