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

// e^x for -100 <= x <= 80 as a double-float, by table-driven range
// reduction (P. T. P. Tang, "Table-driven implementation of the exponential
// function in IEEE floating-point arithmetic", ACM TOMS 15(2), 1989):
// x = n ln2/64 + r with |r| <= ln2/128, e^x = 2^(n/64) e^r, the 64 values
// 2^(j/64) from a table of fp32 pairs, e^r by its Taylor series to r^5 (the
// r^3.. terms in fp32, the rest in double-float). The pair arithmetic uses
// the error-free transformations TwoSum (Knuth, TAOCP vol. 2, 4.2.2),
// Fast-TwoSum (Dekker 1971) and the FMA form of TwoProduct (Dekker's exact
// product, with the error term taken by one fma).
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

struct Tally {                  // one thread's counts (far below 2^32: its blocks are at most its CTA's / 32)
    uint32_t blocks = 0, scales = 0, nibbles = 0;
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
// The inputs are read again from memory (keeping the loaded words live
// across the block's arithmetic costs registers on the hot path).
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

// Elements whose value t = v / d (|v| as given, half step h, residual rr =
// |t| - h) could lie across a nibble-changing half-step boundary: |rr| +
// W h > 0.25 (1 - W), with the boundary between half steps k and k+1 among
// kNibbleChangingBoundaries.
__device__ __forceinline__ uint32_t near_boundary_elements(const FusedArgs& A, const float* v, float inv) {
    uint32_t todo = 0;
    for (int i = 0; i < 16; i++) {
        const float av = fabsf(v[i]);
        const float h = fmaf(av, inv, kHalfStepBias) - kHalfStepBias;
        const float rr = fmaf(av, inv, -h);
        if (fmaf(A.W, h, fabsf(rr)) > A.near_thr) {
            const int k = __float2int_rn(2.0f * h) - (rr < 0.0f ? 1 : 0);
            if (k >= 0 && k < 12 && ((kNibbleChangingBoundaries >> k) & 1u)) todo |= 1u << i;
        }
    }
    return todo;
}

// Replaces nibble i (0..15) of the stored block at `packed_blk` (its 8
// packed bytes) with `nib`: clear, then set, by atomics on the 32-bit word
// holding it, so lanes patching other nibbles of the same word concurrently
// do not interfere.
__device__ __forceinline__ void patch_nibble(uint8_t* packed_blk, int i, uint32_t nib) {
    uint32_t* word = reinterpret_cast<uint32_t*>(packed_blk) + (i >> 3);
    const int sh = 4 * (i & 7);
    atomicAnd(word, ~(0xFu << sh));
    atomicOr(word, nib << sh);
}

// Re-decides the elements the lanes of a warp left to the definition, after
// their blocks were stored with the fast nibbles: lane l's `mask` has bit
// 16 k + i for element i of its k-th block of the chunk, whose scale code is
// byte k of `codes`. The elements are evaluated 32 at a time, one per lane,
// whichever lane they belong to (a block near many boundaries, with values
// on ties, costs its warp one pass, not one pass per element);
// eval(owner, k, i, code) returns the nibble and patch(owner, k, i, nib,
// tag) writes it over the stored one (`tag`: the owner's lane value tag0
// for k = 0, tag1 for k = 1, e.g. where its block was stored). Every lane
// of the warp calls this together, after the stores it patches.
template <typename Eval, typename Patch>
__device__ __forceinline__ void resolve_nibbles_warp(int lane, uint32_t mask, uint32_t codes, Eval eval,
                                                     Patch patch, int64_t tag0 = 0, int64_t tag1 = 0) {
    __syncwarp();                                               // the owners' stores before the patches
    const int cnt = __popc(mask);
    int pre = cnt;                                              // inclusive prefix over lanes
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(kFullMask, pre, off);
        if (lane >= off) pre += v;
    }
    const int total = __shfl_sync(kFullMask, pre, 31);
    for (int q0 = 0; q0 < total; q0 += 32) {
        const int q = min(q0 + lane, total - 1);
        int owner = 0;                                          // first lane whose prefix exceeds q
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
            const int p = __shfl_sync(kFullMask, pre, owner + step - 1);
            if (p <= q) owner += step;
        }
        const uint32_t omask = __shfl_sync(kFullMask, mask, owner);
        const int oexcl = __shfl_sync(kFullMask, pre - cnt, owner);
        const uint32_t ocodes = __shfl_sync(kFullMask, codes, owner);
        const int64_t otag0 = __shfl_sync(kFullMask, tag0, owner);
        const int64_t otag1 = __shfl_sync(kFullMask, tag1, owner);
        if (q0 + lane < total) {
            uint32_t m = omask;
            for (int t = q - oexcl; t > 0; t--) m &= m - 1u;    // the (q - oexcl)-th set bit
            const int bit = __ffs(m) - 1;
            const int k = bit >> 4, i = bit & 15;
            patch(owner, k, i, eval(owner, k, i, (ocodes >> (8 * k)) & 0xFFu), k ? otag1 : otag0);
        }
    }
}

// The fused step's fast path for one block of each lane of a warp (blk =
// the lane's block, valid = inside the lane's range): the block is stored
// with its fast nibbles; the elements that lie within the window of a
// nibble-changing boundary are returned (bit i = element i) with the scale
// code, for resolve_nibbles_warp. Every lane calls this together.
template <bool kCount, bool kBf16Clamp>
__device__ __forceinline__ uint32_t fused_block(const FusedArgs& A, int64_t blk, bool valid, const uint32_t* w,
                                                uint32_t& code_out, Tally& tally) {
    const float L = A.L;
    float y[16];
    fast_swiglu16<kBf16Clamp>(A, w, y);

    // scale: safe when both ends of the window round to the same code (the
    // product by RN(1/6) is within an ulp of amax / 6, inside the window)
    const float amax = abs_max16(y);
    const float q = amax * kInv6;
    const uint32_t ends = e4m3x2_rn_sat(q * A.Wp1, q * A.Wm1);
    uint32_t code = ends & 0xFFu;
    if (valid && (ends >> 8) != code) {
        code = scale_by_definition(A.gu + blk * 32, L, A.W, amax, y);
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
    if (valid) {
        *reinterpret_cast<uint2*>(A.packed + blk * 8) = make_uint2(e2m1x8(hs), e2m1x8(hs + 8));
        A.sf[blk] = static_cast<uint8_t>(code);
        if (kCount) tally.blocks++;
    }
    const bool near = valid && closeness > A.near_fast;
    uint32_t todo = 0u;
    if (__any_sync(kFullMask, near) && near) todo = near_boundary_elements(A, y, inv);
    if (kCount) tally.nibbles += __popc(todo);
    code_out = code;
    return todo;
}

// resolve_nibbles_warp for the plain step's chunk of a warp whose block k
// of lane l is base + 32 k + l. Out of line: the hot loop keeps none of
// its registers, and the call runs only when some element of the chunk lies
// within the window of a boundary.
__device__ __noinline__ void resolve_chunk(const uint16_t* gu, uint8_t* packed, float L, int64_t base, int lane,
                                          uint32_t mask, uint32_t codes) {
    resolve_nibbles_warp(
        lane, mask, codes,
        [&](int owner, int k, int i, uint32_t code) {
            float g, u;
            gate_up_at(gu + (base + 32 * k + owner) * 32, i, g, u);
            return nibble_by_definition(swiglu_precise(g, u, L), e4m3_value(code), code);
        },
        [&](int owner, int k, int i, uint32_t nib, int64_t) { patch_nibble(packed + (base + 32 * k + owner) * 8, i, nib); });
}

// The diagnostic variant: the fast fp32 values of one block, in output
// column order.
template <bool kBf16Clamp>
__device__ __forceinline__ void fast_values_block(const FusedArgs& A, int64_t blk, bool valid, const uint32_t* w) {
    float y[16];
    fast_swiglu16<kBf16Clamp>(A, w, y);
    if (valid) {
        float4* out = reinterpret_cast<float4*>(A.values + blk * 16);
#pragma unroll
        for (int k = 0; k < 4; k++) out[k] = make_float4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
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
    // by exact re-evaluations (or slow memory) takes fewer chunks and the
    // CTA's other warps absorb the delay. A chunk is two blocks per lane.
    constexpr int64_t kChunk = 32 * kUnroll;
    const int64_t total = b1 - b0;
    int64_t per_cta = (total + gridDim.x - 1) / gridDim.x;
    per_cta = (per_cta + kChunk - 1) / kChunk * kChunk;
    const int64_t cta_begin = b0 + static_cast<int64_t>(blockIdx.x) * per_cta;
    const int64_t cta_end = cta_begin + per_cta < b1 ? cta_begin + per_cta : b1;
    __shared__ int next_chunk;
    if (threadIdx.x == 0) next_chunk = 0;
    __syncthreads();
    static_assert(kUnroll == 2, "two blocks per lane per chunk");
    auto claim = [&]() {                                    // warp-uniform
        int c = 0;
        if (lane == 0) c = atomicAdd(&next_chunk, 1);
        c = __shfl_sync(kFullMask, c, 0);
        return cta_begin + static_cast<int64_t>(c) * kChunk;
    };
    auto load_block = [&](int64_t blk, uint32_t* w) {
        if (blk < cta_end) {
            const uint16_t* p = A.gu + blk * 32;
            load_stream_32B(p, pol, w);
            load_stream_32B(p + 16, pol, w + 8);
        } else {
#pragma unroll
            for (int j = 0; j < 16; j++) w[j] = 0u;
        }
    };
    Tally tally;
    // Software pipeline over the lane's blocks, one block ahead: while a
    // block is computed, the next one's loads are in flight (the second
    // block of the chunk, then the first block of the next chunk, claimed
    // early), so a warp never computes with none of its own loads pending.
    // Then one warp-wide re-decision of every element of the chunk left to
    // the definition.
    uint32_t w0[16], w1[16];
    int64_t base = claim();
    load_block(base + lane, w0);
    while (base < cta_end) {                                // warp-uniform
        load_block(base + 32 + lane, w1);
        if (kValues) {
            fast_values_block<kBf16Clamp>(A, base + lane, base + lane < cta_end, w0);
            const int64_t next = claim();
            load_block(next + lane, w0);
            fast_values_block<kBf16Clamp>(A, base + 32 + lane, base + 32 + lane < cta_end, w1);
            base = next;
            continue;
        }
        uint32_t code0, code1;
        const uint32_t m0 =
            fused_block<kCount, kBf16Clamp>(A, base + lane, base + lane < cta_end, w0, code0, tally);
        const int64_t next = claim();
        load_block(next + lane, w0);
        const uint32_t m1 =
            fused_block<kCount, kBf16Clamp>(A, base + 32 + lane, base + 32 + lane < cta_end, w1, code1, tally);
        const uint32_t mask = m0 | (m1 << 16);
        if (__any_sync(kFullMask, mask != 0u))
            resolve_chunk(A.gu, A.packed, A.L, base, lane, mask, code0 | (code1 << 8));
        base = next;
    }
    if (kCount) {
        atomicAdd(A.counters + 0, static_cast<unsigned long long>(tally.blocks));
        if (tally.scales) atomicAdd(A.counters + 1, static_cast<unsigned long long>(tally.scales));
        if (tally.nibbles) atomicAdd(A.counters + 2, static_cast<unsigned long long>(tally.nibbles));
    }
}

// Small problems, where every block fits in one wave of resident threads at
// one block per thread: thread t of the grid takes block first + t, so every
// warp has work, every lane's loads are in flight before any arithmetic, and
// there is no chunk loop (the persistent shape above would give a few CTAs
// several chunks each and leave most warps idle). CTAs of whole warps;
// blockDim.x is chosen on the host.
template <bool kBf16Clamp>
__global__ void __launch_bounds__(kThreads)
swiglu_nvfp4_small_kernel(const FusedArgs A) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    int64_t b0, b1;
    active_block_range(A.offsets, A.E, A.rows, A.bpr, b0, b1);
    const int64_t blk = b0 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool valid = blk < b1;
    if (__all_sync(kFullMask, !valid)) return;             // warp-uniform
    uint32_t w[16];
    if (valid) {
        const uint64_t pol = l2_evict_first_policy();
        const uint16_t* p = A.gu + blk * 32;
        load_stream_32B(p, pol, w);
        load_stream_32B(p + 16, pol, w + 8);
    } else {
#pragma unroll
        for (int j = 0; j < 16; j++) w[j] = 0u;
    }
    Tally tally;
    uint32_t code;
    const uint32_t todo = fused_block<false, kBf16Clamp>(A, blk, valid, w, code, tally);
    if (__any_sync(kFullMask, todo != 0u))
        resolve_chunk(A.gu, A.packed, A.L, blk - (threadIdx.x & 31), threadIdx.x & 31, todo, code);
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

// Results near and inside the fp32 subnormal range need no test of their
// own: for gates at or above the window's floor the fast value's error is
// the silu's relative error (measured over every BF16 gate, subnormal gates
// included) plus half an ulp for the product, which rounds as IEEE does
// when it underflows; below 2^-126 that is at most (k + 1) / 2 + 1 ulps of
// 2^-149 for a relative bound of k units of 2^-24, inside the tolerance.
// A BF16 rounding midpoint is still the fp32 value whose low half is
// 0x8000, so the midpoint test decides them as it decides normal values.
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
    // A value is near a midpoint when ((bits + tol - 0x8000) mod 2^16) <= 2
    // tol. Block test first, two values per word: the low halves of a pair
    // side by side, tol + 0x8000 added to both halves by one 32-bit add (a
    // carry out of the low half raises the high half by one, so both are
    // held to 2 tol + 1: false alarms only), and the least half over the
    // block by min.u16x2. Element by element only when it fires.
    const uint32_t both = (tol + 0x8000u) * 0x10001u;
    uint32_t least = 0xFFFFFFFFu;
#pragma unroll
    for (int q = 0; q < 8; q++) {
        yb[q] = bf16x2_rn(y[2 * q + 1], y[2 * q]);
        least = u16x2_min(least, __byte_perm(__float_as_uint(y[2 * q]), __float_as_uint(y[2 * q + 1]), 0x5410) + both);
    }
    uint32_t amb = 0;
    if ((least & 0xFFFFu) <= 2u * tol + 1u || (least >> 16) <= 2u * tol + 1u) {
        // the test in the top half of the word: one multiply-add and a compare
        const uint32_t c16 = (tol - 0x8000u) << 16, t16 = ((2u * tol) << 16) | 0xFFFFu;
#pragma unroll
        for (int q = 0; q < 8; q++)
            amb |= (near_bf16_midpoint(y[2 * q], c16, t16) << (2 * q)) |
                   (near_bf16_midpoint(y[2 * q + 1], c16, t16) << (2 * q + 1));
    }
    // block pre-test for the window's range (gates below the floor);
    // element by element only when it fires
    if (gmin < X.gate_floor) {
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

// The two-level step's fast path for one block of each lane of a warp (as
// fused_block, on v = RN(y gs) with the window widened by the product's
// roundings): lo / hi / code get the fast nibbles and scale (the scale
// decided by the definition where the window leaves it open); the elements
// within the window of a nibble-changing boundary are returned for
// resolve_chunk_scaled. Every lane calls this together.
template <bool kBf16Clamp>
__device__ __forceinline__ uint32_t scaled_fast_block(const ExArgs& X, int64_t blk, bool valid, const uint32_t* w,
                                                      uint32_t& lo, uint32_t& hi, uint32_t& code_out) {
    const FusedArgs& A = X.f;
    const float gs = X.gs;
    float y[16];
    fast_swiglu16<kBf16Clamp>(A, w, y);
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
    uint32_t code = ends & 0xFFu;
    if (valid && (ends >> 8) != code) {
        const float lim = amax * (1.0f - 2.0f * A.W);
        float am = 0.0f;
        for (int i = 0; i < 16; i++) {
            if (fabsf(v[i]) >= lim) {
                float g, u;
                gate_up_at(A.gu + blk * 32, i, g, u);
                am = fmaxf(am, fabsf(__fmul_rn(swiglu_precise(g, u, A.L), gs)));
            }
        }
        code = e4m3x2_rn_sat(0.0f, __fdiv_rn(am, 6.0f)) & 0xFFu;
    }
    const float d = e4m3_value(code);
    const float inv = (code == 0u) ? 0.0f : rcp_approx(d);
    float hs[16];
    const float closeness = half_steps16(v, inv, hs);
    lo = e2m1x8(hs);
    hi = e2m1x8(hs + 8);
    const bool near = valid && closeness > A.near_fast;
    uint32_t todo = 0u;
    if (__any_sync(kFullMask, near) && near) todo = near_boundary_elements(A, v, inv);
    code_out = code;
    return todo;
}

// resolve_nibbles_warp for the two-level step's chunk of a warp (block k of
// lane l at base + 32 k + l, stored at output block oblk0 / oblk1 for k = 0
// / 1): each element by RN(definition * gs) under its block's scale. Out of
// line, as resolve_chunk.
__device__ __noinline__ void resolve_chunk_scaled(const uint16_t* gu, uint8_t* packed, float L, float gs,
                                                  int64_t base, int lane, uint32_t mask, uint32_t codes,
                                                  int64_t oblk0, int64_t oblk1) {
    resolve_nibbles_warp(
        lane, mask, codes,
        [&](int owner, int k, int i, uint32_t code) {
            float g, u;
            gate_up_at(gu + (base + 32 * k + owner) * 32, i, g, u);
            return nibble_by_definition(__fmul_rn(swiglu_precise(g, u, L), gs), e4m3_value(code), code);
        },
        [&](int, int, int i, uint32_t nib, int64_t oblk) { patch_nibble(packed + oblk * 8, i, nib); }, oblk0, oblk1);
}

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
    // the compat modes without padded output: each warp's queue of blocks
    // with an element to re-evaluate (at most 31 left plus 32 kUnroll from
    // one chunk), as offsets from cta_begin (the launcher admits fewer than
    // 2^32 blocks in all). The compact writer resolves in place: it streams
    // near the copy floor, where the passes over a queue lengthen the launch
    // more than the queue saves on data with few undecided elements.
    constexpr bool kDefer = (kMode == kExCompat || kMode == kExCompatUnit) && !kPadded;
    constexpr int kQueue = 31 + 32 * kUnroll;
    __shared__ uint32_t defer_q[kDefer ? kThreads / 32 : 1][kDefer ? kQueue : 1];
    int deferred = 0;                                        // warp-uniform
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
    // the end of a BF16-mode block: the compact writer stores its BF16
    // values; the compat mode quantizes them (and stores where out_block says)
    auto finish_block = [&](int64_t blk, bool valid, const uint32_t* b) {
        if (kMode == kExCompact) {
            if (valid) {
                uint4* dst = reinterpret_cast<uint4*>(X.out_bf16 + blk * 16);
                dst[0] = make_uint4(b[0], b[1], b[2], b[3]);
                dst[1] = make_uint4(b[4], b[5], b[6], b[7]);
            }
            return;
        }
        float v[16];
        uint32_t lo, hi, code;
        if (kMode == kExCompatUnit) {                       // BF16 values: the cheap exact form
#pragma unroll
            for (int q = 0; q < 8; q++) {
                v[2 * q] = bf16_lo(b[q]);
                v[2 * q + 1] = bf16_hi(b[q]);
            }
            code = quantize16_exact<false, true>(v, lo, hi);
        } else {
#pragma unroll
            for (int q = 0; q < 8; q++) {
                const float2 vv = __fmul2_rn(make_float2(bf16_lo(b[q]), bf16_hi(b[q])), make_float2(X.gs, X.gs));
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
    };
    // one pass over up to 32 queued blocks, one per lane (have: this lane
    // has one, block blk; a warp-uniform call): reloaded (still in L2),
    // recomputed, the undecided elements re-evaluated by the definition,
    // then finished
    auto finish_pass = [&](bool have, int64_t blk) {
        uint32_t w1[16];
        if (have) {
            load_nc_32B(A.gu + blk * 32, w1);
            load_nc_32B(A.gu + blk * 32 + 16, w1 + 8);
        } else {
#pragma unroll
            for (int j = 0; j < 16; j++) w1[j] = 0u;
        }
        float y[16];
        fast_swiglu16<kBf16Clamp>(A, w1, y);
        uint32_t b[8];
        const uint32_t m = bf16_fast_of_block(X, have, w1, y, b);
        resolve_bf16_elements<16>(A, blk, m, b);
        if (have) finish_block(blk, true, b);
    };
    // the warp's n queued blocks (n warp-uniform), 32 per pass
    auto finish_deferred = [&](int n) {
        __syncwarp();
        const uint32_t* q = defer_q[threadIdx.x >> 5];
        for (int p0 = 0; p0 < n; p0 += 32)
            finish_pass(p0 + lane < n, p0 + lane < n ? cta_begin + q[p0 + lane] : 0);
        __syncwarp();
    };
    auto claim = [&]() {                                    // warp-uniform
        int c = 0;
        if (lane == 0) c = atomicAdd(&next_chunk, 1);
        c = __shfl_sync(kFullMask, c, 0);
        return cta_begin + static_cast<int64_t>(c) * kChunk;
    };
    auto load_block = [&](int64_t blk, uint32_t* w) {
        if (blk < cta_end) {
            const uint16_t* p = A.gu + blk * 32;
            if (kMode == kExCompact) {
                // the compact writer (2 output bytes per 4 input bytes)
                // streams 8 % faster with plain loads; the quantizing
                // modes are faster with the evict-first hint
                load_nc_32B(p, w);
                load_nc_32B(p + 16, w + 8);
            } else {
                load_stream_32B(p, pol, w);
                load_stream_32B(p + 16, pol, w + 8);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; j++) w[j] = 0u;
        }
    };
    // Without padded output, the two-level and compat modes load one block
    // ahead: the next chunk's first block is claimed and its loads issued
    // after the first block's fast path (two-level) or after the fast passes
    // (compat), so they are in flight while the chunk is finished (the
    // padded and compact-writer modes measured slower that way; with an
    // fp32 clamp the extra registers spill).
    constexpr bool kPipe = (kDefer || (kMode == kExQuantize && !kPadded)) && kBf16Clamp;
    static_assert(kUnroll == 2, "two blocks per lane per chunk");
    uint32_t w0[16], w1[16];
    int64_t base = 0;
    if (kPipe) {
        base = claim();
        load_block(base + lane, w0);
    }
    for (;;) {                                              // warp-uniform
        if (!kPipe) {
            base = claim();
            if (base >= cta_end) break;
            load_block(base + lane, w0);
        } else if (base >= cta_end) {
            break;
        }
        load_block(base + 32 + lane, w1);
        int64_t next = 0;
        if (kMode == kExQuantize && kPadded) {
            // padded output: each block decided on its own (the warp-wide
            // re-decision below measured slower with the segment lookups)
#pragma unroll
            for (int k = 0; k < kUnroll; k++) {
                const int64_t blk = base + 32 * k + lane;
                const bool valid = blk < cta_end;
                float y[16];
                fast_swiglu16<kBf16Clamp>(A, k ? w1 : w0, y);
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
        } else if (kMode == kExQuantize) {
            // fast nibbles stored, then one warp-wide re-decision of the
            // chunk's elements left to the definition
            auto two_level_block = [&](int64_t blk, const uint32_t* w, uint32_t& todo, uint32_t& code,
                                       int64_t& oblk) {
                const bool valid = blk < cta_end;
                uint32_t lo, hi;
                todo = scaled_fast_block<kBf16Clamp>(X, blk, valid, w, lo, hi, code);
                bool store;
                out_block(blk, valid, oblk, store);
                if (store) {
                    *reinterpret_cast<uint2*>(A.packed + oblk * 8) = make_uint2(lo, hi);
                    A.sf[oblk] = static_cast<uint8_t>(code);
                } else {
                    todo = 0u;
                }
            };
            uint32_t t0, t1, c0, c1;
            int64_t o0, o1;
            two_level_block(base + lane, w0, t0, c0, o0);
            if (kPipe) {
                next = claim();
                load_block(next + lane, w0);
            }
            two_level_block(base + 32 + lane, w1, t1, c1, o1);
            const uint32_t mask = t0 | (t1 << 16);
            if (__any_sync(kFullMask, mask != 0u))
                resolve_chunk_scaled(A.gu, A.packed, A.L, X.gs, base, lane, mask, c0 | (c1 << 8), o0, o1);
        } else {
            // BF16 values: fast pass over all blocks; blocks with an element
            // whose BF16 rounding the fast value cannot decide are finished
            // later (below), then store or quantize
            uint32_t yb[8 * kUnroll];
            uint32_t elems = 0;
#pragma unroll
            for (int k = 0; k < kUnroll; k++) {
                float y[16];
                fast_swiglu16<kBf16Clamp>(A, k ? w1 : w0, y);
                elems |= bf16_fast_of_block(X, base + 32 * k + lane < cta_end, k ? w1 : w0, y,
                                                       yb + 8 * k)
                         << (16 * k);
            }
            if (kPipe) {
                next = claim();
                load_block(next + lane, w0);
            }
            if constexpr (!kDefer) {
                // resolved here: padded output keeps each thread's blocks in
                // order (its segment cache moves forward only); the compact
                // writer is faster this way on typical data
                resolve_bf16_elements<16 * kUnroll>(A, base + lane, elems, yb);
            } else if (__any_sync(kFullMask, elems != 0u)) {
                // rare (about one block in 130): queued for the warp, which
                // finishes them 32 at a time, one block per lane, instead of
                // one element per pass while the other lanes wait
                uint32_t* q = defer_q[threadIdx.x >> 5];
                const unsigned below = (1u << lane) - 1u;
#pragma unroll
                for (int k = 0; k < kUnroll; k++) {
                    const bool f = ((elems >> (16 * k)) & 0xFFFFu) != 0u;
                    const unsigned bal = __ballot_sync(kFullMask, f);
                    if (f) q[deferred + __popc(bal & below)] = static_cast<uint32_t>(base + 32 * k + lane - cta_begin);
                    deferred += __popc(bal);
                }
                if (deferred >= 32) {
                    finish_deferred(deferred);
                    deferred = 0;
                }
            }
#pragma unroll
            for (int k = 0; k < kUnroll; k++) {
                const int64_t blk = base + 32 * k + lane;
                if (kDefer && ((elems >> (16 * k)) & 0xFFFFu) != 0u) continue;       // queued
                finish_block(blk, blk < cta_end, yb + 8 * k);
            }
        }
        if (kPipe) base = next;
    }
    if constexpr (kDefer) {
        // the CTA's leftover queues (each under 32 blocks), concatenated in
        // warp order: warp w finishes entries [32 w, 32 w + 32), so the CTA
        // runs as many passes as its leftovers need instead of one per warp
        __shared__ int defer_n[kThreads / 32];
        const int warp = threadIdx.x >> 5;
        if (lane == 0) defer_n[warp] = deferred;
        __syncthreads();
        const int i = 32 * warp + lane;
        int total = 0, owner = -1, pos = 0;
#pragma unroll
        for (int v = 0; v < kThreads / 32; v++) {
            const int c = defer_n[v];
            if (i >= total && i < total + c) {
                owner = v;
                pos = i - total;
            }
            total += c;
        }
        if (32 * warp < total)                                 // warp-uniform
            finish_pass(owner >= 0, owner >= 0 ? cta_begin + defer_q[owner][pos] : 0);
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
    // kUnrollQuant blocks per lane per pass, each slot reloaded with the
    // same block of the next pass as soon as its words are unpacked, so a
    // lane keeps loads in flight while it quantizes
    uint32_t w[kUnrollQuant][8];
    int64_t base = warp * 32 * kUnrollQuant;
#pragma unroll
    for (int k = 0; k < kUnrollQuant; k++) {
        const int64_t blk = base + 32 * k + lane;
        if (blk < nblk) load_stream_32B(x + blk * 16, pol, w[k]);
    }
    for (; base < nblk; base += step) {
#pragma unroll
        for (int k = 0; k < kUnrollQuant; k++) {
            const int64_t blk = base + 32 * k + lane;
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; i++) {
                v[i] = (i & 1) ? bf16_hi(w[k][i >> 1]) : bf16_lo(w[k][i >> 1]);
                if (kScaled) v[i] = __fmul_rn(v[i], gs);          // two-level: v = fl(x * gs)
            }
            if (blk + step < nblk) load_stream_32B(x + (blk + step) * 16, pol, w[k]);
            if (blk >= nblk) continue;
            uint32_t lo, hi;
            // packed quotient steps (the register budget of 3 CTAs per SM
            // holds them and the 4 blocks in flight without spilling)
            const uint32_t code = quantize16_exact<kScaled, true>(v, lo, hi);
            *reinterpret_cast<uint2*>(packed + blk * 8) = make_uint2(lo, hi);
            sf[blk] = static_cast<uint8_t>(code);
        }
    }
}

// Quantize-only for small problems: one block per thread (as
// swiglu_nvfp4_small_kernel), the load issued first.
template <bool kScaled>
__global__ void __launch_bounds__(kThreads)
nvfp4_quantize_small_kernel(const uint16_t* __restrict__ x, int64_t nblk, float gs,
                            uint8_t* __restrict__ packed, uint8_t* __restrict__ sf) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (blk >= nblk) return;
    uint32_t w[8];
    load_stream_32B(x + blk * 16, l2_evict_first_policy(), w);
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
        v[i] = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
        if (kScaled) v[i] = __fmul_rn(v[i], gs);
    }
    uint32_t lo, hi;
    const uint32_t code = quantize16_exact<kScaled, true>(v, lo, hi);
    *reinterpret_cast<uint2*>(packed + blk * 8) = make_uint2(lo, hi);
    sf[blk] = static_cast<uint8_t>(code);
}

// ---------------------------------------------------------------------------
// Dequantization: NVFP4 -> BF16, value = e2m1 * e4m3 / gs
// ---------------------------------------------------------------------------

enum DequantDivision { kDivNone = 0, kDivMarkstein = 1, kDivIeee = 2 };

// One 16-element block: 8 packed bytes (p), scale value d -> 16 BF16 values,
// stored with the L2 policy pol.
template <int kDiv>
__device__ __forceinline__ void dequantize_block(uint2 p, float d, float gs, float inv_gs,
                                                 uint16_t* dst16, uint64_t pol) {
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
    store_32B_hint(dst16, o, pol);
}

// Lanes take consecutive pairs of blocks, so every load and store of a warp
// covers whole 32-byte sectors: 16 packed bytes and 2 scale bytes in, two
// 32-byte stores out. Two pairs per lane per iteration; an odd last block is
// done at the end.
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
    // The output (4 bytes per element against 0.5625 read) is stored
    // evict-first: it is larger than L2 at the sizes that matter, and
    // keeping it there measured 3.6 % slower. The next iteration's loads
    // are issued before this one's conversion.
    constexpr int kPairs = 2;
    uint32_t w[kPairs][4], s2[kPairs];
    auto load_pairs = [&](int64_t p0) {
#pragma unroll
        for (int k = 0; k < kPairs; k++) {
            const int64_t pi = p0 + k * stride;
            if (pi < npair) {
                load_stream_16B(packed + pi * 16, pol, w[k]);
                s2[k] = __ldg(reinterpret_cast<const uint16_t*>(sf + 2 * pi));
            }
        }
    };
    load_pairs(tid);
    for (int64_t p0 = tid; p0 < npair; p0 += kPairs * stride) {
        uint32_t cw[kPairs][4], cs[kPairs];
#pragma unroll
        for (int k = 0; k < kPairs; k++) {
            cs[k] = s2[k];
#pragma unroll
            for (int t = 0; t < 4; t++) cw[k][t] = w[k][t];
        }
        load_pairs(p0 + kPairs * stride);
#pragma unroll
        for (int k = 0; k < kPairs; k++) {
            const int64_t pi = p0 + k * stride;
            if (pi < npair) {
                dequantize_block<kDiv>(make_uint2(cw[k][0], cw[k][1]), e4m3_value(cs[k] & 0xFFu), gs,
                                       inv_gs, out + pi * 32, pol);
                dequantize_block<kDiv>(make_uint2(cw[k][2], cw[k][3]), e4m3_value(cs[k] >> 8), gs,
                                       inv_gs, out + pi * 32 + 16, pol);
            }
        }
    }
    if ((nblk & 1) && tid == 0) {
        const int64_t blk = nblk - 1;
        dequantize_block<kDiv>(*reinterpret_cast<const uint2*>(packed + blk * 8), e4m3_value(sf[blk]),
                               gs, inv_gs, out + blk * 16, pol);
    }
}

// ---------------------------------------------------------------------------
// Diagnostics: the memory system's limit for this step's traffic, and the
// preconditions on expert offsets
// ---------------------------------------------------------------------------

template <int n>
__device__ __forceinline__ uint32_t xor_fold(const uint32_t* w) {
    uint32_t r = w[0];
#pragma unroll
    for (int i = 1; i < n; i++) r ^= w[i];
    return r;
}

// The loads and stores of one block with none of the arithmetic: the folded
// input words stand in for the 8 packed bytes and the scale byte, so no
// load is dead.
template <int kInWords>
__device__ __forceinline__ void floor_store(const uint32_t* w, int64_t blk, uint8_t* packed, uint8_t* sf) {
    const uint32_t a = xor_fold<kInWords / 2>(w), b = xor_fold<kInWords / 2>(w + kInWords / 2);
    *reinterpret_cast<uint2*>(packed + blk * 8) = make_uint2(a, b);
    sf[blk] = static_cast<uint8_t>(a ^ b);
}

template <int kInWords>
__device__ __forceinline__ void floor_load(const uint32_t* in, int64_t blk, uint64_t pol, uint32_t* w) {
    load_stream_32B(in + blk * kInWords, pol, w);
    if (kInWords == 16) load_stream_32B(in + blk * kInWords + 8, pol, w + 8);
}

// The fused step's traffic (64 input bytes per block) in its persistent
// shape: CTA ranges, 64-block chunks claimed from a shared counter, two
// blocks per lane, loaded one block ahead as the step does.
__global__ void __launch_bounds__(kThreads, kMinBlocksFused)
fused_traffic_kernel(const uint32_t* in, int64_t nblk, uint8_t* packed, uint8_t* sf) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const uint64_t pol = l2_evict_first_policy();
    const int lane = threadIdx.x & 31;
    constexpr int64_t kChunk = 32 * kUnroll;
    int64_t per_cta = (nblk + gridDim.x - 1) / gridDim.x;
    per_cta = (per_cta + kChunk - 1) / kChunk * kChunk;
    const int64_t cta_begin = static_cast<int64_t>(blockIdx.x) * per_cta;
    const int64_t cta_end = cta_begin + per_cta < nblk ? cta_begin + per_cta : nblk;
    __shared__ int next_chunk;
    if (threadIdx.x == 0) next_chunk = 0;
    __syncthreads();
    auto claim = [&]() {                                    // warp-uniform
        int c = 0;
        if (lane == 0) c = atomicAdd(&next_chunk, 1);
        c = __shfl_sync(kFullMask, c, 0);
        return cta_begin + static_cast<int64_t>(c) * kChunk;
    };
    static_assert(kUnroll == 2, "two blocks per lane per chunk");
    uint32_t w0[16], w1[16];
    int64_t base = claim();
    if (base + lane < cta_end) floor_load<16>(in, base + lane, pol, w0);
    while (base < cta_end) {                                // warp-uniform
        if (base + 32 + lane < cta_end) floor_load<16>(in, base + 32 + lane, pol, w1);
        if (base + lane < cta_end) floor_store<16>(w0, base + lane, packed, sf);
        const int64_t next = claim();
        if (next + lane < cta_end) floor_load<16>(in, next + lane, pol, w0);
        if (base + 32 + lane < cta_end) floor_store<16>(w1, base + 32 + lane, packed, sf);
        base = next;
    }
}

// The quantize-only step's traffic (32 input bytes per block) in its
// persistent shape: grid-stride, four block slots per lane, each reloaded
// for the next pass as soon as it is read, as the step does.
__global__ void __launch_bounds__(kThreads, kMinBlocksQuant)
quantize_traffic_kernel(const uint32_t* in, int64_t nblk, uint8_t* packed, uint8_t* sf) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const uint64_t pol = l2_evict_first_policy();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t step = (static_cast<int64_t>(gridDim.x) * kThreads >> 5) * 32 * kUnrollQuant;
    uint32_t w[kUnrollQuant][8];
    int64_t base = warp * 32 * kUnrollQuant;
#pragma unroll
    for (int k = 0; k < kUnrollQuant; k++)
        if (base + 32 * k + lane < nblk) floor_load<8>(in, base + 32 * k + lane, pol, w[k]);
    for (; base < nblk; base += step) {
#pragma unroll
        for (int k = 0; k < kUnrollQuant; k++) {
            const int64_t blk = base + 32 * k + lane;
            const uint32_t fold[2] = {xor_fold<4>(w[k]), xor_fold<4>(w[k] + 4)};
            if (blk + step < nblk) floor_load<8>(in, blk + step, pol, w[k]);
            if (blk < nblk) floor_store<2>(fold, blk, packed, sf);
        }
    }
}

// Either step's traffic in the small-problem shape: one block per thread.
template <int kInWords>
__global__ void __launch_bounds__(kThreads)
traffic_small_kernel(const uint32_t* in, int64_t nblk, uint8_t* packed, uint8_t* sf) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (blk >= nblk) return;
    uint32_t w[kInWords];
    floor_load<kInWords>(in, blk, l2_evict_first_policy(), w);
    floor_store<kInWords>(w, blk, packed, sf);
}

// A launch and nothing else.
__global__ void empty_kernel() {
    wait_for_preceding_grid();
    allow_next_grid_launch();
}

// Reads n32 32-byte pieces with the default L2 policy (four in flight per
// thread) and XORs them into *sink, one atomic per CTA: a read-only sweep
// that replaces the L2's contents with clean lines.
__global__ void __launch_bounds__(kThreads)
read_sweep_kernel(const uint32_t* in, int64_t n32, uint32_t* sink) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    uint32_t acc = 0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n32; i += 4 * stride) {
        uint32_t w[4][8];
#pragma unroll
        for (int k = 0; k < 4; k++)
            if (i + k * stride < n32) load_nc_32B(in + (i + k * stride) * 8, w[k]);
#pragma unroll
        for (int k = 0; k < 4; k++)
            if (i + k * stride < n32) acc ^= xor_fold<8>(w[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(kFullMask, acc, o);
    __shared__ uint32_t warp_acc[kThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_acc[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t a = 0;
        for (int k = 0; k < kThreads / 32; k++) a ^= warp_acc[k];
        atomicXor(sink, a);
    }
}

// Preconditions of the expert offsets, checked on the device (the offsets
// live there): bit MOE_NVFP4_CHECK_DECREASING when offsets[e+1] <
// offsets[e], MOE_NVFP4_CHECK_OUTSIDE when an offset lies outside [0, rows],
// and with padded output MOE_NVFP4_CHECK_OVERLAP when the destination rows
// of two segments (each clipped to [0, out_rows)) intersect. Bits are OR-ed
// into *status; nothing traps. Grid: x over offsets (and segments i), y over
// tiles of segments j compared with i (only tiles at or past i's tile).
constexpr int kCheckTile = 256;

__device__ __forceinline__ void dest_range(const int32_t* offsets, const int32_t* out_offsets, int64_t out_rows,
                                           int64_t e, int64_t& lo, int64_t& hi) {
    const int64_t n = static_cast<int64_t>(__ldg(offsets + e + 1)) - __ldg(offsets + e);
    lo = __ldg(out_offsets + e);
    hi = lo + (n > 0 ? n : 0);
    lo = lo < 0 ? 0 : lo;
    hi = hi > out_rows ? out_rows : hi;
}

__global__ void __launch_bounds__(kCheckTile)
check_offsets_kernel(const int32_t* offsets, int E, int64_t rows, const int32_t* out_offsets,
                     int64_t out_rows, int32_t* status) {
    wait_for_preceding_grid();
    allow_next_grid_launch();
    int bits = 0;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kCheckTile + threadIdx.x;
    if (blockIdx.y == 0 && i <= E) {
        const int64_t o = __ldg(offsets + i);
        if (o < 0 || o > rows) bits |= MOE_NVFP4_CHECK_OUTSIDE;
        if (i < E && __ldg(offsets + i + 1) < o) bits |= MOE_NVFP4_CHECK_DECREASING;
    }
    if (out_offsets != nullptr && blockIdx.y >= blockIdx.x) {
        __shared__ int64_t lo_s[kCheckTile], hi_s[kCheckTile];
        const int64_t j = static_cast<int64_t>(blockIdx.y) * kCheckTile + threadIdx.x;
        int64_t lo = 0, hi = 0;
        if (j < E) dest_range(offsets, out_offsets, out_rows, j, lo, hi);
        lo_s[threadIdx.x] = lo;
        hi_s[threadIdx.x] = hi;
        __syncthreads();
        if (i < E) {
            int64_t ilo, ihi;
            dest_range(offsets, out_offsets, out_rows, i, ilo, ihi);
            if (ilo < ihi) {
                for (int t = 0; t < kCheckTile; t++) {
                    const int64_t jj = static_cast<int64_t>(blockIdx.y) * kCheckTile + t;
                    if (jj > i && jj < E && lo_s[t] < hi_s[t] &&
                        (ilo > lo_s[t] ? ilo : lo_s[t]) < (ihi < hi_s[t] ? ihi : hi_s[t])) {
                        bits |= MOE_NVFP4_CHECK_OVERLAP;
                        break;
                    }
                }
            }
        }
    }
    if (bits != 0) atomicOr(status, bits);
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
    int occ_traffic[2] = {0, 0};                // [fused, quantize] traffic-floor kernels
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
                &di.occ_dequant, nvfp4_dequantize_kernel<kDivMarkstein>, kThreads, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_traffic[0], fused_traffic_kernel, kThreads, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_traffic[1], quantize_traffic_kernel, kThreads, 0) != cudaSuccess)
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

// Small-problem shape: when every block fits in one wave of the resident
// threads at one block per thread, one block per thread in CTAs of
// kSmallThreads (small CTAs spread the few blocks over every SM).
constexpr int kSmallThreads = 128;

bool small_problem(int64_t nblk, int sms, int occ) {
    return nblk <= static_cast<int64_t>(sms) * (occ > 0 ? occ : 1) * kThreads;
}

int small_grid(int64_t nblk) {
    const int64_t g = (nblk + kSmallThreads - 1) / kSmallThreads;
    return static_cast<int>(g < 1 ? 1 : g);
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
cudaError_t launch_shaped(void (*kernel)(KArgs...), dim3 grid, int threads, cudaStream_t stream,
                          Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), int grid, cudaStream_t stream, Args&&... args) {
    return launch_shaped(kernel, dim3(static_cast<unsigned>(grid)), kThreads, stream,
                         std::forward<Args>(args)...);
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH; }

template <bool kBf16Clamp>
cudaError_t launch_fused_kernel(const FusedArgs& A, int64_t nblk, const DeviceInfo& di, bool counted,
                                bool values, cudaStream_t stream) {
    const int* occ = di.occ[kBf16Clamp ? 1 : 0];
    if (values)
        return launch(swiglu_nvfp4_kernel<false, true, kBf16Clamp>, grid_for(nblk, di.sms, occ[2]), stream, A);
    if (counted)
        return launch(swiglu_nvfp4_kernel<true, false, kBf16Clamp>, grid_for(nblk, di.sms, occ[1]), stream, A);
    if (small_problem(nblk, di.sms, occ[0]))
        return launch_shaped(swiglu_nvfp4_small_kernel<kBf16Clamp>, dim3(small_grid(nblk)), kSmallThreads,
                             stream, A);
    return launch(swiglu_nvfp4_kernel<false, false, kBf16Clamp>, grid_for(nblk, di.sms, occ[0]), stream, A);
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
cudaError_t launch_ex_kernel(const ExArgs& X, int mode, int64_t nblk, const DeviceInfo& di,
                             cudaStream_t stream) {
    const int* occ = di.occ_ex[kBf16Clamp ? 1 : 0];
    const bool padded = X.out_offsets != nullptr && X.f.offsets != nullptr;
    if (mode == kExQuantize && padded)
        return launch(swiglu_ex_kernel<kExQuantize, kBf16Clamp, true>, grid_for(nblk, di.sms, occ[4]), stream, X);
    if (mode == kExQuantize)
        return launch(swiglu_ex_kernel<kExQuantize, kBf16Clamp, false>, grid_for(nblk, di.sms, occ[0]), stream, X);
    if (mode == kExCompat && X.gs == 1.0f && padded)
        return launch(swiglu_ex_kernel<kExCompatUnit, kBf16Clamp, true>, grid_for(nblk, di.sms, occ[6]), stream, X);
    if (mode == kExCompat && X.gs == 1.0f)
        return launch(swiglu_ex_kernel<kExCompatUnit, kBf16Clamp, false>, grid_for(nblk, di.sms, occ[3]), stream, X);
    if (mode == kExCompat && padded)
        return launch(swiglu_ex_kernel<kExCompat, kBf16Clamp, true>, grid_for(nblk, di.sms, occ[5]), stream, X);
    if (mode == kExCompat)
        return launch(swiglu_ex_kernel<kExCompat, kBf16Clamp, false>, grid_for(nblk, di.sms, occ[1]), stream, X);
    return launch(swiglu_ex_kernel<kExCompact, kBf16Clamp, false>, grid_for(nblk, di.sms, occ[2]), stream, X);
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
    // the compat modes queue blocks by a 32-bit offset inside a CTA's range
    // (2^32 blocks are 256 GiB of input, beyond one device with its outputs)
    if (rows * (I / 16) >= (int64_t(1) << 32)) return MOE_NVFP4_ESIZE;
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
    return launch_status(bf16_bits_of(L) >= 0 ? launch_ex_kernel<true>(X, mode, nblk, di, stream)
                                              : launch_ex_kernel<false>(X, mode, nblk, di, stream));
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
    return launch_status(
        lb >= 0 ? launch_fused_kernel<true>(A, nblk, di, counters != nullptr, values != nullptr, stream)
                : launch_fused_kernel<false>(A, nblk, di, counters != nullptr, values != nullptr, stream));
}

// The quantize-only kernels in the shape for nblk blocks.
template <bool kScaled>
cudaError_t launch_quantize(const uint16_t* x, int64_t nblk, float gs, uint8_t* packed, uint8_t* sf,
                            const DeviceInfo& di, cudaStream_t stream) {
    const int occ = di.occ_quant[kScaled ? 1 : 0];
    if (small_problem(nblk, di.sms, occ))
        return launch_shaped(nvfp4_quantize_small_kernel<kScaled>, dim3(small_grid(nblk)), kSmallThreads,
                             stream, x, nblk, gs, packed, sf);
    return launch(nvfp4_quantize_kernel<kScaled>, grid_for(nblk, di.sms, occ, kUnrollQuant), stream, x, nblk,
                  gs, packed, sf);
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
    return launch_status(launch_quantize<false>(x, nblk, 1.0f, packed, sf, di,
                                                reinterpret_cast<cudaStream_t>(stream)));
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
    return launch_status(launch(swiglu_precise_values_kernel, di.sms * 8, reinterpret_cast<cudaStream_t>(stream),
                                gu, rows, I, clamp_L, y));
}

int moe_nvfp4_e4m3_codes(const float* x, int64_t n, uint8_t* codes, moe_nvfp4_stream_t stream) {
    if (n < 0) return MOE_NVFP4_ESIZE;
    if (n > 0 && (x == nullptr || codes == nullptr)) return MOE_NVFP4_ENULL;
    if (n > 0 && !aligned(x, 4)) return MOE_NVFP4_EALIGN;
    if (n == 0) return MOE_NVFP4_OK;
    DeviceInfo di;
    int rc;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    return launch_status(launch(e4m3_codes_kernel, di.sms * 8, reinterpret_cast<cudaStream_t>(stream), x, n,
                                codes));
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
    return launch_status(launch_quantize<true>(x, nblk, global_scale, packed, sf, di,
                                               reinterpret_cast<cudaStream_t>(stream)));
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
        return launch_status(launch(nvfp4_dequantize_kernel<kDivNone>, static_cast<int>(grid), st, packed,
                                    sf, nblk, global_scale, out));
    if (global_scale >= 0x1p-90f && global_scale <= 0x1p90f)
        return launch_status(launch(nvfp4_dequantize_kernel<kDivMarkstein>, static_cast<int>(grid), st,
                                    packed, sf, nblk, global_scale, out));
    return launch_status(launch(nvfp4_dequantize_kernel<kDivIeee>, static_cast<int>(grid), st, packed, sf,
                                nblk, global_scale, out));
}

int moe_nvfp4_traffic_floor(const uint16_t* in, int64_t rows, int64_t width, int32_t kind,
                            uint8_t* packed, uint8_t* sf, moe_nvfp4_stream_t stream) {
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (kind < MOE_NVFP4_TRAFFIC_FUSED || kind > MOE_NVFP4_TRAFFIC_READ) return MOE_NVFP4_EMODE;
    int rc;
    DeviceInfo di;
    if (kind == MOE_NVFP4_TRAFFIC_EMPTY) {
        if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
        return launch_status(launch_shaped(empty_kernel, dim3(1), 32, st));
    }
    if (kind == MOE_NVFP4_TRAFFIC_READ) {
        if (rows < 0) return MOE_NVFP4_ESIZE;
        if (width <= 0 || width % 16 != 0) return MOE_NVFP4_EWIDTH;
        if (rows > 0 && width > INT64_MAX / 2 / rows) return MOE_NVFP4_ESIZE;
        if (rows == 0) return MOE_NVFP4_OK;
        if (in == nullptr || packed == nullptr) return MOE_NVFP4_ENULL;
        if (!aligned(in, 32) || !aligned(packed, 4)) return MOE_NVFP4_EALIGN;
        if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
        return launch_status(launch(read_sweep_kernel, di.sms * 4, st, reinterpret_cast<const uint32_t*>(in),
                                    rows * width / 16, reinterpret_cast<uint32_t*>(packed)));
    }
    const bool fused = kind == MOE_NVFP4_TRAFFIC_FUSED;
    if ((rc = check_common(in, rows, width, fused ? 4 : 2, packed, sf)) != MOE_NVFP4_OK || rows == 0) return rc;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    const int64_t nblk = rows * (width / 16);
    const uint32_t* in32 = reinterpret_cast<const uint32_t*>(in);
    // the launch shape the step itself takes for this size
    if (fused) {
        if (small_problem(nblk, di.sms, di.occ[1][0]))
            return launch_status(launch_shaped(traffic_small_kernel<16>, dim3(small_grid(nblk)), kSmallThreads,
                                               st, in32, nblk, packed, sf));
        return launch_status(launch(fused_traffic_kernel, grid_for(nblk, di.sms, di.occ_traffic[0]), st, in32,
                                    nblk, packed, sf));
    }
    if (small_problem(nblk, di.sms, di.occ_quant[0]))
        return launch_status(launch_shaped(traffic_small_kernel<8>, dim3(small_grid(nblk)), kSmallThreads, st,
                                           in32, nblk, packed, sf));
    return launch_status(launch(quantize_traffic_kernel, grid_for(nblk, di.sms, di.occ_traffic[1], kUnrollQuant),
                                st, in32, nblk, packed, sf));
}

int moe_nvfp4_check_offsets(const int32_t* expert_offsets, int32_t num_experts, int64_t rows,
                            const int32_t* out_offsets, int64_t out_rows, int32_t* status,
                            moe_nvfp4_stream_t stream) {
    if (num_experts < 0 || rows < 0 || out_rows < 0) return MOE_NVFP4_ESIZE;
    if (expert_offsets == nullptr || status == nullptr) return MOE_NVFP4_ENULL;
    if (!aligned(expert_offsets, 4) || !aligned(status, 4) || (out_offsets != nullptr && !aligned(out_offsets, 4)))
        return MOE_NVFP4_EALIGN;
    const int64_t tiles_x = (static_cast<int64_t>(num_experts) + 1 + kCheckTile - 1) / kCheckTile;
    const int64_t tiles_y = out_offsets == nullptr ? 1 : (static_cast<int64_t>(num_experts) + kCheckTile - 1) / kCheckTile;
    if (tiles_y > 65535) return MOE_NVFP4_ESIZE;
    DeviceInfo di;
    int rc;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    return launch_status(launch_shaped(check_offsets_kernel,
                                       dim3(static_cast<unsigned>(tiles_x), static_cast<unsigned>(tiles_y < 1 ? 1 : tiles_y)),
                                       kCheckTile, reinterpret_cast<cudaStream_t>(stream), expert_offsets,
                                       static_cast<int>(num_experts), rows, out_offsets, out_rows, status));
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

int moe_nvfp4_abi_version(void) { return 6; }

}  // extern "C"
