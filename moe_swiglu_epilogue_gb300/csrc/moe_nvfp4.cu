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
//     so a thread walks blocks in a grid-stride loop over [first, last) of
//     the active rows, with 256-bit L1-bypassing loads marked evict-first in
//     L2 (the stream is read once) and U blocks in flight per thread.
//   * Each thread owns whole blocks, so the amax needs no shuffles.
//   * E4M3 scale: cvt.rn.satfinite.e4m3x2.f32 (RNE, saturating at 448);
//     E2M1 nibbles: the half step is rounded with the exact fp32 trick
//     (t + 1.5*2^22) - 1.5*2^22, then cvt.rn.satfinite.e2m1x2.f32 maps the
//     signed half step to its nibble (RNE onto the E2M1 grid is exactly the
//     pages' step_to_idx table for half-step inputs).
//   * Fused path: SwiGLU in fast fp32 (ex2.approx + rcp.approx). A scale or
//     nibble decision whose input lies within a relative window W of a
//     rounding boundary (W bounds the fast path's error, with margin) is
//     redone from a double-precision SwiGLU value, the definition's value.
//     Quantize-only: exact division by a Markstein correction
//     (q = x*rcp_rn(d), r = fma(-q, d, x), q' = fma(r, rcp_rn(d), q)).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "moe_nvfp4.h"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;                 // blocks in flight per thread
constexpr int kMaxDevices = 64;

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

// Eight signed half steps (exact multiples of 0.5 in [-6, 6]) -> eight E2M1
// nibbles, element 0 in the low nibble of the low byte.
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

// ---------------------------------------------------------------------------
// Scalar pieces
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Nearest multiple of 0.5 to t in [0, 6], ties to an even multiple: at
// 1.5 * 2^22 the fp32 spacing is 0.5, so the add rounds t exactly so.
__device__ __forceinline__ float round_half_step(float t) {
    return __fadd_rn(__fadd_rn(t, 6291456.0f), -6291456.0f);
}

__device__ __forceinline__ float with_sign_of(float mag, float s) {
    return __uint_as_float(__float_as_uint(mag) | (__float_as_uint(s) & 0x80000000u));
}

// silu(min(g, L)) * clamp(u, -L, L) in fast fp32.
__device__ __forceinline__ float swiglu_fast(float g, float u, float L) {
    const float a = fminf(g, L);
    const float b = fminf(fmaxf(u, -L), L);
    const float e = ex2_approx(a * -1.44269504088896341f);   // exp(-a)
    const float r = rcp_approx(1.0f + e);
    return (a * r) * b;
}

// The definition's value: the formula in double precision, rounded once.
__device__ __noinline__ float swiglu_double(float g, float u, float L) {
    const double a = static_cast<double>(fminf(g, L));
    const double b = static_cast<double>(fminf(fmaxf(u, -L), L));
    const double y = a / (1.0 + exp(-a)) * b;
    return __double2float_rn(y);
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

// ---------------------------------------------------------------------------
// Fused deinterleave + clamped SwiGLU + NVFP4 quantize
// ---------------------------------------------------------------------------

struct FusedArgs {
    const uint16_t* gu;        // [rows, 2I]
    int64_t rows;
    int64_t bpr;               // blocks per row = I / 16
    float L;
    float W;                   // relative decision window
    const int32_t* offsets;    // [E+1] or null
    int E;
    uint8_t* packed;           // [rows, I/2]
    uint8_t* sf;               // [rows, I/16]
    unsigned long long* counters;   // [3] or null (counted variant)
    float* values;             // [rows, I] (fast-values variant)
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

template <bool kCount, bool kValues>
__device__ __forceinline__ void fused_block(const FusedArgs& A, int64_t blk, const uint32_t* w,
                                            unsigned long long& n_scale,
                                            unsigned long long& n_elem) {
    const float L = A.L, W = A.W;
    float y[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const int grp = i >> 3, j = i & 7;
        const uint32_t gw = w[8 * grp + (j >> 1)], uw = w[8 * grp + 4 + (j >> 1)];
        const float g = (j & 1) ? bf16_hi(gw) : bf16_lo(gw);
        const float u = (j & 1) ? bf16_hi(uw) : bf16_lo(uw);
        y[i] = swiglu_fast(g, u, L);
        amax = fmaxf(amax, fabsf(y[i]));
    }
    if (kValues) {
        float4* out = reinterpret_cast<float4*>(A.values + blk * 16);
#pragma unroll
        for (int k = 0; k < 4; k++) out[k] = make_float4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
        return;
    }
    const uint16_t* blk_in = A.gu + blk * 32;

    // scale: safe when both ends of the window round to the same code
    const float q = __fdiv_rn(amax, 6.0f);
    const uint32_t ends = e4m3x2_rn_sat(q * (1.0f + W), q * (1.0f - W));
    uint32_t code = ends & 0xFFu;
    if ((ends >> 8) != code) {
        // re-evaluate every element that could be the true maximum
        const float lim = amax * (1.0f - 2.0f * W);
        float am = 0.0f;
        for (int i = 0; i < 16; i++) {
            if (fabsf(y[i]) >= lim) {
                float g, u;
                gate_up_at(blk_in, i, g, u);
                y[i] = swiglu_double(g, u, L);
            }
            am = fmaxf(am, fabsf(y[i]));
        }
        code = e4m3x2_rn_sat(0.0f, __fdiv_rn(am, 6.0f)) & 0xFFu;
        if (kCount) n_scale++;
    }

    const float d = e4m3_value(code);
    const float inv = (code == 0u) ? 0.0f : rcp_approx(d);
    float hs[16];
    uint32_t near = 0;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const float t = fminf(fabsf(y[i]) * inv, 6.0f);
        const float h = round_half_step(t);
        near |= (fmaf(W, t, fabsf(t - h)) > 0.25f ? 1u : 0u) << i;
        hs[i] = with_sign_of(h, y[i]);
    }
    uint32_t lo = e2m1x8(hs), hi = e2m1x8(hs + 8);
    if (near != 0u) {
        for (int i = 0; i < 16; i++) {
            if (!((near >> i) & 1u)) continue;
            float g, u;
            gate_up_at(blk_in, i, g, u);
            const uint32_t nib = nibble_by_definition(swiglu_double(g, u, L), d, code);
            const int sh = 4 * (i & 7);
            if (i < 8) lo = (lo & ~(0xFu << sh)) | (nib << sh);
            else       hi = (hi & ~(0xFu << sh)) | (nib << sh);
            if (kCount) n_elem++;
        }
    }
    *reinterpret_cast<uint2*>(A.packed + blk * 8) = make_uint2(lo, hi);
    A.sf[blk] = static_cast<uint8_t>(code);
}

template <bool kCount, bool kValues>
__global__ void __launch_bounds__(kThreads)
swiglu_nvfp4_kernel(const FusedArgs A) {
    int64_t b0, b1;
    active_block_range(A.offsets, A.E, A.rows, A.bpr, b0, b1);
    const uint64_t pol = l2_evict_first_policy();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    unsigned long long n_blk = 0, n_scale = 0, n_elem = 0;
    for (int64_t base = b0 + static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; base < b1;
         base += stride * kUnroll) {
        uint32_t w[kUnroll][16];
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t blk = base + k * stride;
            if (blk < b1) {
                const uint16_t* p = A.gu + blk * 32;
                load_stream_32B(p, pol, w[k]);
                load_stream_32B(p + 16, pol, w[k] + 8);
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t blk = base + k * stride;
            if (blk < b1) {
                fused_block<kCount, kValues>(A, blk, w[k], n_scale, n_elem);
                n_blk++;
            }
        }
    }
    if (kCount) {
        atomicAdd(A.counters + 0, n_blk);
        if (n_scale) atomicAdd(A.counters + 1, n_scale);
        if (n_elem) atomicAdd(A.counters + 2, n_elem);
    }
}

// ---------------------------------------------------------------------------
// Quantize-only
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads)
nvfp4_quantize_kernel(const uint16_t* __restrict__ x, int64_t nblk,
                      uint8_t* __restrict__ packed, uint8_t* __restrict__ sf) {
    const uint64_t pol = l2_evict_first_policy();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; base < nblk;
         base += stride * kUnroll) {
        uint32_t w[kUnroll][8];
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t blk = base + k * stride;
            if (blk < nblk) load_stream_32B(x + blk * 16, pol, w[k]);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; k++) {
            const int64_t blk = base + k * stride;
            if (blk >= nblk) continue;
            float v[16];
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                v[i] = (i & 1) ? bf16_hi(w[k][i >> 1]) : bf16_lo(w[k][i >> 1]);
                amax = fmaxf(amax, fabsf(v[i]));
            }
            const uint32_t code = e4m3x2_rn_sat(0.0f, __fdiv_rn(amax, 6.0f)) & 0xFFu;
            const float d = e4m3_value(code);
            const float inv = (code == 0u) ? 0.0f : __frcp_rn(d);
            float hs[16];
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const float ax = fabsf(v[i]);
                const float q0 = ax * inv;                       // |x| / d to ~1 ulp
                const float r = fmaf(-q0, d, ax);                // exact residual
                const float q1 = fmaf(r, inv, q0);               // correctly rounded |x| / d
                hs[i] = with_sign_of(round_half_step(fminf(q1, 6.0f)), v[i]);
            }
            *reinterpret_cast<uint2*>(packed + blk * 8) = make_uint2(e2m1x8(hs), e2m1x8(hs + 8));
            sf[blk] = static_cast<uint8_t>(code);
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int occ_fused = 0, occ_fused_count = 0, occ_values = 0, occ_quant = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_NVFP4_ELAUNCH;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_NVFP4_ELAUNCH;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_fused, swiglu_nvfp4_kernel<false, false>, kThreads, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_fused_count, swiglu_nvfp4_kernel<true, false>, kThreads, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_values, swiglu_nvfp4_kernel<false, true>, kThreads, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &di.occ_quant, nvfp4_quantize_kernel, kThreads, 0) != cudaSuccess)
            return MOE_NVFP4_ELAUNCH;
        di.ready = true;
    }
    out = di;
    return MOE_NVFP4_OK;
}

int grid_for(int64_t nblk, int sms, int occ) {
    const int64_t want = (nblk + static_cast<int64_t>(kThreads) * kUnroll - 1) /
                         (static_cast<int64_t>(kThreads) * kUnroll);
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
    const double x_max = z * 1.4426950408889634;
    // exponent-argument rounding (|x| * 1.22 * 2^-24 in x, * ln 2 in exp),
    // ex2.approx (<= 2^-21), and nine fp32 roundings / approximate
    // reciprocals on the way from y to the scaled value t
    const double bound = x_max * 0.85 * std::ldexp(1.0, -24) + std::ldexp(1.0, -21) +
                         9.0 * std::ldexp(1.0, -24);
    return 2.0 * bound;
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
    if (rows == 0) return MOE_NVFP4_OK;
    DeviceInfo di;
    if ((rc = device_info(di)) != MOE_NVFP4_OK) return rc;
    FusedArgs A;
    A.gu = gu; A.rows = rows; A.bpr = I / 16; A.L = L; A.W = static_cast<float>(W);
    A.offsets = (E > 0) ? offsets : nullptr; A.E = E;
    A.packed = packed; A.sf = sf;
    A.counters = reinterpret_cast<unsigned long long*>(counters); A.values = values;
    const int64_t nblk = rows * (I / 16);
    if (values != nullptr) {
        swiglu_nvfp4_kernel<false, true><<<grid_for(nblk, di.sms, di.occ_values), kThreads, 0, stream>>>(A);
    } else if (counters != nullptr) {
        swiglu_nvfp4_kernel<true, false><<<grid_for(nblk, di.sms, di.occ_fused_count), kThreads, 0, stream>>>(A);
    } else {
        swiglu_nvfp4_kernel<false, false><<<grid_for(nblk, di.sms, di.occ_fused), kThreads, 0, stream>>>(A);
    }
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
    nvfp4_quantize_kernel<<<grid_for(nblk, di.sms, di.occ_quant), kThreads, 0,
                            reinterpret_cast<cudaStream_t>(stream)>>>(x, nblk, packed, sf);
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

int moe_swiglu_nvfp4_quantize_counted(const uint16_t* gu, int64_t rows, int64_t I, float clamp_L,
                                      const int32_t* expert_offsets, int32_t num_experts,
                                      uint8_t* packed, uint8_t* sf, uint64_t* counters,
                                      moe_nvfp4_stream_t stream) {
    if (rows > 0 && counters == nullptr) return MOE_NVFP4_ENULL;
    if (counters != nullptr && !aligned(counters, 8)) return MOE_NVFP4_EALIGN;
    return launch_fused(gu, rows, I, clamp_L, expert_offsets, num_experts, packed, sf, counters,
                        nullptr, reinterpret_cast<cudaStream_t>(stream));
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
        default: return "unknown error code";
    }
}

int moe_nvfp4_abi_version(void) { return 1; }

}  // extern "C"
