/*
 * moe_nvfp4.h -- C ABI of libmoe_swiglu_nvfp4.so, the GB300 (sm_103a)
 * kernels for the MoE expert activation step between the L1 and L2 GEMMs:
 * deinterleave the L1 output, clamped SwiGLU, NVFP4 quantize.
 *
 * Source of the operations (nvfp4-megamoe-kernel project pages):
 *  - "NVFP4-1.1 Approach Update", section "Revised approach: Compact SwiGLU
 *    output": the L1 GEMM writes BF16 column groups [gate*8, swiglu*8, ...];
 *    a deinterleave + quantize kernel turns them into x2-packed FP4
 *    (tokens, I/2) plus FP8 E4M3 scales (tokens, I/16); the compact plan
 *    quantizes a plain BF16 (tokens, I) tensor instead (quantize-only).
 *  - "2026-05-28 Status", commit "NVFP4-1.1: FP4 quantization primitives":
 *    E4M3 with bias 7, exponents 0-15, exp 15 / mant 7 NaN (max 448),
 *    subnormals m * 2^-9, round-to-nearest-even with mantissa carry; the
 *    half-step index 0..12 -> E2M1 index 0..7; per-element quantize + sign +
 *    pack. Table "What's DONE and PROVEN": SwiGLU clamping in the kernel.
 *  - "NVFP4-1.1 Approach, Part 2": the RNE half-step fix (s = 5.25 -> nibble
 *    6) and 16 values -> 8 packed bytes + 1 scale byte per block.
 *
 * What every call computes, per row and per block of 16 consecutive outputs:
 *    y_i   = the fp32 value of silu(min(g_i, L)) * clamp(u_i, -L, L),
 *            silu(a) = a / (1 + exp(-a))     (quantize-only: y_i = x_i)
 *    amax  = max |y_i|;   sf = E4M3_RNE_saturating(amax / 6)
 *    s_i   = y_i / value(sf)   (+-0 with the sign of y_i when sf == 0)
 *    h_i   = round_half_even(2 * min(|s_i|, 6))            in 0..12
 *    nib_i = {0,1,2,3,4,4,5,6,6,6,6,7,7}[h_i] | (sign(s_i) ? 8 : 0)
 *    packed[row, c/2] = nib(c even) | nib(c odd) << 4;  sf[row, c/16] = sf
 * The fp32 value y_i is the double-precision evaluation of the formula
 * rounded once to fp32. The fused kernel computes y_i with fast fp32
 * arithmetic (relative error far below the window below) and, wherever a
 * fast value lies within the window of a rounding boundary of the scale or
 * of a nibble, re-evaluates it with about 46 significant bits (double-float
 * arithmetic), so its scale and nibble decisions are those of the
 * definition. Quantize-only is exact throughout.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *    rows contiguous (leading dimension = width). Nothing is allocated,
 *    freed or synchronised; the work is launched on `stream` (a
 *    cudaStream_t; NULL = the legacy default stream) and the call returns
 *    without waiting for it.
 *  - Input pointers must be 32-byte aligned (256-bit loads); `packed` and
 *    `sf` must be 16-byte aligned; expert and output row offsets and the
 *    GEMMs' status word 4-byte aligned (every entry point below).
 *  - Return 0 on success or a negative MOE_NVFP4_E* code; arguments are
 *    checked on the host before any launch, so a rejected call launches
 *    nothing and leaves the outputs untouched. Faults inside a launched
 *    kernel surface, as with any CUDA launch, at the caller's next
 *    synchronisation.
 *  - Kernels are launched with programmatic stream serialization
 *    (programmatic dependent launch): each one waits until the preceding
 *    work in the stream has completed and is visible before it reads any
 *    memory, so stream order holds as usual, while its launch overlaps the
 *    tail of the preceding kernel. It also lets the kernel after it launch
 *    early; a following kernel that is itself launched with that attribute
 *    must wait for its dependency (griddepcontrol.wait /
 *    cudaGridDependencySynchronize) before reading these outputs, as any
 *    programmatic-launch consumer must.
 *  - The library caches, per device, the SM count and the kernels'
 *    occupancy on first use; it is otherwise stateless and thread-safe.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden visibility; these are its only exports. */
#if defined(__GNUC__)
#define MOE_NVFP4_API __attribute__((visibility("default")))
#else
#define MOE_NVFP4_API
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *moe_nvfp4_stream_t;

enum {
    MOE_NVFP4_OK = 0,
    MOE_NVFP4_ENULL = -1,       /* a required pointer is NULL while rows > 0 */
    MOE_NVFP4_EWIDTH = -2,      /* K or I is not a positive multiple of 16 */
    MOE_NVFP4_EALIGN = -3,      /* a pointer breaks the alignment rule above */
    MOE_NVFP4_ESIZE = -4,       /* rows < 0, or a byte count overflows int64 */
    MOE_NVFP4_ECLAMP = -5,      /* clamp_L not finite, not > 0, or > 2^64 */
    MOE_NVFP4_EOFFSETS = -6,    /* num_experts < 0, or offsets NULL with num_experts > 0 */
    MOE_NVFP4_ELAUNCH = -7,     /* the CUDA launch (or a device query) failed */
    MOE_NVFP4_ESCALE = -8,      /* global_scale not finite, or not > 0 */
    MOE_NVFP4_EMODE = -9,       /* an unknown output selector */
};

/*
 * Quantize-only (the pages' quantize_nvfp4_gpu; the "compact" flow):
 *   x      BF16 [rows, K]      (uint16 bit patterns)
 *   packed uint8 [rows, K/2]   two E2M1 nibbles per byte, even column low
 *   sf     uint8 [rows, K/16]  FP8 E4M3 scale codes (torch.float8_e4m3fn)
 * Bit-exact with the definition above for every finite input.
 */
MOE_NVFP4_API int moe_nvfp4_quantize(const uint16_t *x, int64_t rows, int64_t K,
                       uint8_t *packed, uint8_t *sf, moe_nvfp4_stream_t stream);

/*
 * Fused deinterleave + clamped SwiGLU + quantize (the pages'
 * deinterleave_quantize_nvfp4_cuda with the SwiGLU math in the kernel):
 *   gu       BF16 [rows, 2I], column groups [gate x8, up x8, ...]: output
 *            column c takes gate = gu[r, 16*(c/8) + c%8] and
 *            up = gu[r, 16*(c/8) + 8 + c%8]
 *   clamp_L  the SwiGLU clamp L, finite, 0 < L <= 2^64
 *   expert_offsets, num_experts
 *            optional DEVICE int32 [num_experts + 1], non-decreasing; segment
 *            e is rows [offsets[e], offsets[e+1]). When given, only rows in
 *            [offsets[0], offsets[num_experts]) (clamped to [0, rows]) are
 *            written and every other row of packed/sf is left untouched.
 *            Pass NULL and 0 to process all rows. The offsets are read on
 *            the device, so the call never synchronises and can be captured
 *            in a CUDA graph with offsets that change between replays.
 *   packed   uint8 [rows, I/2];  sf uint8 [rows, I/16]
 */
MOE_NVFP4_API int moe_swiglu_nvfp4_quantize(const uint16_t *gu, int64_t rows, int64_t I, float clamp_L,
                              const int32_t *expert_offsets, int32_t num_experts,
                              uint8_t *packed, uint8_t *sf, moe_nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * Extensions. The pages pass a global scale and use a BF16 intermediate and
 * padded per-expert rows without defining them ("NVFP4-1.1 Approach, Part 2":
 * quantize_activation_nvfp4's global_scale, the epilogue's l2_global_scale;
 * "NVFP4-1.1 Approach Update": the BF16 [gate*8, swiglu*8] store, the compact
 * BF16 (tokens, I) plan, padded_activated_fp4). The readings implemented:
 *  - two-level NVFP4: every value is multiplied by the FP32 global scale gs
 *    (v = fl(value * gs)) and v is quantized as above; dequantization divides
 *    by gs. Products must not overflow fp32.
 *  - BF16 compat: the fp32 SwiGLU is rounded to BF16 (RNE) before the
 *    global scale and the quantization, as the pages' two-kernel flow did;
 *    the compact writer stores that BF16 tensor [rows, I].
 *  - padded output: input row r of segment e is written to output row
 *    out_offsets[e] + (r - offsets[e]); rows of the output not written keep
 *    their contents; destinations outside [0, out_rows) are skipped. The
 *    destination ranges of different segments must not overlap (where they
 *    do, which segment's row lands there is unspecified).
 * All are exact (bit-equal to the definitions, like the entry points above).
 * ------------------------------------------------------------------------- */

typedef struct moe_nvfp4_fused_options {
    float global_scale;          /* > 0 and finite; 1 = single-level NVFP4 */
    int32_t round_to_bf16;       /* nonzero: quantize the BF16-rounded SwiGLU */
    const int32_t *out_offsets;  /* DEVICE int32 [num_experts + 1], or NULL: padded output rows */
    int64_t out_rows;            /* rows of packed / sf when out_offsets is given */
} moe_nvfp4_fused_options;

/* Quantize-only with a global scale: x BF16 [rows, K] -> packed [rows, K/2],
 * sf [rows, K/16] of v = fl(x * global_scale). Same rules as
 * moe_nvfp4_quantize; MOE_NVFP4_ESCALE for a bad scale. */
MOE_NVFP4_API int moe_nvfp4_quantize_scaled(const uint16_t *x, int64_t rows, int64_t K,
                                            float global_scale, uint8_t *packed, uint8_t *sf,
                                            moe_nvfp4_stream_t stream);

/* The fused step with options (NULL = the plain step). With out_offsets,
 * packed and sf have out_rows rows and num_experts must be > 0.
 * MOE_NVFP4_ESIZE also for rows * I / 16 >= 2^32 (256 GiB of input or more,
 * beyond one device's memory with the outputs); the same for
 * moe_swiglu_bf16. */
MOE_NVFP4_API int moe_swiglu_nvfp4_quantize_ex(const uint16_t *gu, int64_t rows, int64_t I,
                                               float clamp_L, const int32_t *expert_offsets,
                                               int32_t num_experts,
                                               const moe_nvfp4_fused_options *options,
                                               uint8_t *packed, uint8_t *sf,
                                               moe_nvfp4_stream_t stream);

/* Compact writer: out BF16 [rows, I] (16-byte aligned) = RN_bf16 of the fp32
 * SwiGLU, for the rows of the segments (others untouched) or all rows. */
MOE_NVFP4_API int moe_swiglu_bf16(const uint16_t *gu, int64_t rows, int64_t I, float clamp_L,
                                  const int32_t *expert_offsets, int32_t num_experts,
                                  uint16_t *out, moe_nvfp4_stream_t stream);

/* Dequantization (the consumer's view): packed [rows, K/2], sf [rows, K/16]
 * (16-byte aligned) -> out BF16 [rows, K] (32-byte aligned) =
 * RN_bf16(e2m1 * e4m3 / global_scale); the product is exact in fp32. */
MOE_NVFP4_API int moe_nvfp4_dequantize(const uint8_t *packed, const uint8_t *sf, int64_t rows,
                                       int64_t K, float global_scale, uint16_t *out,
                                       moe_nvfp4_stream_t stream);

/*
 * Diagnostic: the fp32 SwiGLU values y [rows, I] of the fused kernel's fast
 * path (before its boundary re-evaluation), in output-column order. Used to
 * measure the fast path's error against a double-precision evaluation.
 * Same argument rules as moe_swiglu_nvfp4_quantize; y must be 16-byte
 * aligned.
 */
MOE_NVFP4_API int moe_swiglu_fast_values(const uint16_t *gu, int64_t rows, int64_t I, float clamp_L,
                           float *y, moe_nvfp4_stream_t stream);

/*
 * Diagnostic: the fp32 SwiGLU values y [rows, I] by the definition (the
 * formula evaluated with about 46 significant bits and rounded once to fp32),
 * as the fused kernel computes them wherever a fast value falls inside its
 * decision window. Same argument rules as moe_swiglu_fast_values.
 */
MOE_NVFP4_API int moe_swiglu_precise_values(const uint16_t *gu, int64_t rows, int64_t I,
                                            float clamp_L, float *y, moe_nvfp4_stream_t stream);

/*
 * Diagnostic: the E4M3 conversion every kernel here takes its scale codes
 * with (the pages' "FP8 E4M3" scale format: round to nearest even, values
 * past 448 saturate to 448 = 0x7E), applied to n fp32 values: codes[i] =
 * E4M3(x[i]). x (fp32 [n]) and codes (uint8 [n]) are DEVICE buffers owned
 * by the caller. Errors: MOE_NVFP4_ESIZE for n < 0, MOE_NVFP4_ENULL for a
 * null pointer with n > 0, MOE_NVFP4_EALIGN for x not 4-byte aligned; n == 0
 * launches nothing.
 */
MOE_NVFP4_API int moe_nvfp4_e4m3_codes(const float *x, int64_t n, uint8_t *codes,
                                       moe_nvfp4_stream_t stream);

/*
 * Diagnostic: as moe_swiglu_nvfp4_quantize, and also adds to the caller's
 * DEVICE counters (uint64 [3], not cleared by the call):
 *   [0] blocks processed, [1] blocks whose scale needed the re-evaluation,
 *   [2] elements whose nibble needed the re-evaluation.
 */
MOE_NVFP4_API int moe_swiglu_nvfp4_quantize_counted(const uint16_t *gu, int64_t rows, int64_t I,
                                      float clamp_L, const int32_t *expert_offsets,
                                      int32_t num_experts, uint8_t *packed, uint8_t *sf,
                                      uint64_t *counters, moe_nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * The step fused into the MoE L1 GEMM's epilogue (the pages' target:
 * "2026-05-28 Status", priority 3, fuse the amax and FP4 pack into the
 * L1 -> L2 path; "NVFP4-1.1 Approach, Part 2", the TMEM -> registers -> FP4
 * epilogue plan). For every expert segment e, rows [offsets[e], offsets[e+1])
 * of x are multiplied by that expert's weights:
 *   gu[r, c] = sum_k x[r, k] * w1[e, c, k]     (fp32 accumulation)
 * and the epilogue applies the fused step above to gu's fp32 values (no
 * BF16 rounding of gu): output column c takes gate gu[r, 16*(c/8) + c%8]
 * and up gu[r, 16*(c/8) + 8 + c%8], y = silu(min(g, L)) * clamp(u, -L, L)
 * in fast fp32, then the NVFP4 block quantization of y exactly as
 * moe_nvfp4_quantize defines it (applied to fp32 values).
 *   x        BF16 [rows, H], row-major, 16-byte aligned; H % 64 == 0
 *   w1       BF16 [num_experts, 2I, H], row-major, 16-byte aligned: row c of
 *            expert e holds the weights of gu column c (so the rows come in
 *            [gate x8, up x8] groups); I % 128 == 0
 *   expert_offsets, num_experts
 *            DEVICE int32 [num_experts + 1], non-decreasing, required
 *            (1 <= num_experts <= 2048; one segment [0, rows) for a dense
 *            GEMM). Offsets are clamped into [0, rows]; rows outside every
 *            segment are left untouched in packed / sf.
 *   packed   uint8 [rows, I/2], sf uint8 [rows, I/16], 16-byte aligned
 *   status   optional DEVICE int32: the kernel writes a nonzero code there
 *            if one of its internal waits expired (about a second; a fault
 *            elsewhere on the device); untouched otherwise. May be NULL.
 *            After an expired wait the kernel still waits (bounded) for
 *            the TMA loads and MMAs it issued before it releases its TMEM
 *            and exits.
 * Uses every SM (one CTA each, ~206 KB of shared memory and all 512 TMEM
 * columns of the SM), tcgen05 tensor cores and TMA. Allocates nothing.
 * Returns the codes above; MOE_NVFP4_ELAUNCH also when the CUDA driver's
 * tensor-map encoder is unavailable or rejects the tensors.
 * ------------------------------------------------------------------------- */
MOE_NVFP4_API int moe_l1_gemm_swiglu_nvfp4(const uint16_t *x, const uint16_t *w1, int64_t rows,
                                           int64_t H, int64_t I, float clamp_L,
                                           const int32_t *expert_offsets, int32_t num_experts,
                                           uint8_t *packed, uint8_t *sf, int32_t *status,
                                           moe_nvfp4_stream_t stream);

/* Diagnostic: the same GEMM's fp32 accumulators gu [rows, 2I] (16-byte
 * aligned) for the rows of the segments, in the same accumulation order as
 * moe_l1_gemm_swiglu_nvfp4 (the same kernel with the epilogue storing the
 * accumulators instead). */
MOE_NVFP4_API int moe_l1_gemm_accumulators(const uint16_t *x, const uint16_t *w1, int64_t rows,
                                           int64_t H, int64_t I, const int32_t *expert_offsets,
                                           int32_t num_experts, float *acc, int32_t *status,
                                           moe_nvfp4_stream_t stream);

/* The unfused flows the pages describe, with the same GEMM (for the
 * comparison with the fused step and for BF16 consumers):
 *   output = MOE_L1_GEMM_GU:     out = BF16 gu [rows, 2I] (RN of the fp32
 *                                accumulators, [gate x8, up x8] columns:
 *                                "NVFP4-1.1 Approach Update", current flow)
 *   output = MOE_L1_GEMM_SWIGLU: out = BF16 SwiGLU [rows, I] (RN of the
 *                                epilogue's fp32 SwiGLU values: the planned
 *                                compact flow); clamp_L is used only here
 * out is 16-byte aligned; other arguments as moe_l1_gemm_swiglu_nvfp4.
 * MOE_NVFP4_EMODE for any other output value. */
enum { MOE_L1_GEMM_GU = 0, MOE_L1_GEMM_SWIGLU = 1 };
MOE_NVFP4_API int moe_l1_gemm_bf16(const uint16_t *x, const uint16_t *w1, int64_t rows, int64_t H,
                                   int64_t I, float clamp_L, const int32_t *expert_offsets,
                                   int32_t num_experts, int32_t output, uint16_t *out, int32_t *status,
                                   moe_nvfp4_stream_t stream);

/* The same fused L1 GEMM with NVFP4 weights:
 *   w1_packed  uint8 [num_experts, 2I, H/2]: two E2M1 nibbles per byte along
 *              K, even k in the low nibble -- the layout moe_nvfp4_quantize
 *              writes for a BF16 [num_experts * 2I, H] weight matrix
 *   w1_sf      uint8 [num_experts, 2I, H/16]: E4M3 codes, one per 16 along K
 * The kernel expands each weight tile to BF16 in shared memory (exactly:
 * e2m1 * e4m3 has at most 6 significant bits), so its outputs equal those
 * of moe_l1_gemm_swiglu_nvfp4 on the dequantized weights bit for bit, while
 * a weight costs 0.5625 bytes of HBM traffic instead of 2. H % 256 == 0;
 * both weight pointers 16-byte aligned; other arguments as above. Wait
 * codes in `status` also include 5 (MMA issuer / expanded weight tile),
 * 6 (expanders / loaded stage) and 7 (expanders / free expanded tile). */
MOE_NVFP4_API int moe_l1_gemm_w4_swiglu_nvfp4(const uint16_t *x, const uint8_t *w1_packed,
                                              const uint8_t *w1_sf, int64_t rows, int64_t H, int64_t I,
                                              float clamp_L, const int32_t *expert_offsets,
                                              int32_t num_experts, uint8_t *packed, uint8_t *sf,
                                              int32_t *status, moe_nvfp4_stream_t stream);

/* Diagnostic: the fp32 accumulators [rows, 2I] of moe_l1_gemm_w4_swiglu_nvfp4. */
MOE_NVFP4_API int moe_l1_gemm_w4_accumulators(const uint16_t *x, const uint8_t *w1_packed,
                                              const uint8_t *w1_sf, int64_t rows, int64_t H, int64_t I,
                                              const int32_t *expert_offsets, int32_t num_experts,
                                              float *acc, int32_t *status, moe_nvfp4_stream_t stream);

/* Diagnostic of the failure path of moe_l1_gemm_swiglu_nvfp4's kernel,
 * with every internal wait limited to wait_cycles SM clock cycles (1000 ..
 * 2e9) and one of two faults made on purpose (no GPU fault: a wait that can
 * never complete):
 *   MOE_L1_GEMM_SELFTEST_NO_LOADS    the producer issues no loads, so the
 *                                    first MMA wait never completes
 *   MOE_L1_GEMM_SELFTEST_NO_RELEASE  the epilogue never releases an
 *                                    accumulator; the grid is one CTA, which
 *                                    runs every tile, so the MMA issuer
 *                                    stops after two tiles with loads and
 *                                    MMAs issued before it
 * Each role stops when its wait expires or another role's did: the DEVICE
 * int32 status (required here) receives the code of an expired wait (1
 * producer / free stage, 2 MMA issuer / free accumulator, 3 MMA issuer /
 * loaded stage, 4 epilogue / finished accumulator; 8 if a load or MMA
 * issued before the stop did not complete within the limit). Before the
 * TMEM is released the producer waits for its issued loads and the MMA
 * issuer for its issued MMAs (the same drain every abort takes); packed / sf
 * are not written. The kernels run normally afterwards. MOE_NVFP4_EMODE for
 * another mode. */
enum { MOE_L1_GEMM_SELFTEST_NO_LOADS = 1, MOE_L1_GEMM_SELFTEST_NO_RELEASE = 2 };
MOE_NVFP4_API int moe_l1_gemm_wait_selftest(const uint16_t *x, const uint16_t *w1, int64_t rows,
                                            int64_t H, int64_t I, const int32_t *expert_offsets,
                                            int32_t num_experts, uint8_t *packed, uint8_t *sf,
                                            int32_t *status, int64_t wait_cycles, int32_t mode,
                                            moe_nvfp4_stream_t stream);

/*
 * Diagnostic: the memory traffic of a step with none of its arithmetic, in
 * the launch shape the step itself takes for the same size (the floor its
 * kernel can reach on this GPU), or a bare launch, or a read-only sweep:
 *   MOE_NVFP4_TRAFFIC_FUSED     in BF16 [rows, 2*width]: per 16 outputs, the
 *                               64 input bytes of moe_swiglu_nvfp4_quantize
 *                               read, 8 bytes of packed [rows, width/2] and
 *                               1 byte of sf [rows, width/16] written (the
 *                               XOR of the words read, so no load is dead)
 *   MOE_NVFP4_TRAFFIC_QUANTIZE  as above with the 32 input bytes of
 *                               moe_nvfp4_quantize, in BF16 [rows, width]
 *   MOE_NVFP4_TRAFFIC_EMPTY     one CTA that does nothing (the cost of a
 *                               launch); every other argument is ignored
 *   MOE_NVFP4_TRAFFIC_READ      reads rows * width BF16 values of `in` with
 *                               the default L2 policy and XORs them into the
 *                               4 bytes at `packed` (4-byte aligned): a sweep
 *                               larger than L2 leaves it holding clean lines
 *                               (a cache flush that creates no write-backs)
 * Alignment and size rules as moe_swiglu_nvfp4_quantize / moe_nvfp4_quantize;
 * MOE_NVFP4_EMODE for an unknown kind. No counterpart on the pages: used to
 * measure how close the kernels run to what their memory access pattern
 * allows.
 */
enum {
    MOE_NVFP4_TRAFFIC_FUSED = 0,
    MOE_NVFP4_TRAFFIC_QUANTIZE = 1,
    MOE_NVFP4_TRAFFIC_EMPTY = 2,
    MOE_NVFP4_TRAFFIC_READ = 3,
};
MOE_NVFP4_API int moe_nvfp4_traffic_floor(const uint16_t *in, int64_t rows, int64_t width,
                                          int32_t kind, uint8_t *packed, uint8_t *sf,
                                          moe_nvfp4_stream_t stream);

/*
 * Checks, on the device, the preconditions the fused entry points place on
 * their offsets (the expert segments [offsets[e], offsets[e+1]) of
 * moe_swiglu_nvfp4_quantize and, with padded output, the destination rows
 * out_offsets[e] + (r - offsets[e]) of moe_swiglu_nvfp4_quantize_ex), which
 * the kernels themselves do not check: they clamp offsets into the buffers,
 * so bad offsets never make them access memory out of bounds, but
 * non-monotone offsets drop or repeat rows, and overlapping destination
 * ranges make two segments race for the same output rows.
 *   expert_offsets  DEVICE int32 [num_experts + 1] (required)
 *   rows            rows of the input
 *   out_offsets     DEVICE int32 [num_experts + 1] or NULL (then not checked)
 *   out_rows        rows of the padded output (destination rows are clipped
 *                   to [0, out_rows) before the overlap test, as the kernel
 *                   skips the others)
 *   status          DEVICE int32: the kernel ORs in
 *                     MOE_NVFP4_CHECK_DECREASING  some offsets[e+1] < offsets[e]
 *                     MOE_NVFP4_CHECK_OUTSIDE     some offsets[e] outside [0, rows]
 *                     MOE_NVFP4_CHECK_OVERLAP     two segments' destination rows intersect
 *                   and never clears a bit: zero it before the call. The
 *                   kernel never traps; it only writes this word.
 * Launched on `stream` like the step, so it can be enqueued just before it
 * (or captured with it in a CUDA graph). The overlap test compares every
 * pair of segments (num_experts^2 / 2 tests; num_experts <= 16,776,960 with
 * out_offsets). Errors: MOE_NVFP4_ESIZE for negative sizes or too many
 * segments, MOE_NVFP4_ENULL, MOE_NVFP4_EALIGN (4-byte alignment).
 * The specification of the step makes monotone offsets a precondition and
 * asks for a device-side flag that never traps; this is that check, as a
 * call of its own rather than a separate build of the library.
 */
enum {
    MOE_NVFP4_CHECK_DECREASING = 1,
    MOE_NVFP4_CHECK_OUTSIDE = 2,
    MOE_NVFP4_CHECK_OVERLAP = 4,
};
MOE_NVFP4_API int moe_nvfp4_check_offsets(const int32_t *expert_offsets, int32_t num_experts,
                                          int64_t rows, const int32_t *out_offsets,
                                          int64_t out_rows, int32_t *status,
                                          moe_nvfp4_stream_t stream);

/* The relative window the fused kernel uses for a clamp L: a scale or
 * nibble decision whose fast-path input lies within this relative distance
 * of a rounding boundary is redone from the definition's SwiGLU value.
 * It bounds the fast path's relative error with margin: when every gate
 * that can still reach a nonzero nibble for this L is >= -16 (L up to about
 * 135), from the fast silu's largest error over every BF16 gate >= -16
 * (measured exhaustively by the test suite) plus four roundings, times 1.5;
 * beyond that, from an analytic bound that grows with the most negative
 * such gate, times 2. Returns a negative value for an invalid L. */
MOE_NVFP4_API double moe_swiglu_nvfp4_window(float clamp_L);

/* Static text for a return code. */
MOE_NVFP4_API const char *moe_nvfp4_strerror(int code);

/* ABI version of this header (incremented on any signature change or added entry point). */
MOE_NVFP4_API int moe_nvfp4_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
