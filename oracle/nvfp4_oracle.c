/*
 * NVFP4 oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, single-threaded C99 restatement of what the MoE expert
 * activation step computes: deinterleave the L1 GEMM's BF16 [gate x8, up x8]
 * column groups, apply clamped SwiGLU, and quantize to NVFP4 (E2M1 nibbles,
 * one FP8 E4M3 scale per 16 consecutive outputs of a row).
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library. The CUDA library never links it, and the two share
 * no source, header, table or helper.
 *
 * Sources, all from the nvfp4-megamoe-kernel project pages:
 *   [P2]  "NVFP4-1.1 Approach, Part 2" -- the debugging log on the FP8 E4M3
 *         cast (subnormal dequantization, the exponent-15 / 448 clamp, the
 *         250 -> 256 mantissa-overflow case) and on the E2M1 nibble
 *         round-to-nearest-even fix (the s = 5.25 case).
 *   [ST]  "2026-05-28 Status", the commit "NVFP4-1.1: FP4 quantization
 *         primitives for CuTeDSL kernels" (bias 7, exponents 0-15, NaN at
 *         exp 15 / mant 7, subnormal m * 2^-9, RNE, overflow carry) and the
 *         table row "MoE fused SwiGLU (NVFP4): clamping in kernel".
 *   [AU]  "NVFP4-1.1 Approach Update", section "Revised approach: Compact
 *         SwiGLU output" (the interleaved [gate*8, swiglu*8, ...] layout, the
 *         (tokens, I/2) x2-packed FP4 and (tokens, I/16) E4M3 scale outputs).
 *
 * Arithmetic: formats and rounding are done with integer/bit arithmetic on
 * the exact binary value. The SwiGLU value is evaluated in double precision
 * and rounded once to fp32 (the pages fix fp32 only for the quantization
 * steps, which operate on the fp32 activation). Readings of points the pages
 * leave open are marked READING.
 *
 * Every function is pinned, independently of this file, by
 * tests/test_oracle_pins.py (pages' printed values, exhaustive and
 * brute-force searches, torch's float8_e4m3fn cast, exact rational
 * arithmetic, decimal high-precision SwiGLU).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

static uint32_t f32_bits(float v) { uint32_t b; memcpy(&b, &v, 4); return b; }
static float bits_f32(uint32_t b) { float v; memcpy(&v, &b, 4); return v; }

/* BF16 is the top half of an fp32 bit pattern; widening is exact. */
EXPORT float bf16_to_float32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* n / 2^k rounded to the nearest integer, ties to even (n >= 0, k >= 1). */
static uint64_t round_shift_nearest_even(uint64_t n, int k)
{
    if (k > 62) return 0;              /* n < 2^24 here, so n / 2^k < 1/2 */
    uint64_t q = n >> k;
    uint64_t rem = n & ((1ull << k) - 1);
    uint64_t half = 1ull << (k - 1);
    if (rem > half || (rem == half && (q & 1))) q += 1;
    return q;
}

/*
 * fp32 -> FP8 E4M3 bit pattern, round to nearest even, saturating [ST] [P2].
 *   bias 7; exponent fields 0..15 are all finite except exp 15 / mant 7 (NaN);
 *   so the largest finite value is exp 15 / mant 6 = 448;
 *   subnormals (exp field 0) are m * 2^-9;
 *   a mantissa that rounds up to 8 carries into the exponent (250 -> 256).
 * READING: results that would pass 448 (or land on the NaN code) clamp to
 * 448, as the pages' cast clamps; +-inf also clamps; NaN stays NaN.
 */
EXPORT uint8_t fp8_e4m3_from_float32(float v)
{
    uint32_t b = f32_bits(v);
    uint8_t sign = (uint8_t)((b >> 24) & 0x80u);
    uint32_t mag = b & 0x7fffffffu;
    if (mag > 0x7f800000u) return (uint8_t)(sign | 0x7f);
    if (mag == 0x7f800000u) return (uint8_t)(sign | 0x7e);
    if (mag == 0) return sign;

    /* |v| = sig * 2^x exactly */
    uint32_t ebits = mag >> 23, frac = mag & 0x7fffffu;
    uint64_t sig;
    int x;
    if (ebits == 0) { sig = frac; x = -149; }
    else { sig = frac | 0x800000u; x = (int)ebits - 150; }
    int top = 0;                                  /* index of the leading 1 */
    while ((sig >> (top + 1)) != 0) top++;
    int e = top + x;                              /* floor(log2 |v|) */

    if (e < -6) {
        /* below the smallest normal 2^-6: m = RNE(|v| * 2^9); m == 8 is
         * 2^-6 itself, whose code (exp 1, mant 0) is also 8 */
        uint64_t m = round_shift_nearest_even(sig, -(x + 9));
        return (uint8_t)(sign | (uint8_t)m);
    }
    /* |v| = 2^e * (1 + f); mantissa = RNE(8 f); here top == 23 */
    uint64_t q = round_shift_nearest_even(sig, top - 3);   /* 8 .. 16 */
    if (q == 16) { q = 8; e += 1; }                         /* carry */
    int mant = (int)q - 8;
    int E = e + 7;
    if (E > 15 || (E == 15 && mant == 7)) return (uint8_t)(sign | 0x7e);
    return (uint8_t)(sign | (uint8_t)((E << 3) | mant));
}

/* FP8 E4M3 bit pattern -> value [ST] [P2]: exp 0 gives m * 2^-9,
 * otherwise 2^(E-7) * (1 + m/8); exp 15 / mant 7 is NaN. */
EXPORT float fp8_e4m3_to_float32(uint8_t c)
{
    int E = (c >> 3) & 15, m = c & 7;
    if (E == 15 && m == 7) return (c & 0x80) ? -NAN : NAN;
    double mag = (E == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, E - 7);
    return (float)((c & 0x80) ? -mag : mag);
}

/*
 * Half-step index h (0..12, h/2 = the magnitude on a 0.5 grid) -> E2M1
 * magnitude index 0..7 [ST] [P2]. The pages print step_to_idx[11] = 7 and,
 * through the s = 5.25 case, step_to_idx[10] = 6.
 * READING: every entry maps h/2 to the nearest E2M1 magnitude
 * {0, .5, 1, 1.5, 2, 3, 4, 6}, a tie going to the code with an even
 * mantissa bit: 2.5 -> 2 (idx 4), 3.5 -> 4 (idx 6), 5 -> 4 (idx 6).
 */
static const uint8_t step_to_idx[13] = {0, 1, 2, 3, 4, 4, 5, 6, 6, 6, 6, 7, 7};

EXPORT int half_step_to_e2m1_idx(int h)
{
    if (h < 0 || h > 12) return -1;
    return step_to_idx[h];
}

/* E2M1 nibble (sign bit 3, magnitude index bits 0-2) -> value. */
EXPORT float e2m1_nibble_to_float32(uint8_t nib)
{
    static const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    float v = mag[nib & 7];
    return (nib & 8) ? -v : v;
}

/*
 * Scaled value s -> E2M1 nibble [P2] [ST]:
 *   h = round-half-to-even(2 * min(|s|, 6))   -- the pages' RNE fix; a
 *       round-half-up here was their 22% failure (s = 5.25 must give 6);
 *   idx = step_to_idx[h];  nibble = idx | 8 when s is negative.
 * READING: the sign is the IEEE sign bit, so -0 gives nibble 8.
 */
EXPORT uint8_t quantize_e2m1_nibble(float s)
{
    float m = fminf(fabsf(s), 6.0f);
    int h = (int)nearbyintf(2.0f * m);   /* default rounding mode: RNE */
    return (uint8_t)(step_to_idx[h] | (signbit(s) ? 8 : 0));
}

/*
 * Clamped SwiGLU of one gate/up pair: silu(min(g, L)) * clamp(u, -L, L),
 * silu(a) = a / (1 + exp(-a)) ([ST] table: "clamping in kernel").
 * Evaluated in double precision and rounded once to fp32.
 */
EXPORT float swiglu_clamped(float g, float u, float L)
{
    double a = (double)fminf(g, L);
    double b = (double)fminf(fmaxf(u, -L), L);
    double y = a / (1.0 + exp(-a)) * b;
    return (float)y;
}

/*
 * One 16-element NVFP4 block [P2] [ST]:
 *   amax = max |y_i|;  sf = E4M3(amax / 6)  (fp32 division);
 *   d = value of sf;  s_i = y_i / d (fp32 division)   READING: divide by the
 *   quantized scale; when d == 0, s_i = +-0 with the sign of y_i;
 *   nibble_i = quantize_e2m1_nibble(s_i);
 *   byte j = nibble_{2j} | nibble_{2j+1} << 4   READING: even element in the
 *   low nibble (the float4_e2m1fn_x2 convention).
 */
EXPORT void quantize_nvfp4_block(const float *y, uint8_t *packed8, uint8_t *sf)
{
    float amax = 0.0f;
    for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(y[i]));
    uint8_t code = fp8_e4m3_from_float32(amax / 6.0f);
    float d = fp8_e4m3_to_float32(code);
    uint8_t nib[16];
    for (int i = 0; i < 16; i++) {
        float s = (d == 0.0f) ? copysignf(0.0f, y[i]) : y[i] / d;
        nib[i] = quantize_e2m1_nibble(s);
    }
    for (int j = 0; j < 8; j++) packed8[j] = (uint8_t)(nib[2 * j] | (nib[2 * j + 1] << 4));
    *sf = code;
}

/* Quantize-only: x BF16 [rows, K] -> packed [rows, K/2], sf [rows, K/16]. */
EXPORT int quantize_nvfp4(const uint16_t *x, int64_t rows, int64_t K,
                          uint8_t *packed, uint8_t *sf)
{
    if (rows < 0 || K <= 0 || K % 16 != 0) return -1;
    float y[16];
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < K / 16; b++) {
            for (int i = 0; i < 16; i++) y[i] = bf16_to_float32(x[r * K + 16 * b + i]);
            quantize_nvfp4_block(y, packed + r * (K / 2) + 8 * b, sf + r * (K / 16) + b);
        }
    return 0;
}

/*
 * Clamped SwiGLU of output column c of row r of the interleaved L1 output
 * gu [rows, 2I] ([AU]: "[gate*8, swiglu*8, ...]" column groups of 8):
 * gate at column 16*(c/8) + c%8, up 8 columns further on.
 */
static float swiglu_at(const uint16_t *gu, int64_t I, float L, int64_t r, int64_t c)
{
    const uint16_t *row = gu + r * 2 * I;
    int64_t gcol = 16 * (c / 8) + (c % 8);
    return swiglu_clamped(bf16_to_float32(row[gcol]), bf16_to_float32(row[gcol + 8]), L);
}

static void swiglu_quantize_row(const uint16_t *gu, int64_t I, float L, int64_t r,
                                uint8_t *packed, uint8_t *sf)
{
    float y[16];
    for (int64_t b = 0; b < I / 16; b++) {
        for (int i = 0; i < 16; i++) y[i] = swiglu_at(gu, I, L, r, 16 * b + i);
        quantize_nvfp4_block(y, packed + r * (I / 2) + 8 * b, sf + r * (I / 16) + b);
    }
}

/*
 * Fused: gu BF16 [rows, 2I] -> packed [rows, I/2], sf [rows, I/16].
 * With expert offsets (num_experts > 0), the rows of segment e are
 * [offsets[e], offsets[e+1]); only rows of some segment are written, all
 * other rows of the outputs are left as they were.
 */
EXPORT int swiglu_quantize_nvfp4(const uint16_t *gu, int64_t rows, int64_t I, float L,
                                 const int32_t *offsets, int32_t num_experts,
                                 uint8_t *packed, uint8_t *sf)
{
    if (rows < 0 || I <= 0 || I % 16 != 0) return -1;
    if (num_experts <= 0) {
        for (int64_t r = 0; r < rows; r++) swiglu_quantize_row(gu, I, L, r, packed, sf);
        return 0;
    }
    for (int32_t e = 0; e < num_experts; e++)
        for (int64_t r = offsets[e]; r < offsets[e + 1]; r++)
            if (r >= 0 && r < rows) swiglu_quantize_row(gu, I, L, r, packed, sf);
    return 0;
}

/* Sampled evaluation: block `blk[k]` of row `row[k]` of the fused step,
 * written to packed_out[8k..8k+7] and sf_out[k]. */
EXPORT void swiglu_quantize_nvfp4_blocks(const uint16_t *gu, int64_t I, float L,
                                         const int64_t *row, const int64_t *blk, int64_t n,
                                         uint8_t *packed_out, uint8_t *sf_out)
{
    float y[16];
    for (int64_t k = 0; k < n; k++) {
        for (int i = 0; i < 16; i++) y[i] = swiglu_at(gu, I, L, row[k], 16 * blk[k] + i);
        quantize_nvfp4_block(y, packed_out + 8 * k, sf_out + k);
    }
}

/* Sampled evaluation of the quantize-only step, as above. */
EXPORT void quantize_nvfp4_blocks(const uint16_t *x, int64_t K,
                                  const int64_t *row, const int64_t *blk, int64_t n,
                                  uint8_t *packed_out, uint8_t *sf_out)
{
    float y[16];
    for (int64_t k = 0; k < n; k++) {
        for (int i = 0; i < 16; i++) y[i] = bf16_to_float32(x[row[k] * K + 16 * blk[k] + i]);
        quantize_nvfp4_block(y, packed_out + 8 * k, sf_out + k);
    }
}

/* The fp32 SwiGLU values of rows [r0, r1): y_out [(r1-r0), I]. */
EXPORT void swiglu_values(const uint16_t *gu, int64_t I, float L, int64_t r0, int64_t r1,
                          float *y_out)
{
    for (int64_t r = r0; r < r1; r++)
        for (int64_t c = 0; c < I; c++) y_out[(r - r0) * I + c] = swiglu_at(gu, I, L, r, c);
}

/* Elementwise clamped SwiGLU over arrays (input construction in tests). */
EXPORT void swiglu_clamped_array(const float *g, const float *u, int64_t n, float L, float *y)
{
    for (int64_t i = 0; i < n; i++) y[i] = swiglu_clamped(g[i], u[i], L);
}

/* Elementwise scale-and-quantize of y by the scale code sf (helper for the
 * tolerance checker: which nibble would a nearby y have produced). */
EXPORT uint8_t quantize_element_with_scale(float y, uint8_t sf)
{
    float d = fp8_e4m3_to_float32(sf);
    float s = (d == 0.0f) ? copysignf(0.0f, y) : y / d;
    return quantize_e2m1_nibble(s);
}

/* Elementwise forms of the two rounding primitives (for exhaustive sweeps). */
EXPORT void fp8_e4m3_from_float32_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = fp8_e4m3_from_float32(v[i]);
}

EXPORT void quantize_e2m1_nibble_array(const float *s, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = quantize_e2m1_nibble(s[i]);
}

/* ------------------------------------------------------------------------
 * Extensions of the step (the pages pass these without defining them; each
 * definition below is a READING):
 *  - two-level NVFP4 [P2] (quantize_activation_nvfp4 with a global_scale,
 *    "l2_global_scale" passed to the epilogue): the FP32 global scale gs
 *    multiplies every value before the block quantization, v = fl(y * gs);
 *    dequantization divides by it;
 *  - the pages' own two-kernel flow [AU]: the L1 epilogue stores the SwiGLU
 *    as BF16, so y is rounded to BF16 before quantizing ("compat" mode), and
 *    the compact plan writes that BF16 tensor [rows, I] for a separate
 *    quantize-only pass;
 *  - padded per-expert output [AU] ("padded_activated_fp4"): the rows of
 *    segment e land at output rows out_offsets[e] + (r - offsets[e]);
 *  - dequantization, the consumer's view: value = e2m1 * e4m3 / gs, rounded
 *    to BF16.
 * ------------------------------------------------------------------------ */

/* fp32 -> BF16 value, round to nearest even (finite inputs). */
EXPORT float bf16_round(float v)
{
    uint32_t b = f32_bits(v);
    uint32_t lsb = (b >> 16) & 1u;
    b = (b + 0x7fffu + lsb) & 0xffff0000u;
    return bits_f32(b);
}

EXPORT int quantize_nvfp4_scaled(const uint16_t *x, int64_t rows, int64_t K, float gs,
                                 uint8_t *packed, uint8_t *sf)
{
    if (rows < 0 || K <= 0 || K % 16 != 0) return -1;
    float y[16];
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < K / 16; b++) {
            for (int i = 0; i < 16; i++) y[i] = bf16_to_float32(x[r * K + 16 * b + i]) * gs;
            quantize_nvfp4_block(y, packed + r * (K / 2) + 8 * b, sf + r * (K / 16) + b);
        }
    return 0;
}

/* The activation value of output column c of input row r, in the given
 * mode: the fp32 SwiGLU, optionally rounded to BF16, times gs. */
static float activation_at(const uint16_t *gu, int64_t I, float L, int64_t r, int64_t c,
                           int round_bf16, float gs)
{
    float y = swiglu_at(gu, I, L, r, c);
    if (round_bf16) y = bf16_round(y);
    return y * gs;
}

/*
 * Fused step with the extensions: rows of segment e (or all rows when
 * num_experts == 0) are quantized; input row r of segment e is written to
 * output row out_offsets[e] + (r - offsets[e]) when out_offsets is given
 * (rows outside [0, out_rows) are skipped), else to row r.
 */
EXPORT int swiglu_quantize_nvfp4_ex(const uint16_t *gu, int64_t rows, int64_t I, float L,
                                    const int32_t *offsets, int32_t num_experts,
                                    const int32_t *out_offsets, int64_t out_rows,
                                    float gs, int round_bf16, uint8_t *packed, uint8_t *sf)
{
    if (rows < 0 || I <= 0 || I % 16 != 0) return -1;
    float y[16];
    int32_t nseg = num_experts > 0 ? num_experts : 1;
    for (int32_t e = 0; e < nseg; e++) {
        int64_t r0 = num_experts > 0 ? offsets[e] : 0;
        int64_t r1 = num_experts > 0 ? offsets[e + 1] : rows;
        for (int64_t r = r0; r < r1; r++) {
            if (r < 0 || r >= rows) continue;
            int64_t ro = r;
            if (num_experts > 0 && out_offsets != NULL) {
                ro = out_offsets[e] + (r - r0);
                if (ro < 0 || ro >= out_rows) continue;
            }
            for (int64_t b = 0; b < I / 16; b++) {
                for (int i = 0; i < 16; i++) y[i] = activation_at(gu, I, L, r, 16 * b + i, round_bf16, gs);
                quantize_nvfp4_block(y, packed + ro * (I / 2) + 8 * b, sf + ro * (I / 16) + b);
            }
        }
    }
    return 0;
}

/* Compact writer: the BF16-rounded SwiGLU of the rows of the segments (or of
 * all rows), out_bf16 [rows, I] as BF16 bit patterns. */
EXPORT int swiglu_bf16(const uint16_t *gu, int64_t rows, int64_t I, float L,
                       const int32_t *offsets, int32_t num_experts, uint16_t *out_bf16)
{
    if (rows < 0 || I <= 0 || I % 16 != 0) return -1;
    int32_t nseg = num_experts > 0 ? num_experts : 1;
    for (int32_t e = 0; e < nseg; e++) {
        int64_t r0 = num_experts > 0 ? offsets[e] : 0;
        int64_t r1 = num_experts > 0 ? offsets[e + 1] : rows;
        for (int64_t r = r0; r < r1; r++) {
            if (r < 0 || r >= rows) continue;
            for (int64_t c = 0; c < I; c++)
                out_bf16[r * I + c] = (uint16_t)(f32_bits(bf16_round(swiglu_at(gu, I, L, r, c))) >> 16);
        }
    }
    return 0;
}

/* Dequantization: out_bf16 [rows, K] = RN_bf16((e2m1 value * e4m3 value) / gs). */
EXPORT int dequantize_nvfp4(const uint8_t *packed, const uint8_t *sf, int64_t rows, int64_t K,
                            float gs, uint16_t *out_bf16)
{
    if (rows < 0 || K <= 0 || K % 16 != 0) return -1;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < K; c++) {
            uint8_t byte = packed[r * (K / 2) + c / 2];
            uint8_t nib = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
            float d = fp8_e4m3_to_float32(sf[r * (K / 16) + c / 16]);
            float v = (e2m1_nibble_to_float32(nib) * d) / gs;
            out_bf16[r * K + c] = (uint16_t)(f32_bits(bf16_round(v)) >> 16);
        }
    return 0;
}

/* ---------------------------------------------------------------------------
 * The step fused into the L1 GEMM's epilogue ("2026-05-28 Status", priority
 * 3; "NVFP4-1.1 Approach, Part 2", the TMEM -> registers -> FP4 plan): the
 * GEMM's accumulators gu are real numbers (the test computes them exactly
 * enough in double precision with a library matmul); the clamped SwiGLU is
 * applied to them and rounded once to fp32, and the fp32 values are then
 * quantized block by block exactly as quantize_nvfp4_block defines.
 * ------------------------------------------------------------------------- */

/* silu(min(g, L)) * clamp(u, -L, L) of double inputs, rounded once to fp32. */
EXPORT float swiglu_clamped_f64(double g, double u, float L)
{
    double a = fmin(g, (double)L);
    double b = fmin(fmax(u, -(double)L), (double)L);
    double y = a / (1.0 + exp(-a)) * b;
    return (float)y;
}

EXPORT void swiglu_clamped_f64_array(const double *g, const double *u, int64_t n, float L, float *y)
{
    for (int64_t i = 0; i < n; i++) y[i] = swiglu_clamped_f64(g[i], u[i], L);
}

/* fp32 values y [rows, K] -> packed [rows, K/2], sf [rows, K/16]. */
EXPORT int quantize_nvfp4_f32(const float *y, int64_t rows, int64_t K, uint8_t *packed, uint8_t *sf)
{
    if (rows < 0 || K <= 0 || K % 16 != 0) return -1;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < K / 16; b++)
            quantize_nvfp4_block(y + r * K + 16 * b, packed + r * (K / 2) + 8 * b, sf + r * (K / 16) + b);
    return 0;
}
