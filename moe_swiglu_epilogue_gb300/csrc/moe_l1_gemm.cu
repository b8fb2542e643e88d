// GB300 (sm_103a) MoE L1 GEMM with the activation step in its epilogue:
// for every expert segment e (rows [offsets[e], offsets[e+1]) of x),
//   gu = x_e @ w1[e]^T   (BF16 operands, fp32 accumulators in TMEM)
// and the epilogue turns the accumulators straight into NVFP4: clamped
// SwiGLU of the [gate x8, up x8] column groups, then the block scale and
// nibbles, without writing gu anywhere.
//
// From the nvfp4-megamoe-kernel pages: "NVFP4-1.1 Approach Update" (the L1
// GEMM's epilogue writes the interleaved [gate*8, swiglu*8, ...] columns that
// a separate kernel then quantizes); "2026-05-28 Status" (priority 3: fuse
// the amax and FP4 pack into the L1 -> L2 path); "NVFP4-1.1 Approach, Part 2"
// (the planned epilogue: TMEM -> registers -> FP4 pack -> global memory, 16
// SwiGLU values -> 8 packed bytes + 1 scale byte per block).
//
// Design:
//   * Persistent grid, one CTA per SM, 192 threads in three roles: warp 0
//     issues TMA loads of 128 x 64 (x) and 256 x 64 (w1) BF16 tiles into a
//     4-stage shared-memory ring (128-byte swizzle, K-major); warp 1 owns the
//     TMEM allocation and issues tcgen05.mma (kind::f16, M = 128, N = 256,
//     K = 16) into one of two 256-column fp32 accumulators; warps 2-5 read
//     an accumulator back with tcgen05.ld (warp w sees TMEM lanes
//     32 (w % 4) .. + 31, one tile row per thread) while the next tile's
//     MMAs run into the other one.
//   * Tiles never straddle experts: expert e has ceil(rows_e / 128) M-tiles
//     times 2I / 256 N-tiles; tiles are ordered expert, N-tile, M-tile, so
//     the M-tiles sharing a weight slice run side by side and the N-tiles
//     sharing an expert's rows stay in L2. Rows past a segment's end are
//     computed but not stored; rows past the tensor are zero-filled by TMA.
//   * Epilogue per thread and output block (32 accumulator columns = 8 gate,
//     8 up, 8 gate, 8 up): SwiGLU of the fp32 accumulators in fast fp32
//     (packed fp32x2), then the exact NVFP4 quantization of those values
//     (correctly rounded amax / 6, E4M3 cast, correctly rounded quotients,
//     half steps, E2M1 cast). The 8 blocks of a tile row are stored as 64
//     packed bytes and 8 scale bytes.
//   * Every wait on an mbarrier is bounded (about a second); on expiry the
//     kernel records a status code and every role stops at its next wait.
//     Before the TMEM is released and the CTA exits, the producer waits for
//     the TMA loads it issued to land and the MMA issuer for the MMAs it
//     issued to complete (both bounded), so no asynchronous write into this
//     CTA's shared memory or TMEM outlives it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "moe_nvfp4.h"
#include "nvfp4_device.cuh"

namespace {

using namespace nvfp4dev;

constexpr int kBM = 128;                     // rows per tile (TMEM lanes)
constexpr int kBN = 256;                     // accumulator columns per tile (128 outputs)
constexpr int kBK = 64;                      // K per stage: one 128-byte swizzle row of BF16
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;
constexpr int kMaxGemmExperts = 2048;
constexpr uint32_t kStageA = kBM * kBK * 2;
constexpr uint32_t kStageB = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr uint32_t kTmemCols = 2 * kBN;      // two accumulators
constexpr long long kWaitCycles = 2000000000LL;   // about a second
constexpr int kMaxGemmDevices = 64;

// tcgen05 instruction descriptor, kind::f16: fp32 D (bits 4-5 = 1), BF16 A
// and B (bits 7-9, 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at 24.
constexpr uint32_t kInstrDesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                (static_cast<uint32_t>(kBN >> 3) << 17) |
                                (static_cast<uint32_t>(kBM >> 4) << 24);

struct GemmArgs {
    const int32_t* offsets;    // [E+1] device
    int E;
    int64_t rows;
    int64_t H;                 // K of the GEMM
    int64_t I;                 // outputs per row (2I accumulator columns)
    int nt;                    // N-tiles per expert: 2I / 256
    float L;
    uint8_t* packed;           // [rows, I/2]
    uint8_t* sf;               // [rows, I/16]
    float* acc;                // [rows, 2I] (accumulator diagnostic) or null
    uint16_t* out_bf16;        // BF16 gu [rows, 2I] or SwiGLU [rows, I] outputs
    int32_t* status;           // optional: nonzero after a wait expired
    long long wait_cycles;     // limit of every mbarrier wait
    int selftest;              // diagnostic: 1 the producer issues nothing; 2 the epilogue
                               // never releases an accumulator (one CTA runs every tile)
};

// What the epilogue writes: the NVFP4 activations (the fused step), the
// fp32 accumulators (diagnostic), or the BF16 tensors of the unfused flows
// the pages describe: gu itself ([gate x8, up x8] columns, 2I per row) or
// the compact SwiGLU (I per row).
enum GemmOut : int { kOutNvfp4 = 0, kOutAcc = 1, kOutGuBf16 = 2, kOutSwigluBf16 = 3 };

struct SharedState {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int tile_prefix[kMaxGemmExperts + 1];    // M-tiles before expert e
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Waits for the phase of the given parity; false once the CTA aborted or
// the wait expired (which records `code` and aborts the CTA). Codes: 1 the
// producer waiting for a free stage, 2 the MMA issuer for a free
// accumulator, 3 the MMA issuer for a loaded stage, 4 the epilogue for a
// finished accumulator.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* abort,
                                          int32_t* status, int code, long long limit) {
    const long long t0 = clock64();
    for (uint32_t n = 0;; n++) {
        if (mbar_try(bar, parity)) return true;
        if ((n & 31) == 31) {
            if (*reinterpret_cast<volatile int*>(abort)) return false;
            if (clock64() - t0 > limit) {
                *reinterpret_cast<volatile int*>(abort) = 1;
                if (status != nullptr) atomicExch(status, code);
                return false;
            }
        }
    }
}

// Waits, bounded, for the phase of the given parity whatever the abort flag
// says: the drain after an abort. False if the limit passed first.
__device__ __forceinline__ bool mbar_wait_quiet(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    for (uint32_t n = 0;; n++) {
        if (mbar_try(bar, parity)) return true;
        if ((n & 31) == 31 && clock64() - t0 > limit) return false;
    }
}

// Status code of a drain wait that expired (recorded only if no other code
// was): an issued TMA load or MMA did not complete.
constexpr int kDrainExpired = 8;

__device__ __forceinline__ void drain_failed(int32_t* status) {
    if (status != nullptr) atomicCAS(status, 0, kDrainExpired);
}

// The producer's drain: the last `stages` of the `issued` stage loads (a
// stage's previous load completed before its next was issued) have landed.
// Only the producer arrives on a full barrier, so a completed phase stays
// completed.
__device__ __forceinline__ void drain_loads(const uint64_t* full, int stages, uint32_t issued, long long limit,
                                            int32_t* status) {
    for (uint32_t j = issued > static_cast<uint32_t>(stages) ? issued - stages : 0u; j < issued; j++)
        if (!mbar_wait_quiet(smem_u32(&full[j % stages]), (j / stages) & 1u, limit)) drain_failed(status);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// 2-D TMA tile load (x = innermost coordinate, in elements) completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: start address >> 4, leading offset 16 B (unused for this
// layout), 1024 B between 8-row groups, descriptor version 1, swizzle mode 2.
// Advancing K by 16 BF16 elements adds 32 bytes (2 in the address field).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(const void* tile) {
    return static_cast<uint64_t>((smem_u32(tile) >> 4) & 0x3FFFu) | (1ull << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(kInstrDesc), "r"(accumulate) : "memory");
}

// The mbarrier receives one arrival when every MMA issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// The MMA issuer's drain: every MMA it issued has completed (one commit to
// a barrier used for nothing else, then a bounded wait on it).
__device__ __forceinline__ void drain_mmas(uint64_t* drain, long long limit, int32_t* status) {
    mma_commit(drain);
    if (!mbar_wait_quiet(smem_u32(drain), 0u, limit)) drain_failed(status);
}

__device__ __forceinline__ void tmem_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr) : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Rows [begin, end) of expert e, offsets clamped into [0, rows].
__device__ __forceinline__ void expert_rows(const GemmArgs& G, int e, int64_t& begin, int64_t& end) {
    int64_t b = __ldg(G.offsets + e), f = __ldg(G.offsets + e + 1);
    b = b < 0 ? 0 : (b > G.rows ? G.rows : b);
    f = f < b ? b : (f > G.rows ? G.rows : f);
    begin = b;
    end = f;
}

struct TileCoords {
    int e, nt, mt;
    int64_t row0, row_end;     // first row of the tile, end of the expert's rows
};

// Tile t -> (expert, N-tile, M-tile): the last expert whose first tile is
// <= t (empty experts share their successor's start, so it is non-empty).
__device__ __forceinline__ TileCoords tile_coords(const GemmArgs& G, const int* tile_prefix, int64_t t) {
    int lo = 0, hi = G.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(tile_prefix[mid]) * G.nt <= t) lo = mid; else hi = mid - 1;
    }
    TileCoords c;
    c.e = lo;
    const int mtiles = tile_prefix[lo + 1] - tile_prefix[lo];
    const int64_t r = t - static_cast<int64_t>(tile_prefix[lo]) * G.nt;
    c.nt = static_cast<int>(r / mtiles);
    c.mt = static_cast<int>(r - static_cast<int64_t>(c.nt) * mtiles);
    int64_t begin, end;
    expert_rows(G, lo, begin, end);
    c.row0 = begin + static_cast<int64_t>(kBM) * c.mt;
    c.row_end = end;
    return c;
}

// M-tiles per expert, prefix-summed by one warp: tile_prefix[e] = M-tiles
// before expert e, tile_prefix[E] = all of them.
__device__ __forceinline__ void tile_prefix_sum(const GemmArgs& G, int* tile_prefix, int lane) {
    int carry = 0;
    for (int e0 = 0; e0 < G.E; e0 += 32) {
        const int e = e0 + lane;
        int m = 0;
        if (e < G.E) {
            int64_t b, f;
            expert_rows(G, e, b, f);
            m = static_cast<int>((f - b + kBM - 1) / kBM);
        }
        int incl = m;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(kFullMask, incl, d);
            if (lane >= d) incl += v;
        }
        if (e < G.E) tile_prefix[e] = carry + incl - m;
        carry += __shfl_sync(kFullMask, incl, 31);
    }
    if (lane == 0) tile_prefix[G.E] = carry;
}

// SwiGLU of one output block (16 outputs) from its 32 accumulator columns.
__device__ __forceinline__ void swiglu_block(const uint32_t* r, float L, float* y) {
#pragma unroll
    for (int half = 0; half < 2; half++) {
#pragma unroll
        for (int p = 0; p < 4; p++) {
            const int gi = 16 * half + 2 * p;           // gate columns; ups 8 further on
            const float2 g = make_float2(fminf(__uint_as_float(r[gi]), L),
                                         fminf(__uint_as_float(r[gi + 1]), L));
            const float2 u = make_float2(fminf(fmaxf(__uint_as_float(r[gi + 8]), -L), L),
                                         fminf(fmaxf(__uint_as_float(r[gi + 9]), -L), L));
            const float2 v = silu_times_fast2(g, u);
            y[8 * half + 2 * p] = v.x;
            y[8 * half + 2 * p + 1] = v.y;
        }
    }
}

// ... then its exact NVFP4 quantization.
__device__ __forceinline__ uint32_t epilogue_block(const uint32_t* r, float L, uint32_t& lo, uint32_t& hi) {
    float y[16];
    swiglu_block(r, L, y);
    return quantize16_exact<true, true>(y, lo, hi);
}

// The epilogue of one tile row (one thread): reads the row's 256
// accumulator columns from TMEM (at taddr) and stores what kOut asks for.
// Every lane of the warp calls this together (tcgen05.ld is collective).
template <int kOut>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& G, const TileCoords& c, int64_t row, bool valid,
                                              uint32_t taddr) {
    if (kOut == kOutGuBf16 || kOut == kOutSwigluBf16) {
#pragma unroll 1
        for (int ob = 0; ob < kBN / 32; ob++) {
            uint32_t r[32];
            tmem_load32(taddr + 32 * ob, r);
            if (kOut == kOutGuBf16) {                       // 32 columns of gu
                uint32_t h[16];
#pragma unroll
                for (int j = 0; j < 16; j++)
                    h[j] = bf16x2_rn(__uint_as_float(r[2 * j + 1]), __uint_as_float(r[2 * j]));
                if (valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(G.out_bf16 + row * 2 * G.I + kBN * c.nt + 32 * ob);
#pragma unroll
                    for (int j = 0; j < 4; j++) d4[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
                }
            } else {                                        // 16 SwiGLU outputs
                float y[16];
                swiglu_block(r, G.L, y);
                uint32_t h[8];
#pragma unroll
                for (int j = 0; j < 8; j++) h[j] = bf16x2_rn(y[2 * j + 1], y[2 * j]);
                if (valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(G.out_bf16 + row * G.I + (kBN / 2) * c.nt + 16 * ob);
                    d4[0] = make_uint4(h[0], h[1], h[2], h[3]);
                    d4[1] = make_uint4(h[4], h[5], h[6], h[7]);
                }
            }
        }
    } else if (kOut == kOutAcc) {
        float* dst = G.acc + row * 2 * G.I + static_cast<int64_t>(kBN) * c.nt;
#pragma unroll 1
        for (int ob = 0; ob < kBN / 32; ob++) {
            uint32_t r[32];
            tmem_load32(taddr + 32 * ob, r);
            if (valid) {
                float4* d4 = reinterpret_cast<float4*>(dst + 32 * ob);
#pragma unroll
                for (int j = 0; j < 8; j++)
                    d4[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
        }
    } else {
        uint32_t pk[16], codes[2] = {0u, 0u};
#pragma unroll
        for (int ob = 0; ob < kBN / 32; ob++) {
            uint32_t r[32];
            tmem_load32(taddr + 32 * ob, r);
            const uint32_t code = epilogue_block(r, G.L, pk[2 * ob], pk[2 * ob + 1]);
            codes[ob >> 2] |= code << (8 * (ob & 3));
        }
        if (valid) {
            uint4* dp = reinterpret_cast<uint4*>(G.packed + row * (G.I / 2) + 64 * c.nt);
#pragma unroll
            for (int j = 0; j < 4; j++) dp[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            *reinterpret_cast<uint2*>(G.sf + row * (G.I / 16) + 8 * c.nt) = make_uint2(codes[0], codes[1]);
        }
    }
}

template <int kOut>
__global__ void __launch_bounds__(kGemmThreads, 1)
l1_gemm_swiglu_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const GemmArgs G) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    SharedState& S = *reinterpret_cast<SharedState*>(base + kStages * kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&S.tmem_base)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) { mbar_init(&S.full[s], 1); mbar_init(&S.empty[s], 1); }
        for (int b = 0; b < 2; b++) { mbar_init(&S.acc_full[b], 1); mbar_init(&S.acc_empty[b], 128); }
        mbar_init(&S.drain, 1);
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    wait_for_preceding_grid();
    if (warp == 2) tile_prefix_sum(G, S.tile_prefix, lane);
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    allow_next_grid_launch();

    const int64_t total = static_cast<int64_t>(S.tile_prefix[G.E]) * G.nt;
    const int nkb = static_cast<int>(G.H / kBK);

    if (warp == 0) {
        if (lane == 0 && G.selftest != 1) {                         // TMA producer
            uint32_t it = 0;                                        // stage loads issued
            for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
                const TileCoords c = tile_coords(G, S.tile_prefix, t);
                const int y_w = static_cast<int>(static_cast<int64_t>(c.e) * 2 * G.I) + kBN * c.nt;
                for (int kb = 0; kb < nkb; kb++, it++) {
                    const int s = static_cast<int>(it % kStages);
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&S.empty[s]), ph ^ 1u, &S.abort, G.status, 1, G.wait_cycles))
                        goto producer_end;
                    uint8_t* st = base + s * kStageBytes;
                    mbar_expect_tx(&S.full[s], kStageBytes);
                    tma_load_2d(st, &tmX, kb * kBK, static_cast<int>(c.row0), &S.full[s]);
                    tma_load_2d(st + kStageA, &tmW, kb * kBK, y_w, &S.full[s]);
                }
            }
        producer_end:
            drain_loads(S.full, kStages, it, G.wait_cycles, G.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {                                            // MMA issuer
            uint32_t it = 0, local = 0;
            for (int64_t t = blockIdx.x; t < total; t += gridDim.x, local++) {
                const int b = static_cast<int>(local & 1u);
                const uint32_t aph = (local >> 1) & 1u;
                if (!mbar_wait(smem_u32(&S.acc_empty[b]), aph ^ 1u, &S.abort, G.status, 2, G.wait_cycles))
                    goto issuer_end;
                tmem_fence_after();
                const uint32_t d_tmem = S.tmem_base + static_cast<uint32_t>(b * kBN);
                for (int kb = 0; kb < nkb; kb++, it++) {
                    const int s = static_cast<int>(it % kStages);
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&S.full[s]), ph, &S.abort, G.status, 3, G.wait_cycles)) goto issuer_end;
                    tmem_fence_after();
                    const uint8_t* st = base + s * kStageBytes;
                    const uint64_t da = sw128_kmajor_desc(st), db = sw128_kmajor_desc(st + kStageA);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; kk++)
                        mma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, (kb | kk) != 0 ? 1u : 0u);
                    mma_commit(&S.empty[s]);                        // frees the stage when read
                }
                mma_commit(&S.acc_full[b]);                         // accumulator complete
            }
        issuer_end:
            drain_mmas(&S.drain, G.wait_cycles, G.status);
        }
    } else if (G.selftest != 2) {                                   // epilogue, warps 2-5
        const int quarter = warp & 3;
        const int trow = 32 * quarter + lane;
        uint32_t local = 0;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x, local++) {
            const int b = static_cast<int>(local & 1u);
            const uint32_t aph = (local >> 1) & 1u;
            // tcgen05.ld is warp-collective: the warp goes on only if every
            // lane saw the accumulator complete
            const bool ok = mbar_wait(smem_u32(&S.acc_full[b]), aph, &S.abort, G.status, 4, G.wait_cycles);
            if (!__all_sync(kFullMask, ok)) break;
            tmem_fence_after();
            const TileCoords c = tile_coords(G, S.tile_prefix, t);
            const int64_t row = c.row0 + trow;
            const bool valid = row < c.row_end;
            const uint32_t taddr = S.tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) +
                                   static_cast<uint32_t>(b * kBN);
            epilogue_tile<kOut>(G, c, row, valid, taddr);
            tmem_fence_before();
            mbar_arrive(&S.acc_empty[b]);
        }
    }
    tmem_fence_before();
    __syncthreads();
    if (warp == 1) {
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(S.tmem_base), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// The same GEMM with NVFP4 weights (BF16 activations). The weights arrive as
// packed E2M1 nibbles [E, 2I, H/2] with one E4M3 scale per 16 along K
// [E, 2I, H/16] -- the layout moe_nvfp4_quantize writes -- so a weight tile
// costs 0.5625 bytes per element in HBM instead of 2. Eight expander warps
// turn each stage in shared memory into the BF16 tile the MMA reads, in the
// layout a 128-byte-swizzled TMA load would give; e2m1 * e4m3 has at most 6
// significant bits, so the expansion is exact, and the result equals the
// BF16 GEMM on the dequantized weights bit for bit. The latency of the
// expansion pipeline (nibbles from shared memory, BF16 back into it, then
// the MMA) sets the pace, not HBM: the kernel saves weight memory and HBM
// traffic, not time, against the BF16-weight kernel.
// ---------------------------------------------------------------------------

constexpr int kW4RawStages = 4;                          // x tile + packed weight tile
constexpr int kW4BStages = 3;                            // expanded BF16 weight tiles
constexpr uint32_t kW4FpBytes = kBN * kBK / 2;           // 8 KB of nibbles per stage
constexpr uint32_t kW4RawBytes = kStageA + kW4FpBytes;   // 24 KB
constexpr uint32_t kW4ScaleBytes = kBN * 16;             // scales of 4 stages: 16 per row
constexpr int kW4ScaleSlots = 2;
// a scale slot serves 4 stages and is reloaded 4 * kW4ScaleSlots stages
// later, by the producer once the raw stage kW4RawStages back is free: its
// last reader must be at least that old
static_assert(kW4RawStages <= 4 * kW4ScaleSlots - 3, "a scale slot outlives its readers");
constexpr int kW4ConvThreads = 256;
constexpr int kW4Threads = kGemmThreads + kW4ConvThreads;   // warps 6-13 expand the weights

struct W4Shared {
    uint64_t full[kW4RawStages];       // x + nibbles (+ scales every 4th stage) landed
    uint64_t empty[kW4RawStages];      // the MMA done with x, the expanders with the nibbles
    uint64_t bready[kW4BStages];       // expanded tile written
    uint64_t bempty[kW4BStages];       // the MMA done with it
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int tile_prefix[kMaxGemmExperts + 1];
};

constexpr size_t kW4Smem = 1024 + static_cast<size_t>(kW4RawStages) * kW4RawBytes +
                           static_cast<size_t>(kW4ScaleSlots) * kW4ScaleBytes +
                           static_cast<size_t>(kW4BStages) * kStageB + sizeof(W4Shared);

static_assert(kW4Smem <= 227 * 1024, "shared memory of one CTA");

// Tiles of this CTA in the grid-stride order.
__device__ __forceinline__ int64_t tiles_of_cta(int64_t total) {
    return total > blockIdx.x ? (total - 1 - blockIdx.x) / gridDim.x + 1 : 0;
}

// One 16-byte piece of a weight row (32 nibbles = two 16-element scale
// blocks) expanded into four 16-byte BF16 chunks of the swizzled tile.
__device__ __forceinline__ void expand_piece(const uint8_t* nibbles, uint32_t scale2, uint8_t* tile, int row,
                                             int half) {
    const uint4 p = *reinterpret_cast<const uint4*>(nibbles);
    const float d0 = e4m3_value(scale2 & 0xFFu), d1 = e4m3_value(scale2 >> 8);
    const uint32_t words[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int w = 0; w < 4; w++) {
        const float d = w < 2 ? d0 : d1;
        const uint32_t h2[4] = {e2m1x2_to_f16x2<0>(words[w]), e2m1x2_to_f16x2<1>(words[w]),
                                e2m1x2_to_f16x2<2>(words[w]), e2m1x2_to_f16x2<3>(words[w])};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float lo = __half2float(__ushort_as_half(static_cast<uint16_t>(h2[k] & 0xFFFFu))) * d;
            const float hi = __half2float(__ushort_as_half(static_cast<uint16_t>(h2[k] >> 16))) * d;
            o[k] = bf16x2_rn(hi, lo);                       // exact: at most 6 significant bits
        }
        const int chunk = 4 * half + w;                     // 8 elements along K
        *reinterpret_cast<uint4*>(tile + row * 128 + ((chunk ^ (row & 7)) << 4)) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int kOut>
__global__ void __launch_bounds__(kW4Threads, 1)
l1_gemm_w4_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmS, const GemmArgs G) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* scale_base = base + kW4RawStages * kW4RawBytes;
    uint8_t* bconv = scale_base + kW4ScaleSlots * kW4ScaleBytes;
    W4Shared& S = *reinterpret_cast<W4Shared*>(bconv + kW4BStages * kStageB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&S.tmem_base)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kW4RawStages; s++) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1 + kW4ConvThreads);
        }
        for (int j = 0; j < kW4BStages; j++) { mbar_init(&S.bready[j], kW4ConvThreads); mbar_init(&S.bempty[j], 1); }
        for (int b = 0; b < 2; b++) { mbar_init(&S.acc_full[b], 1); mbar_init(&S.acc_empty[b], 128); }
        mbar_init(&S.drain, 1);
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    wait_for_preceding_grid();
    if (warp == 2) tile_prefix_sum(G, S.tile_prefix, lane);
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    allow_next_grid_launch();

    const int64_t total = static_cast<int64_t>(S.tile_prefix[G.E]) * G.nt;
    const int nkb = static_cast<int>(G.H / kBK);            // a multiple of 4 (H % 256 == 0)

    if (warp == 0) {
        if (lane == 0 && G.selftest != 1) {                         // TMA producer
            uint32_t it = 0;                                        // stage loads issued
            for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
                const TileCoords c = tile_coords(G, S.tile_prefix, t);
                const int y_w = static_cast<int>(static_cast<int64_t>(c.e) * 2 * G.I) + kBN * c.nt;
                for (int kb = 0; kb < nkb; kb++, it++) {
                    const int s = static_cast<int>(it % kW4RawStages);
                    const uint32_t ph = (it / kW4RawStages) & 1u;
                    if (!mbar_wait(smem_u32(&S.empty[s]), ph ^ 1u, &S.abort, G.status, 1, G.wait_cycles))
                        goto producer_end;
                    uint8_t* st = base + s * kW4RawBytes;
                    const bool scales = (kb & 3) == 0;                // one scale tile per 4 stages
                    mbar_expect_tx(&S.full[s], kW4RawBytes + (scales ? kW4ScaleBytes : 0u));
                    tma_load_2d(st, &tmX, kb * kBK, static_cast<int>(c.row0), &S.full[s]);
                    tma_load_2d(st + kStageA, &tmQ, kb * (kBK / 2), y_w, &S.full[s]);
                    if (scales)
                        tma_load_2d(scale_base + ((it >> 2) % kW4ScaleSlots) * kW4ScaleBytes, &tmS, (kb >> 2) * 16, y_w,
                                    &S.full[s]);
                }
            }
        producer_end:
            drain_loads(S.full, kW4RawStages, it, G.wait_cycles, G.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {                                            // MMA issuer
            uint32_t it = 0, local = 0;
            for (int64_t t = blockIdx.x; t < total; t += gridDim.x, local++) {
                const int b = static_cast<int>(local & 1u);
                const uint32_t aph = (local >> 1) & 1u;
                if (!mbar_wait(smem_u32(&S.acc_empty[b]), aph ^ 1u, &S.abort, G.status, 2, G.wait_cycles))
                    goto issuer_end;
                tmem_fence_after();
                const uint32_t d_tmem = S.tmem_base + static_cast<uint32_t>(b * kBN);
                for (int kb = 0; kb < nkb; kb++, it++) {
                    const int s = static_cast<int>(it % kW4RawStages);
                    const int j = static_cast<int>(it % kW4BStages);
                    if (!mbar_wait(smem_u32(&S.full[s]), (it / kW4RawStages) & 1u, &S.abort, G.status, 3,
                                   G.wait_cycles) ||
                        !mbar_wait(smem_u32(&S.bready[j]), (it / kW4BStages) & 1u, &S.abort, G.status, 5,
                                   G.wait_cycles))
                        goto issuer_end;
                    tmem_fence_after();
                    const uint64_t da = sw128_kmajor_desc(base + s * kW4RawBytes);
                    const uint64_t db = sw128_kmajor_desc(bconv + j * kStageB);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; kk++)
                        mma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, (kb | kk) != 0 ? 1u : 0u);
                    mma_commit(&S.empty[s]);                        // x tile read
                    mma_commit(&S.bempty[j]);                       // expanded tile read
                }
                mma_commit(&S.acc_full[b]);
            }
        issuer_end:
            drain_mmas(&S.drain, G.wait_cycles, G.status);
        }
    } else if (warp < 6) {                                          // epilogue, warps 2-5
        const int quarter = warp & 3;
        const int trow = 32 * quarter + lane;
        uint32_t local = 0;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x, local++) {
            const int b = static_cast<int>(local & 1u);
            const uint32_t aph = (local >> 1) & 1u;
            const bool ok = mbar_wait(smem_u32(&S.acc_full[b]), aph, &S.abort, G.status, 4, G.wait_cycles);
            if (!__all_sync(kFullMask, ok)) break;
            tmem_fence_after();
            const TileCoords c = tile_coords(G, S.tile_prefix, t);
            const int64_t row = c.row0 + trow;
            const uint32_t taddr = S.tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) +
                                   static_cast<uint32_t>(b * kBN);
            epilogue_tile<kOut>(G, c, row, row < c.row_end, taddr);
            tmem_fence_before();
            mbar_arrive(&S.acc_empty[b]);
        }
    } else {                                                        // weight expanders, warps 6-13
        const int ct = threadIdx.x - kGemmThreads;
        const int64_t iters = tiles_of_cta(total) * nkb;
        for (int64_t it = 0; it < iters; it++) {
            const int s = static_cast<int>(it % kW4RawStages);
            const int j = static_cast<int>(it % kW4BStages);
            if (!mbar_wait(smem_u32(&S.full[s]), static_cast<uint32_t>(it / kW4RawStages) & 1u, &S.abort, G.status,
                           6, G.wait_cycles) ||
                !mbar_wait(smem_u32(&S.bempty[j]), (static_cast<uint32_t>(it / kW4BStages) & 1u) ^ 1u, &S.abort,
                           G.status, 7, G.wait_cycles))
                break;
            const uint8_t* nib = base + s * kW4RawBytes + kStageA;              // row r at 32 r
            const uint8_t* sc = scale_base + ((it >> 2) % kW4ScaleSlots) * kW4ScaleBytes + (it & 3) * 4;   // row r at 16 r
            uint8_t* tile = bconv + j * kStageB;
#pragma unroll
            for (int i = 0; i < (kBN * 2) / kW4ConvThreads; i++) {
                const int q = ct + kW4ConvThreads * i;                      // consecutive 16-byte pieces
                const int row = q >> 1, half = q & 1;
                const uint32_t scale2 = *reinterpret_cast<const uint16_t*>(sc + row * 16 + 2 * half);
                expand_piece(nib + q * 16, scale2, tile, row, half);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMA
            mbar_arrive(&S.bready[j]);
            mbar_arrive(&S.empty[s]);
        }
    }
    tmem_fence_before();
    __syncthreads();
    if (warp == 1) {
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(S.tmem_base), "r"(kTmemCols) : "memory");
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The CUDA driver's tensor-map encoder, fetched once through the runtime.
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [outer, inner] row-major tensor -> tensor map with a box of box_inner x
// box_rows elements; rows past `outer` read as zeros.
bool make_map(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, int64_t inner,
              int64_t outer, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 K-major operand tiles of 64 x box_rows with the 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, uint32_t box_rows) {
    return make_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, kBK, box_rows,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

constexpr size_t kGemmSmem = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(SharedState);

struct GemmDevice {
    bool ready = false;
    int sms = 0;
};
GemmDevice g_gemm_dev[kMaxGemmDevices];
std::mutex g_gemm_mu;

int gemm_device(int& sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxGemmDevices) return MOE_NVFP4_ELAUNCH;
    std::lock_guard<std::mutex> lock(g_gemm_mu);
    GemmDevice& d = g_gemm_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaFuncSetAttribute(l1_gemm_swiglu_kernel<kOutNvfp4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemmSmem)) != cudaSuccess ||
            cudaFuncSetAttribute(l1_gemm_swiglu_kernel<kOutAcc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemmSmem)) != cudaSuccess ||
            cudaFuncSetAttribute(l1_gemm_swiglu_kernel<kOutGuBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemmSmem)) != cudaSuccess ||
            cudaFuncSetAttribute(l1_gemm_swiglu_kernel<kOutSwigluBf16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemmSmem)) != cudaSuccess ||
            cudaFuncSetAttribute(l1_gemm_w4_kernel<kOutNvfp4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kW4Smem)) != cudaSuccess ||
            cudaFuncSetAttribute(l1_gemm_w4_kernel<kOutAcc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kW4Smem)) != cudaSuccess)
            return MOE_NVFP4_ELAUNCH;
        d.ready = true;
    }
    sms = d.sms;
    return MOE_NVFP4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int launch_gemm(const uint16_t* x, const uint16_t* w1, int64_t rows, int64_t H, int64_t I, float L,
                const int32_t* offsets, int32_t E, int mode, uint8_t* packed, uint8_t* sf, void* out,
                int32_t* status, cudaStream_t stream, long long wait_cycles = kWaitCycles,
                int selftest = 0) {
    if (rows < 0 || rows > (int64_t{1} << 31) - 2 * kBM) return MOE_NVFP4_ESIZE;
    if (H <= 0 || H % kBK != 0 || I <= 0 || I % (kBN / 2) != 0) return MOE_NVFP4_EWIDTH;
    const bool uses_L = mode == kOutNvfp4 || mode == kOutSwigluBf16;
    if (uses_L && !(L > 0.0f && L <= 0x1p64f)) return MOE_NVFP4_ECLAMP;
    if (E < 1 || E > kMaxGemmExperts || offsets == nullptr) return MOE_NVFP4_EOFFSETS;
    if (static_cast<int64_t>(E) * 2 * I > (int64_t{1} << 31) - 1 || H > (int64_t{1} << 31) - 1)
        return MOE_NVFP4_ESIZE;
    if (rows > 0 && 2 * I > INT64_MAX / 4 / rows) return MOE_NVFP4_ESIZE;
    if (rows == 0) return MOE_NVFP4_OK;
    if (x == nullptr || w1 == nullptr) return MOE_NVFP4_ENULL;
    if (mode == kOutNvfp4 ? (packed == nullptr || sf == nullptr) : out == nullptr) return MOE_NVFP4_ENULL;
    if (!aligned16(x) || !aligned16(w1) ||
        (mode == kOutNvfp4 ? (!aligned16(packed) || !aligned16(sf)) : !aligned16(out)) ||
        !aligned4(offsets) || !aligned4(status))
        return MOE_NVFP4_EALIGN;
    int sms = 0;
    int rc = gemm_device(sms);
    if (rc != MOE_NVFP4_OK) return rc;
    CUtensorMap tmX, tmW;
    if (!make_map(&tmX, x, H, rows, kBM) || !make_map(&tmW, w1, H, static_cast<int64_t>(E) * 2 * I, kBN))
        return MOE_NVFP4_ELAUNCH;
    GemmArgs G;
    G.offsets = offsets; G.E = E; G.rows = rows; G.H = H; G.I = I;
    G.nt = static_cast<int>(2 * I / kBN); G.L = uses_L ? L : 1.0f;
    G.packed = packed; G.sf = sf; G.status = status;
    G.wait_cycles = wait_cycles; G.selftest = selftest;
    G.acc = mode == kOutAcc ? static_cast<float*>(out) : nullptr;
    G.out_bf16 = (mode == kOutGuBf16 || mode == kOutSwigluBf16) ? static_cast<uint16_t*>(out) : nullptr;
    cudaLaunchConfig_t cfg = {};
    // the self-test that never releases an accumulator runs every tile on
    // one CTA, so that its producer and MMA issuer have work in flight
    cfg.gridDim = dim3(static_cast<unsigned>(selftest == 2 ? 1 : sms));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kGemmSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    switch (mode) {
        case kOutNvfp4: e = cudaLaunchKernelEx(&cfg, l1_gemm_swiglu_kernel<kOutNvfp4>, tmX, tmW, G); break;
        case kOutAcc: e = cudaLaunchKernelEx(&cfg, l1_gemm_swiglu_kernel<kOutAcc>, tmX, tmW, G); break;
        case kOutGuBf16: e = cudaLaunchKernelEx(&cfg, l1_gemm_swiglu_kernel<kOutGuBf16>, tmX, tmW, G); break;
        default: e = cudaLaunchKernelEx(&cfg, l1_gemm_swiglu_kernel<kOutSwigluBf16>, tmX, tmW, G); break;
    }
    return e == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

// The NVFP4-weight GEMM: the nibbles as 32 x 256-byte boxes, the scales as
// 16 x 256-byte boxes (4 stages of K), both without swizzle.
int launch_gemm_w4(const uint16_t* x, const uint8_t* wq, const uint8_t* ws, int64_t rows, int64_t H, int64_t I,
                   float L, const int32_t* offsets, int32_t E, int mode, uint8_t* packed, uint8_t* sf,
                   float* acc, int32_t* status, cudaStream_t stream) {
    if (rows < 0 || rows > (int64_t{1} << 31) - 2 * kBM) return MOE_NVFP4_ESIZE;
    if (H <= 0 || H % (4 * kBK) != 0 || I <= 0 || I % (kBN / 2) != 0) return MOE_NVFP4_EWIDTH;
    if (mode == kOutNvfp4 && !(L > 0.0f && L <= 0x1p64f)) return MOE_NVFP4_ECLAMP;
    if (E < 1 || E > kMaxGemmExperts || offsets == nullptr) return MOE_NVFP4_EOFFSETS;
    if (static_cast<int64_t>(E) * 2 * I > (int64_t{1} << 31) - 1 || H > (int64_t{1} << 31) - 1)
        return MOE_NVFP4_ESIZE;
    if (rows > 0 && 2 * I > INT64_MAX / 4 / rows) return MOE_NVFP4_ESIZE;
    if (rows == 0) return MOE_NVFP4_OK;
    if (x == nullptr || wq == nullptr || ws == nullptr) return MOE_NVFP4_ENULL;
    if (mode == kOutNvfp4 ? (packed == nullptr || sf == nullptr) : acc == nullptr) return MOE_NVFP4_ENULL;
    if (!aligned16(x) || !aligned16(wq) || !aligned16(ws) ||
        (mode == kOutNvfp4 ? (!aligned16(packed) || !aligned16(sf)) : !aligned16(acc)) ||
        !aligned4(offsets) || !aligned4(status))
        return MOE_NVFP4_EALIGN;
    int sms = 0;
    int rc = gemm_device(sms);
    if (rc != MOE_NVFP4_OK) return rc;
    const int64_t wrows = static_cast<int64_t>(E) * 2 * I;
    CUtensorMap tmX, tmQ, tmS;
    if (!make_map(&tmX, x, H, rows, kBM) ||
        !make_map(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wq, H / 2, wrows, kBK / 2, kBN,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ws, H / 16, wrows, 16, kBN, CU_TENSOR_MAP_SWIZZLE_NONE))
        return MOE_NVFP4_ELAUNCH;
    GemmArgs G;
    G.offsets = offsets; G.E = E; G.rows = rows; G.H = H; G.I = I;
    G.nt = static_cast<int>(2 * I / kBN); G.L = mode == kOutNvfp4 ? L : 1.0f;
    G.packed = packed; G.sf = sf; G.acc = acc; G.out_bf16 = nullptr; G.status = status;
    G.wait_cycles = kWaitCycles; G.selftest = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(kW4Threads);
    cfg.dynamicSmemBytes = kW4Smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = mode == kOutNvfp4
        ? cudaLaunchKernelEx(&cfg, l1_gemm_w4_kernel<kOutNvfp4>, tmX, tmQ, tmS, G)
        : cudaLaunchKernelEx(&cfg, l1_gemm_w4_kernel<kOutAcc>, tmX, tmQ, tmS, G);
    return e == cudaSuccess ? MOE_NVFP4_OK : MOE_NVFP4_ELAUNCH;
}

}  // namespace

extern "C" {

int moe_l1_gemm_swiglu_nvfp4(const uint16_t* x, const uint16_t* w1, int64_t rows, int64_t H, int64_t I,
                             float clamp_L, const int32_t* expert_offsets, int32_t num_experts,
                             uint8_t* packed, uint8_t* sf, int32_t* status, moe_nvfp4_stream_t stream) {
    return launch_gemm(x, w1, rows, H, I, clamp_L, expert_offsets, num_experts, kOutNvfp4, packed, sf,
                       nullptr, status, reinterpret_cast<cudaStream_t>(stream));
}

int moe_l1_gemm_accumulators(const uint16_t* x, const uint16_t* w1, int64_t rows, int64_t H, int64_t I,
                             const int32_t* expert_offsets, int32_t num_experts, float* acc,
                             int32_t* status, moe_nvfp4_stream_t stream) {
    return launch_gemm(x, w1, rows, H, I, 1.0f, expert_offsets, num_experts, kOutAcc, nullptr, nullptr, acc,
                       status, reinterpret_cast<cudaStream_t>(stream));
}

int moe_l1_gemm_wait_selftest(const uint16_t* x, const uint16_t* w1, int64_t rows, int64_t H, int64_t I,
                              const int32_t* expert_offsets, int32_t num_experts, uint8_t* packed,
                              uint8_t* sf, int32_t* status, int64_t wait_cycles, int32_t mode,
                              moe_nvfp4_stream_t stream) {
    if (status == nullptr) return MOE_NVFP4_ENULL;
    if (wait_cycles < 1000 || wait_cycles > kWaitCycles) return MOE_NVFP4_ESIZE;
    if (mode != MOE_L1_GEMM_SELFTEST_NO_LOADS && mode != MOE_L1_GEMM_SELFTEST_NO_RELEASE) return MOE_NVFP4_EMODE;
    return launch_gemm(x, w1, rows, H, I, 7.0f, expert_offsets, num_experts, kOutNvfp4, packed, sf, nullptr,
                       status, reinterpret_cast<cudaStream_t>(stream), wait_cycles, mode);
}

int moe_l1_gemm_bf16(const uint16_t* x, const uint16_t* w1, int64_t rows, int64_t H, int64_t I,
                     float clamp_L, const int32_t* expert_offsets, int32_t num_experts, int32_t output,
                     uint16_t* out, int32_t* status, moe_nvfp4_stream_t stream) {
    if (output != MOE_L1_GEMM_GU && output != MOE_L1_GEMM_SWIGLU) return MOE_NVFP4_EMODE;
    return launch_gemm(x, w1, rows, H, I, clamp_L, expert_offsets, num_experts,
                       output == MOE_L1_GEMM_GU ? kOutGuBf16 : kOutSwigluBf16, nullptr, nullptr, out, status,
                       reinterpret_cast<cudaStream_t>(stream));
}

int moe_l1_gemm_w4_swiglu_nvfp4(const uint16_t* x, const uint8_t* w1_packed, const uint8_t* w1_sf,
                                int64_t rows, int64_t H, int64_t I, float clamp_L, const int32_t* expert_offsets,
                                int32_t num_experts, uint8_t* packed, uint8_t* sf, int32_t* status,
                                moe_nvfp4_stream_t stream) {
    return launch_gemm_w4(x, w1_packed, w1_sf, rows, H, I, clamp_L, expert_offsets, num_experts, kOutNvfp4,
                          packed, sf, nullptr, status, reinterpret_cast<cudaStream_t>(stream));
}

int moe_l1_gemm_w4_accumulators(const uint16_t* x, const uint8_t* w1_packed, const uint8_t* w1_sf,
                                int64_t rows, int64_t H, int64_t I, const int32_t* expert_offsets,
                                int32_t num_experts, float* acc, int32_t* status, moe_nvfp4_stream_t stream) {
    return launch_gemm_w4(x, w1_packed, w1_sf, rows, H, I, 1.0f, expert_offsets, num_experts, kOutAcc, nullptr,
                          nullptr, acc, status, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
