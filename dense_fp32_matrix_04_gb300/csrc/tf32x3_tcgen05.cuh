// 3xTF32 SGEMM on the 5th-generation tensor cores (tcgen05, accumulator in
// TMEM) for sm_103a: C = A * B in FP32 accuracy from TF32 products.
//
// Each FP32 operand is split once, in HBM, into a TF32 "high" part and a TF32
// "low" part, a = a_hi + a_lo + e with a_hi = rna_tf32(a),
// a_lo = rna_tf32(a - a_hi) and |e| <= 2^-22 |a| (a - a_hi is exact in FP32).
// The product keeps the three largest cross terms,
//     C = A_hi B_hi + A_hi B_lo + A_lo B_hi,
// dropping A_lo B_lo (< 2^-22 |a||b|), so each product carries a relative
// error of about 3 * 2^-22 before the FP32 accumulation.  Small integers have
// a_lo = 0 and stay exact.
//
// The split itself is tf32_split.cuh.  The matrix product is the tiled scheme
// of the pages ("Shared Memory Tiling", the tiled kernel; "SGEMM: Shared
// Memory Tiling Visualizer", the masked tile loads) with the inner-product
// loop moved onto the tensor cores, in a persistent kernel of one CTA per SM
// that walks its output tiles:
//  * warp 0 (one thread) copies 128 x BK boxes of A_hi, A_lo and BN x BK boxes
//    of B_hi^T, B_lo^T (all K-major, 64-byte swizzled) into a STAGES-deep ring,
//    zero-filling outside the matrices (the boundary masking), and runs on
//    into the next tile's k-steps while the current one is computed (the
//    pipelining of 'What tiling does not fix');
//  * warp 1 (one thread) issues, per BK-deep k-step, 3 products x BK/8
//    tcgen05.mma of 128 x BN x 8 into the tile's FP32 accumulator in TMEM --
//    two accumulators, used by alternate tiles -- and commits each stage back
//    to the copy thread once the tensor cores have read it;
//  * warps 2..5 read the other accumulator out of TMEM (each warp its 32
//    lanes), hand it back, and store the tile of C with masks, staged through
//    shared memory so that the stores run along rows.
// Every mbarrier wait is bounded; a CTA that gives up writes nothing, records
// an error code in device memory and still frees its TMEM.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "epilogue.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"
#include "tile_map.cuh"

namespace sgemm {

// ---------------------------------------------------------------- tensor-core product

// BK = 32 stores operand rows of 128 bytes (128-byte swizzle); BK = 16 rows of
// 64 bytes (64-byte swizzle), which halves a stage so more stages fit.
template <int BN_, int BK_, int STAGES_>
struct Tf32x3Tile {
    static constexpr int BM = 128, BN = BN_, BK = BK_, STAGES = STAGES_;
    // 6 warps: copies (warp 0), MMA (warp 1), TMEM drain and stores (warps 2..5;
    // warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31)
    static constexpr int THREADS = 192;
    static constexpr int UMMA_K = 8;              // TF32 elements per tcgen05.mma
    static constexpr int ROW = BK * 4;            // bytes per operand row = swizzle span
    static constexpr int A_BYTES = BM * ROW;      // one operand box: 128 rows
    static constexpr int B_BYTES = BN * ROW;
    static constexpr int STAGE = 2 * A_BYTES + 2 * B_BYTES;  // A_hi, A_lo, B_hi^T, B_lo^T
    static constexpr int EPI_BYTES = 4 * 32 * 17 * 4;        // a padded 32 x 17 staging tile per drain warp
    static constexpr int SMEM_BYTES = STAGES * STAGE + EPI_BYTES + 1024 /* alignment */ + 256 /* barriers, flags */;
    // two FP32 accumulators of 128 lanes x BN columns, ACC_COLS apart (a power
    // of two >= 32), so that one tile's drain overlaps the next tile's MMAs
    static constexpr int ACC_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
    static constexpr int TMEM_COLS = 2 * ACC_COLS;
    static constexpr int SBO = 8 * ROW;           // bytes between 8-row groups of a swizzled box
    static constexpr uint32_t LAYOUT = ROW == 128 ? 2u : 4u;  // descriptor swizzle mode: 128-byte or 64-byte
    // instruction descriptor: D = F32 (bits 4-5 = 1), A = B = TF32 (bits 7-9, 10-12 = 2),
    // both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28
    static constexpr uint32_t IDESC =
        (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
    static_assert(BK == 32 || BK == 16, "operand rows of 128 or 64 bytes");
    static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
    static_assert(STAGE % 1024 == 0 || ROW == 64, "128-byte swizzled boxes start on 1024-byte boundaries");
    static_assert(A_BYTES % 512 == 0 && B_BYTES % 512 == 0, "64-byte swizzled boxes start on 512-byte boundaries");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// Shared-memory matrix descriptor for a K-major operand stored in swizzled
// rows (the layout the TMA's 128- or 64-byte swizzle writes): start address,
// leading-byte offset (unused for these layouts, set to 1), stride-byte offset
// between 8-row groups, descriptor version 1 (bit 46), swizzle mode (bits
// 61-63: 2 = 128-byte, 4 = 64-byte).
__device__ __forceinline__ uint64_t umma_desc_swizzled(uint32_t saddr, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1u << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
           ((uint64_t)1u << 46) | ((uint64_t)layout << 61);
}

// Persistent form: one CTA per SM walks the units u = blockIdx.x,
// blockIdx.x + gridDim.x, ... of `splits` x tiles units (unit u is tile
// u % tiles of the grouped raster, k-split u / tiles).  Warp 0 streams the
// units' k-steps through a STAGES-deep ring, warp 1 issues their MMAs into
// accumulator (i % 2) of the CTA's i-th unit, and warps 2..5 drain the other
// accumulator and store its tile meanwhile.  With splits > 1 each unit writes
// its partial tile to its own M x ldp slab of `partials` (the host then adds
// the slabs in split order into C).
template <class T, bool VEC_C>
__global__ void __launch_bounds__(T::THREADS, 1)
    sgemm_3xtf32_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                        const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl, int M,
                        int N, int K, int splits, float alpha, float beta, float *__restrict__ C, int ldc,
                        float *__restrict__ partials, int ldp, int *__restrict__ err_word,
                        unsigned long long wait_limit_ns, int debug) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);
    // ring, staging tiles, then full[S], empty[S], acc_full[2], acc_empty[2], drained, flags
    const uint32_t bars = base + T::STAGES * T::STAGE + T::EPI_BYTES;
    const uint32_t full0 = bars, empty0 = bars + 8 * T::STAGES;
    const uint32_t acc_full0 = bars + 16 * T::STAGES, acc_empty0 = acc_full0 + 16, drained = acc_full0 + 32;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + (bars - base) + 16 * T::STAGES + 40);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + (bars - base) + 16 * T::STAGES + 44);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles_m = (M + T::BM - 1) / T::BM, tiles_n = (N + T::BN - 1) / T::BN;
    const int tiles = tiles_m * tiles_n;
    const int units = tiles * splits;
    const int KT_all = (K + T::BK - 1) / T::BK;
    const int per_split = (KT_all + splits - 1) / splits;
    // unit u: output tile origin, first k-step and k-step count
    auto unit = [&](int u, int &m0, int &n0, int &kt0, int &kts) {
        int tm, tn;
        grouped_tile<8>(u % tiles, tiles_m, tiles_n, tm, tn);
        m0 = tm * T::BM;
        n0 = tn * T::BN;
        kt0 = (u / tiles) * per_split;
        kts = max(0, min(KT_all, kt0 + per_split) - kt0);
    };

    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), T::TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full0 + 8 * b, 1);
            mbar_init(acc_empty0 + 8 * b, 4);  // one arrival per drain warp
        }
        mbar_init(drained, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    int issued = 0;  // copy thread: k-steps issued over all of this CTA's units
    if (warp == 0 && lane == 0) {
        // ---- copies: k-step g of the CTA goes to stage g % STAGES once the
        // tensor cores have read that stage's previous contents
        prefetch_tensor_map(&tmAh);
        prefetch_tensor_map(&tmAl);
        prefetch_tensor_map(&tmBh);
        prefetch_tensor_map(&tmBl);
        const bool copies = !(debug & 1);
        for (int u = blockIdx.x; copies && u < units && !*abort_flag; u += gridDim.x) {
            int m0, n0, kt0, kts;
            unit(u, m0, n0, kt0, kts);
            for (int kt = 0; kt < kts; ++kt) {
                const int s = issued % T::STAGES, use = issued / T::STAGES;
                if (use > 0 && !mbar_wait_bounded(empty0 + 8 * s, (use - 1) & 1, wait_limit_ns)) *abort_flag = 1;
                if (*abort_flag) break;
                const uint32_t dst = base + s * T::STAGE, bar = full0 + 8 * s;
                mbar_arrive_expect_tx(bar, T::STAGE);
                const int kx = (kt0 + kt) * T::BK;
                tma_load_2d(dst, &tmAh, kx, m0, bar);
                tma_load_2d(dst + T::A_BYTES, &tmAl, kx, m0, bar);
                tma_load_2d(dst + 2 * T::A_BYTES, &tmBh, kx, n0, bar);
                tma_load_2d(dst + 2 * T::A_BYTES + T::B_BYTES, &tmBl, kx, n0, bar);
                ++issued;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- tensor cores: unit i of this CTA into accumulator i % 2,
        // D = A_hi B_hi + A_hi B_lo + A_lo B_hi over its k-steps
        int g = 0;  // k-steps consumed
        int i = 0;
        for (int u = blockIdx.x; u < units && !*abort_flag; u += gridDim.x, ++i) {
            int m0, n0, kt0, kts;
            unit(u, m0, n0, kt0, kts);
            const int b = i & 1, use = i >> 1;
            // the drain warps are done with this accumulator's previous tile
            if (use > 0 && !mbar_wait_bounded(acc_empty0 + 8 * b, (use - 1) & 1, wait_limit_ns)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after_sync();
            const uint32_t acc = tmem + (uint32_t)(b * T::ACC_COLS);
            bool ok = true;
            for (int kt = 0; kt < kts; ++kt, ++g) {
                const int s = g % T::STAGES;
                if (!mbar_wait_bounded(full0 + 8 * s, (g / T::STAGES) & 1, wait_limit_ns)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t ah = base + s * T::STAGE, al = ah + T::A_BYTES;
                const uint32_t bh = ah + 2 * T::A_BYTES, bl = bh + T::B_BYTES;
#pragma unroll
                for (int p = 0; p < 3; ++p) {
                    const uint32_t a = p == 2 ? al : ah;
                    const uint32_t bb = p == 1 ? bl : bh;
#pragma unroll
                    for (int kk = 0; kk < T::BK / T::UMMA_K; ++kk) {
                        const uint64_t da = umma_desc_swizzled(a + kk * T::UMMA_K * 4, T::SBO, T::LAYOUT);
                        const uint64_t db = umma_desc_swizzled(bb + kk * T::UMMA_K * 4, T::SBO, T::LAYOUT);
                        umma_tf32(acc, da, db, T::IDESC, (kt | p | kk) != 0);
                    }
                }
                umma_commit(empty0 + 8 * s);  // stage s may be refilled once these MMAs have read it
            }
            if (!ok) break;
            umma_commit(acc_full0 + 8 * b);  // the tile's accumulator is final once its MMAs are done
        }
        // every MMA issued above has completed before the CTA moves on
        umma_commit(drained);
        (void)mbar_wait_bounded(drained, 0, wait_limit_ns);
    } else if (warp >= 2) {
        // ---- drain warps: TMEM lanes 32 q .. 32 q + 31 of each finished tile,
        // staged 16 columns at a time through a padded 32 x 17 tile so that the
        // stores run along rows -- whole row segments per warp instruction
        // instead of one element in each of 32 rows
        const int q = warp & 3;
        float *stage = reinterpret_cast<float *>(smem + T::STAGES * T::STAGE) + (warp - 2) * (32 * 17);
        int i = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
            int m0, n0, kt0, kts;
            unit(u, m0, n0, kt0, kts);
            const int b = i & 1;
            // a finished accumulator is stored whatever another role decided
            // since, so every drain warp stores all of a tile or none of it
            // (the MMA thread commits no tile after giving up, and then every
            // drain warp's wait runs out)
            const bool ready = mbar_wait_bounded(acc_full0 + 8 * b, (i >> 1) & 1, wait_limit_ns);
            if (!__all_sync(0xffffffffu, ready)) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            tc_fence_after_sync();
            float *out = C;
            int ldo = ldc;
            if (splits > 1) {
                out = partials + (int64_t)(u / tiles) * M * ldp;
                ldo = ldp;
            }
            const int row_base = m0 + 32 * q;
            const uint32_t acc = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * T::ACC_COLS);
#pragma unroll 1
            for (int c0 = 0; c0 < T::BN; c0 += 16) {
                float v[32];
                tmem_ld16(acc + (uint32_t)c0, v);
                if (c0 + 16 == T::BN) {
                    // the accumulator is read: hand it back to the MMA thread
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty0 + 8 * b);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) stage[lane * 17 + j] = kts == 0 ? 0.f : v[j];  // kts == 0: zero sums
                __syncwarp();
                if constexpr (VEC_C) {
                    // four lanes per row, each a 4-column quad; 8 rows per instruction
                    const int cq = lane & 3, rr = lane >> 2;
#pragma unroll
                    for (int r = rr; r < 32; r += 8) {
                        const int row = row_base + r;
                        if (row < M) {
                            const float *src = stage + r * 17 + 4 * cq;
                            const float quad[4] = {src[0], src[1], src[2], src[3]};
                            store_quad<true>(out + (int64_t)row * ldo, n0 + c0 + 4 * cq, N, quad, alpha, beta);
                        }
                    }
                } else {
                    // one column per lane; 2 rows per instruction
                    const int j = lane & 15, rr = lane >> 4, col = n0 + c0 + j;
#pragma unroll 4
                    for (int r = rr; r < 32; r += 2) {
                        const int row = row_base + r;
                        if (row < M && col < N) store_one(out + (int64_t)row * ldo + col, stage[r * 17 + j], alpha, beta);
                    }
                }
                __syncwarp();
            }
        }
    }

    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) {
            atomicCAS(err_word, 0, 1);
            // let the copies still in flight land before shared memory is released (bounded)
            for (int t = issued - T::STAGES > 0 ? issued - T::STAGES : 0; t < issued; ++t)
                (void)mbar_wait_bounded(full0 + 8 * (t % T::STAGES), (t / T::STAGES) & 1, wait_limit_ns);
        }
        if (splits > 1 && warp >= 2) {
            // every partial slab of this CTA's units is filled with NaN, so that the
            // reduction cannot add stale partial sums into C
            const int q = warp & 3;
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                int m0, n0, kt0, kts;
                unit(u, m0, n0, kt0, kts);
                const int row = m0 + 32 * q + lane;
                if (row >= M) continue;
                float *slab = partials + (int64_t)(u / tiles) * M * ldp + (int64_t)row * ldp;
                const float nan4[4] = {__int_as_float(0x7fc00000), __int_as_float(0x7fc00000),
                                       __int_as_float(0x7fc00000), __int_as_float(0x7fc00000)};
                for (int c = 0; c < T::BN; c += 4) store_quad<true>(slab, n0 + c, N, nan4, 1.f, 0.f);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, T::TMEM_COLS);
}

// Tile configurations: 128 x BN output tiles, 16-deep k-steps with 64-byte
// swizzled rows, and as many stages as fit beside the drain warps' staging
// tiles (at most 6).  The depth of the ring decides the speed: measured on
// GB300 (GEMM alone, FP32-equivalent TFLOP/s, 8192^3 / 3001 x 4999 x 2047),
// 128 x 208 with 5 stages 340.7 / 300.9, 128 x 256 with 4 (a fifth does not
// fit) 333.3 / 246.4, with 3 286.1 / 213.9, 128 x 240 and 128 x 224 with 4
// 332 / 258 and 320 / 265, 128 x 192 with 5 324.8 / 256.8, 128 x 160 with 6
// 304.6 / 233.9, 128 x 128 with 6 251.7 / 206.5; BK = 32 (128-byte rows)
// with 2 or 3 stages 285 to 300 / 213 to 244.
template <int BN>
struct Tf32x3Stages {
    static constexpr int STAGE = (2 * 128 + 2 * BN) * 64;
    static constexpr int FIT = (227 * 1024 - 4 * 32 * 17 * 4 - 1024 - 256) / STAGE;
    static constexpr int value = FIT > 6 ? 6 : FIT;
};
template <int BN>
using Tf32x3WidthTile = Tf32x3Tile<BN, 16, Tf32x3Stages<BN>::value>;

// The widest tile with five stages: 128 x 208.
using Tf32x3MainTile = Tf32x3WidthTile<208>;
static_assert(Tf32x3MainTile::STAGES == 5, "five stages of the 208-wide tile");

// Tile widths the 3xTF32 product chooses from, widest first (each with at
// least five stages): products whose 128 x 208 tiles would leave a last,
// mostly idle round over the SMs take a narrower tile that fills it better.
constexpr int kTf32x3Widths[] = {208, 192, 176, 160, 144, 128};

}  // namespace sgemm
