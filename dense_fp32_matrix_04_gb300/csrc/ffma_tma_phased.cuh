// TMA-fed FP32 SGEMM for operands whose rows are only 4-byte aligned: a
// leading dimension that is not a multiple of 4 floats, or a base off a
// 16-byte boundary.  The tensor-memory accelerator needs 16-byte aligned bases
// and row pitches, so such an operand cannot be described by one tensor map.
// Its rows r = 4 q + s of one residue s, however, are 4 * ld floats apart -- a
// multiple of 16 bytes for every ld -- so each of the four "phases" s is a
// TMA-addressable matrix:
//  * Phase s starts at the 16-byte boundary at or below row s (d_s floats
//    below it, d_s < 4) and is read in boxes 4 floats wider than the tile, at
//    x-coordinates that are multiples of 4 (a TMA rule).  Element c of a tile
//    row then lands d_s floats to the right of its place in shared memory.
//    The d_s floats in front of a row are the previous row's tail (or, for
//    phase 0, the bytes before the operand in the same 16-byte granule); they
//    are never used.  Each phase map ends at the operand's last column, so the
//    hardware zero-fills everything past it, as it does past the last row.
//  * After a stage lands, every warp shifts its share of the rows with d_s > 0
//    left by d_s floats in place (read the row, __syncwarp, write it back),
//    before the CTA barrier that precedes the stage's FMAs.  The per-thread
//    FMAs, their order and the epilogue's arithmetic are the TMA kernel's;
//    only the shared-memory addresses and the row map differ.
//  * The stage keeps the boxes as they land, phase by phase: A's rows in
//    phase-major order (tile row 4 q + s at shared row s * BM/4 + q, 144-byte
//    pitch: the 36-float box row) and B's k-rows likewise (k = 4 q + s at
//    shared row s * BK/4 + q, pitch BN + 4 floats).  A thread still reads
//    shared rows lm + 8 i; with a 36-word pitch the eight lm values hit eight
//    different 16-byte bank groups (the pages' padding, "Memory hierarchy --
//    visual walkthrough", Step 6), and the epilogue maps shared row rho back
//    to tile row 4 (rho mod BM/4) + rho / (BM/4).
//  * Measured on GB300 against per-thread cp.async copies of the same tile:
//    3001 x 4999 x 2047 (lda 2047, ldb 4999) 51.9 -> 57.2 TFLOP/s, 8192^3
//    with lda = ldb = 8193 59.9 -> 63.5, results bit-identical.
// The reuse scheme is that of the aligned kernel: block tiles staged in shared
// memory ("SGEMM: Shared Memory Tiling Visualizer"), per-thread register outer
// products ("SGEMM: 2D Register Tiling Visualizer"), and masking done by the
// copy engine's zero fill.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "epilogue.cuh"
#include "ffma_tma_sgemm.cuh"
#include "ptx.cuh"
#include "tile_map.cuh"

namespace sgemm {

// The four phase maps of each operand (A: M x K, B: K x N, row-major).  The
// kernel takes their shifts separately, two bits per phase (bits 2 s and
// 2 s + 1 hold d_s).
struct PhasedMaps {
    CUtensorMap a[4];
    CUtensorMap b[4];
};

// Shared-memory layout of tile T read through phase maps.
template <class T>
struct PhasedTile : T {
    static constexpr int A_PITCH = (T::BK + 4) * 4;  // bytes per A row: the box row of BK + 4 floats
    static constexpr int B_PITCH = (T::BN + 4) * 4;  // bytes per B row
    static constexpr int A_PHASE_ROWS = T::BM / 4;   // A rows of one phase in a tile
    static constexpr int B_PHASE_ROWS = T::BK / 4;   // B rows of one phase in a k-step
    static constexpr int A_STAGE = T::BM * A_PITCH;
    static constexpr int B_STAGE = T::BK * B_PITCH;
    static constexpr int STAGE = A_STAGE + B_STAGE;
    static constexpr int SMEM_BYTES = T::STAGES * STAGE + 1024 /* alignment slack */ + 8 * T::STAGES;
    static constexpr bool CSPLIT_OK = T::PACKED && T::TM * T::TN * T::THREADS * 4 + 16 <= T::STAGES * STAGE;
    static constexpr int WARPS = T::THREADS / 32;
    static_assert(T::PACKED, "the phased form uses the packed accumulators");
    static_assert(A_PITCH % 16 == 0 && B_PITCH % 16 == 0, "16-byte rows for the 16-byte fragment loads");
    static_assert((A_PHASE_ROWS * A_PITCH) % 128 == 0 && (B_PHASE_ROWS * B_PITCH) % 128 == 0 && A_STAGE % 128 == 0 &&
                      STAGE % 128 == 0,
                  "every TMA destination on a 128-byte boundary");
    static_assert(A_PHASE_ROWS % WARPS == 0 && B_PHASE_ROWS % WARPS == 0 && T::BN % 32 == 0,
                  "the shift divides each phase's rows evenly among the warps");
    static_assert(T::WM % A_PHASE_ROWS == 0 && A_PHASE_ROWS % 8 == 0, "warp rows cover whole phase blocks");
    static_assert(T::BM + 4 <= 256 && T::BK + 4 <= 256 && T::BN + 4 <= 256, "a TMA box spans at most 256 elements");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// One stage of FMAs on the phased layout: the arithmetic of tile_fma (packed
// column pairs, A duplicated into both halves), with A rows at pitch A_PITCH
// (no swizzle) and the B row of k = 4 g + kk at shared row kk * BK/4 + g.
template <class T>
__device__ __forceinline__ void tile_fma_phased(uint64_t (&acc2)[T::TM][T::TN / 2], const unsigned char *sa,
                                                const unsigned char *sb) {
#pragma unroll T::G_UNROLL
    for (int g = 0; g < T::BK / 4; ++g) {
        const unsigned char *ag = sa + (g << 4);
        float4 a[T::TM];
#pragma unroll
        for (int i = 0; i < T::TM; ++i) a[i] = *reinterpret_cast<const float4 *>(ag + 8 * T::A_PITCH * i);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const unsigned char *bk = sb + (kk * T::B_PHASE_ROWS + g) * T::B_PITCH;
            uint64_t b2[T::TN / 2];
#pragma unroll
            for (int q = 0; q < T::TN / 4; ++q) {
                const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(bk + 64 * q);
                b2[2 * q] = v.x;
                b2[2 * q + 1] = v.y;
            }
            if (T::ORDER == 1) {
                uint64_t ad[T::TM];
#pragma unroll
                for (int i = 0; i < T::TM; ++i)
                    ad[i] = f32x2_dup(kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w);
#pragma unroll
                for (int j = 0; j < T::TN / 2; ++j)
#pragma unroll
                    for (int ii = 0; ii < T::TM; ++ii) {  // rows down and up in turn, as tile_fma
                        const int i = (T::MIN_BLOCKS < 4 && (j & 1)) ? T::TM - 1 - ii : ii;
                        f32x2_fma(acc2[i][j], ad[i], b2[j]);
                    }
            } else {
#pragma unroll
                for (int i = 0; i < T::TM; ++i) {
                    const uint64_t ad = f32x2_dup(kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w);
#pragma unroll
                    for (int j = 0; j < T::TN / 2; ++j) f32x2_fma(acc2[i][j], ad, b2[j]);
                }
            }
        }
    }
}

// Shift this warp's share of a landed stage's rows left by their phase's d_s
// (da, db: two bits per phase): warp w takes rows w * R .. w * R + R - 1 of
// every phase block (R = phase rows / warps).  Each row moves through
// registers: every lane reads its words, __syncwarp, every lane writes them
// back d_s words to the left.  Consecutive lanes touch consecutive words (no
// bank conflicts).  Phases with d_s = 0 are left alone (a warp-uniform test).
template <class T>
__device__ __forceinline__ void shift_stage(unsigned char *stage, int warp, int lane, uint32_t da, uint32_t db) {
    constexpr int AR = T::A_PHASE_ROWS / T::WARPS;
    constexpr int BR = T::B_PHASE_ROWS / T::WARPS;
    constexpr int AW = T::A_PITCH / 4, BW = T::B_PITCH / 4;  // row pitches in words
    constexpr int BC = T::BN / 32;                           // words of a B row per lane
    // A rows move in batches; tiles that run four CTAs per SM (128 registers)
    // take smaller batches
    constexpr int AB = T::MIN_BLOCKS >= 4 && AR > 4 ? 4 : AR;
    static_assert(AR % AB == 0, "whole batches");
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int d = (da >> (2 * s)) & 3;
        if (d == 0) continue;
#pragma unroll
        for (int r0 = 0; r0 < AR; r0 += AB) {
            float *rows = reinterpret_cast<float *>(stage + (s * T::A_PHASE_ROWS + warp * AR + r0) * T::A_PITCH);
            float v[AB];
#pragma unroll
            for (int r = 0; r < AB; ++r) v[r] = rows[r * AW + lane + d];
            __syncwarp();
#pragma unroll
            for (int r = 0; r < AB; ++r) rows[r * AW + lane] = v[r];
        }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int d = (db >> (2 * s)) & 3;
        if (d == 0) continue;
        float *rows = reinterpret_cast<float *>(stage + T::A_STAGE + (s * T::B_PHASE_ROWS + warp * BR) * T::B_PITCH);
        float v[BR][BC];
#pragma unroll
        for (int r = 0; r < BR; ++r)
#pragma unroll
            for (int c = 0; c < BC; ++c) v[r][c] = rows[r * BW + 32 * c + lane + d];
        __syncwarp();
#pragma unroll
        for (int r = 0; r < BR; ++r)
#pragma unroll
            for (int c = 0; c < BC; ++c) rows[r * BW + 32 * c + lane] = v[r][c];
    }
}

// Epilogue of the phased form: the thread's accumulator row i belongs to
// shared row rho = warp_m WM + lm + 8 i, which holds tile row
// 4 (rho mod P) + rho / P (P = BM/4).  With WM a multiple of P and lm < 8 that
// is row_base + 4 (8 i mod P) + 8 i / P, row_base = m0 + warp_m WM / P + 4 lm;
// otherwise as store_tile.
template <class T, bool VEC_C, bool CSPLIT>
__device__ __forceinline__ void store_tile_phased(const uint64_t (&acc2)[T::TM][T::TN / 2], float *C, int ldc, int M,
                                                  int N, int row_base, int c0, float alpha, float beta, int cs,
                                                  int rank) {
    constexpr int P = T::A_PHASE_ROWS;
#pragma unroll
    for (int i = 0; i < T::TM; ++i) {
        const int row = row_base + 4 * ((8 * i) % P) + (8 * i) / P;
        if (row >= M) continue;
        if (CSPLIT && (i * cs) / T::TM != rank) continue;
        float *crow = C + (int64_t)row * ldc;
#pragma unroll
        for (int q = 0; q < T::TN / 4; ++q) {
            const float2 lo = f32x2_unpack(acc2[i][2 * q]), hi = f32x2_unpack(acc2[i][2 * q + 1]);
            const float vp[4] = {lo.x, lo.y, hi.x, hi.y};
            store_quad<VEC_C>(crow, c0 + 16 * q, N, vp, alpha, beta);
        }
    }
}

// The phased kernel: tiles, roles (plain, primary, cluster split), split-K
// slabs, bounded waits and error reporting as sgemm_ffma_tma_kernel.  Per
// k-step one thread issues eight boxes (four phases of A, four of B) onto the
// stage's mbarrier.  The k-loop consumes stage t while the shift of stage t + 1
// waits for it to land and then realigns it, so the one CTA barrier per step
// both releases stage t for its next copy and publishes stage t + 1.
template <class T, bool VEC_C, int ROLE = kRolePlain>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
    sgemm_ffma_tma_phased_kernel(const __grid_constant__ PhasedMaps maps, uint32_t da, uint32_t db, int M, int N, int K,
                                 float alpha, float beta, float *__restrict__ C, int ldc,
                                 float *__restrict__ partials, int ldp, int tile_base, int *__restrict__ err_word,
                                 unsigned long long wait_limit_ns, int debug) {
    constexpr bool CSPLIT = ROLE == kRoleSplit;
    static_assert(!CSPLIT || T::CSPLIT_OK, "the cluster split exchanges packed accumulators through the stage buffers");
    if constexpr (ROLE == kRolePrimary) griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);
    const uint32_t bars = base + T::STAGES * T::STAGE;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    const int tiles_m = (M + T::BM - 1) / T::BM;
    const int tiles_n = (N + T::BN - 1) / T::BN;
    const int cs = CSPLIT ? (int)cluster_nctarank() : 1;
    const int rank = CSPLIT ? (int)cluster_ctarank() : 0;
    int tile_m, tile_n;
    grouped_tile<8>(tile_base + (CSPLIT ? (int)cluster_id_x() : (int)blockIdx.x), tiles_m, tiles_n, tile_m, tile_n);
    const int m0 = tile_m * T::BM;
    const int n0 = tile_n * T::BN;
    const int KT_all = (K + T::BK - 1) / T::BK;
    const int parts = CSPLIT ? cs : (int)gridDim.y;
    const int part = CSPLIT ? rank : (int)blockIdx.y;
    const int per_split = (KT_all + parts - 1) / parts;
    const int kt_begin = part * per_split;
    const int KT = max(0, min(KT_all, kt_begin + per_split) - kt_begin);
    if (!CSPLIT && gridDim.y > 1) {
        C = partials + (int64_t)blockIdx.y * M * ldp;
        ldc = ldp;
    }

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            prefetch_tensor_map(&maps.a[s]);
            prefetch_tensor_map(&maps.b[s]);
        }
#pragma unroll
        for (int s = 0; s < T::STAGES; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // k-step kt into stage s: phase p of A is tile rows 4 q + p (map rows
    // m0 / 4 + q), of B k-rows k0 + 4 q + p (map rows k0 / 4 + q); both x
    // coordinates (k0, n0) are multiples of 4
    auto issue = [&](int kt, int s) {
        const uint32_t bar = bars + 8 * s;
        const uint32_t dst = base + s * T::STAGE;
        const int k0 = (kt_begin + kt) * T::BK;
        mbar_arrive_expect_tx(bar, T::STAGE);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            tma_load_2d(dst + p * T::A_PHASE_ROWS * T::A_PITCH, &maps.a[p], k0, m0 / 4, bar);
            tma_load_2d(dst + T::A_STAGE + p * T::B_PHASE_ROWS * T::B_PITCH, &maps.b[p], n0, k0 / 4, bar);
        }
    };
    const bool copies = !(debug & kDebugSkipCopies);
    if (tid == 0 && copies) {
        const int pre = KT < T::STAGES ? KT : T::STAGES;
        for (int s = 0; s < pre; ++s) issue(s, s);
    }

    const int lm = (lane & 3) | (((lane >> 3) & 1) << 2);
    const int ln = ((lane >> 2) & 1) | (((lane >> 4) & 1) << 1);
    const int warp_m = warp / T::WARPS_N;
    const int warp_n = warp % T::WARPS_N;
    const int row0 = warp_m * T::WM + lm;      // shared rows row0 + 8 i, i < TM
    const int col0 = warp_n * T::WN + ln * 4;  // columns col0 + 16 q + (0..3), q < TN / 4

    uint64_t acc2[T::TM][T::TN / 2];
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
#pragma unroll
        for (int j = 0; j < T::TN / 2; ++j) acc2[i][j] = 0ull;

    // wait for k-step kt and realign it (every thread takes part)
    auto land = [&](int kt) {
        const int s = kt % T::STAGES;
        const bool ok = mbar_wait_bounded(bars + 8 * s, (kt / T::STAGES) & 1, wait_limit_ns);
        if (ok) shift_stage<T>(smem + s * T::STAGE, warp, lane, da, db);
        return ok;
    };

    int failed_kt = -1;
    if (KT > 0 && __syncthreads_or(!land(0))) failed_kt = 0;
    for (int kt = 0; kt < KT && failed_kt < 0; ++kt) {
        const int s = kt % T::STAGES;
        tile_fma_phased<T>(acc2, smem + s * T::STAGE + row0 * T::A_PITCH,
                           smem + s * T::STAGE + T::A_STAGE + col0 * 4);
        const bool ok = kt + 1 >= KT || land(kt + 1);
        // every warp is done with stage s and has realigned its rows of stage s + 1
        if (__syncthreads_or(!ok)) {
            failed_kt = kt + 1;
            break;
        }
        if (tid == 0 && copies && kt + T::STAGES < KT) issue(kt + T::STAGES, s);
    }

    if (failed_kt >= 0) {
        if (tid == 0) {
            atomicCAS(err_word, kDeviceErrNone, kDeviceErrTimeout);
            // let the copies already issued land before the CTA's shared memory is
            // released: the prologue issued k-steps [0, STAGES), and iteration kt
            // (failing on k-step failed_kt = kt + 1) had issued up to kt + STAGES - 1
            const int issued = copies ? min(KT, failed_kt == 0 ? T::STAGES : failed_kt + T::STAGES - 1) : 0;
            for (int t = failed_kt; t < issued; ++t)
                (void)mbar_wait_bounded(bars + 8 * (t % T::STAGES), (t / T::STAGES) & 1, wait_limit_ns);
        }
        __syncthreads();
        if constexpr (!CSPLIT) {
            if (!T::SLABS_OK || gridDim.y <= 1) return;
            // a split-K slab is filled with NaN instead (no stale partials reach C)
            if constexpr (T::SLABS_OK) {
#pragma unroll
                for (int i = 0; i < T::TM; ++i)
#pragma unroll
                    for (int j = 0; j < T::TN / 2; ++j) acc2[i][j] = 0x7fc000007fc00000ull;
            }
        }
    }

    if constexpr (CSPLIT) {
        if (cluster_reduce<T>(acc2, base, smem, tid, cs, rank, failed_kt >= 0)) {
            griddep_wait();
            return;
        }
    }
    store_tile_phased<T, VEC_C, CSPLIT>(acc2, C, ldc, M, N, m0 + warp_m * (T::WM / T::A_PHASE_ROWS) + 4 * lm,
                                        n0 + col0, alpha, beta, cs, rank);
    if constexpr (CSPLIT) griddep_wait();
}

}  // namespace sgemm
