// TMA-fed register-tiled FP32 SGEMM for sm_103a (operands with 16-byte aligned
// bases and leading dimensions).
//
// Same reuse scheme as the cp.async kernel -- block tiles staged in shared
// memory, a multi-stage pipeline, per-thread register outer products, a
// bank-conflict-free layout and zero-filled edges -- with the copies moved off
// the compute threads:
//  * One thread issues two tensor-memory-accelerator (TMA) box copies per
//    k-step (a BM x BK box of A, a BK x BN box of B) that complete on an
//    mbarrier; the hardware zero-fills every element outside the matrix, which
//    is the pages' boundary masking with no per-element predicate
//    ("SGEMM: Shared Memory Tiling Visualizer", the masked tile loads).
//  * STAGES boxes are in flight; a stage is refilled as soon as every warp has
//    finished reading it ("Shared Memory Tiling", 'What tiling does not fix').
//  * A keeps its row-major layout in shared memory (rows of BK = 32 floats, 128
//    bytes), with the TMA's 128-byte swizzle: 16-byte chunk c of row r sits at
//    chunk c ^ (r % 8).  A thread owns rows lm, lm + 8, ... so the eight lanes
//    that read different rows in one 16-byte load always hit eight different
//    bank groups ("Memory hierarchy -- visual walkthrough", Step 6: padding or
//    an equivalent permutation spreads a column across the banks).
//  * Each thread keeps a TM x TN block of C (8 x 16 in the shipped
//    configuration): per group of four k it loads four k-values for each of
//    its TM rows of A (TM loads of 16 bytes), and per k a TN-wide row vector of
//    B (TN/4 loads of 16 bytes), then does TM * TN multiply-adds -- for 8 x 16,
//    24 shared loads per 512 multiply-adds ("SGEMM: 2D Register Tiling
//    Visualizer", 'Why this matters on real GPUs').  The shipped form issues
//    them as 64 packed two-wide FMAs (fma.rn.f32x2, two round-to-nearest FP32
//    FMAs each): half the instructions, which leaves the issue slots the
//    loads need.
//  * Lane bits are split so that every quarter-warp reads at most two distinct
//    16-byte chunks of B (broadcast) and at most four of A.
//  * Every wait on an mbarrier is bounded; on a timeout the CTA leaves the loop
//    together, records an error code in device memory and writes nothing.
//  * Cluster split: for grids that leave SMs idle -- few tiles, or a last
//    partial wave -- the CTAs of a thread-block cluster of 2 to 8 share one
//    tile, each taking an equal run of k-steps.  Every CTA
//    parks its partial sums in its own (now idle) stage buffers; after a
//    cluster barrier, rank r reads its share of the tile's rows from every
//    rank's shared memory in rank order (distributed shared memory), adds them
//    in that fixed order and stores those rows.  No workspace, no atomics, and
//    the same bits on every run.  When full waves of plain tiles come first,
//    the cluster-split grid is launched as a programmatic dependent of theirs:
//    its CTAs take SMs as the last plain CTAs drain instead of after all of
//    them, and each waits for the plain grid to complete before it exits, so
//    the pair completes as one product.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "epilogue.cuh"
#include "ptx.cuh"
#include "tile_map.cuh"

namespace sgemm {

// Tile shape: each thread owns TM rows (lm + 8 i) and TN columns (four
// 4-column quads at ln * 4 + 16 q) of its warp's WM x WN tile; warps form a
// WARPS_M x WARPS_N grid over the BM x BN block tile.
// ORDER selects the FFMA order of the outer product: 0 = row-major (one A value
// reused across a row of B values), 1 = column-major, 2 = rows in pairs.
// G_UNROLL: how many of the BK/4 groups of four k are unrolled (code size vs
// instruction-cache reach).
// PACKED: accumulate column pairs with the packed instruction fma.rn.f32x2
// (two round-to-nearest FP32 FMAs per instruction, the same arithmetic as two
// scalar FFMAs): a row of B gives its pairs directly from the 16-byte loads
// and the A value is duplicated into both halves; half the FMA instructions
// leaves issue slots for the loads.
template <int TM_, int TN_, int WARPS_M_, int WARPS_N_, int STAGES_, int ORDER_, int MIN_BLOCKS_, int G_UNROLL_ = 8,
          bool PACKED_ = false>
struct TmaTile {
    static constexpr int TM = TM_, TN = TN_, WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
    static constexpr int STAGES = STAGES_, ORDER = ORDER_, MIN_BLOCKS = MIN_BLOCKS_, G_UNROLL = G_UNROLL_;
    static constexpr bool PACKED = PACKED_;
    static constexpr int WM = 8 * TM, WN = 4 * TN;
    static constexpr int BM = WARPS_M * WM, BN = WARPS_N * WN, BK = 32;
    static constexpr int THREADS = 32 * WARPS_M * WARPS_N;
    static constexpr int A_STAGE = BM * BK * 4;  // BM swizzled rows of 128 bytes
    static constexpr int B_STAGE = BK * BN * 4;  // BK dense rows of BN floats
    static constexpr int STAGE = A_STAGE + B_STAGE;
    static constexpr int SMEM_BYTES = STAGES * STAGE + 1024 /* alignment slack */ + 8 * STAGES /* barriers */;
    // the cluster split parks a CTA's packed partial sums (and a flag word) in its stage buffers
    static constexpr bool CSPLIT_OK = PACKED && TM * TN * THREADS * 4 + 16 <= STAGES * STAGE;
    // launched with split-K rows (gridDim.y > 1, partial slabs): only the tiles
    // of at most two CTAs per SM (the 128 x 128 tile); the others keep their
    // register budget free of the slab-only code
    static constexpr bool SLABS_OK = MIN_BLOCKS <= 2;
    static_assert(TN % 4 == 0, "columns come in 4-wide quads");
    static_assert(BM <= 256 && BN <= 256, "a TMA box spans at most 256 elements per dimension");
    static_assert(BK * 4 == 128, "A rows must be exactly one 128-byte swizzle span");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// The shipped tile configurations (TmaMainTile, TmaSmallKTile, TmaNarrowTile)
// are in tiles.cuh.

// Error codes written to the device error word.
enum : int { kDeviceErrNone = 0, kDeviceErrTimeout = 1 };

// Debug switches (test-only): bit 0 = never issue the TMA copies, so the
// bounded waits run out.
enum : int { kDebugSkipCopies = 1 };

// A tile_fma hook that does nothing.
struct NoHook {
    __device__ __forceinline__ void operator()(int) const {}
};

// One pipeline stage of the outer-product FMAs: BK k-values for this thread's
// TM x TN block of C, reading its A rows at `sa` (128-byte rows with the
// 128-byte swizzle: the thread's rows are lm + 8 i) and its B row segments at
// `sb`.  hook(g) runs before each group g of four k-values, so a caller can
// spread other work (copies for a later stage) through the FMAs.
template <class T, class Hook = NoHook>
__device__ __forceinline__ void tile_fma(float (&acc)[T::PACKED ? 1 : T::TM][T::PACKED ? 1 : T::TN],
                                         uint64_t (&acc2)[T::PACKED ? T::TM : 1][T::PACKED ? T::TN / 2 : 1],
                                         const unsigned char *sa, const unsigned char *sb, int lm,
                                         Hook hook = Hook{}) {
#pragma unroll T::G_UNROLL
    for (int g = 0; g < T::BK / 4; ++g) {
        hook(g);
        // four k-values for each of the 8 rows, from the swizzled chunk g ^ lm
        const unsigned char *ag = sa + ((g ^ lm) << 4);
        float4 a[T::TM];
#pragma unroll
        for (int i = 0; i < T::TM; ++i) a[i] = *reinterpret_cast<const float4 *>(ag + 1024 * i);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const unsigned char *bk = sb + (4 * g + kk) * (T::BN * 4);
            if constexpr (T::PACKED) {
                uint64_t b2[T::TN / 2];
#pragma unroll
                for (int q = 0; q < T::TN / 4; ++q) {
                    const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(bk + 64 * q);
                    b2[2 * q] = v.x;
                    b2[2 * q + 1] = v.y;
                }
                if (T::ORDER == 1) {
                    // column-pair outer: one B pair reused down the TM rows; with
                    // more than 128 registers a thread, the rows are walked down and
                    // up in turn so that the last A value of one column pair is the
                    // first of the next (measured 1-2 % faster than restarting at
                    // row 0; at 128 registers it spills)
                    uint64_t ad[T::TM];
#pragma unroll
                    for (int i = 0; i < T::TM; ++i)
                        ad[i] = f32x2_dup(kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w);
#pragma unroll
                    for (int j = 0; j < T::TN / 2; ++j)
#pragma unroll
                        for (int ii = 0; ii < T::TM; ++ii) {
                            const int i = (T::MIN_BLOCKS < 4 && (j & 1)) ? T::TM - 1 - ii : ii;
                            f32x2_fma(acc2[i][j], ad[i], b2[j]);
                        }
                } else {
                    // row outer: one duplicated A value reused across the row of pairs
#pragma unroll
                    for (int i = 0; i < T::TM; ++i) {
                        const uint64_t ad =
                            f32x2_dup(kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w);
#pragma unroll
                        for (int j = 0; j < T::TN / 2; ++j) f32x2_fma(acc2[i][j], ad, b2[j]);
                    }
                }
            } else {
            float b[T::TN];
#pragma unroll
            for (int q = 0; q < T::TN / 4; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(bk + 64 * q);
                b[4 * q + 0] = v.x;
                b[4 * q + 1] = v.y;
                b[4 * q + 2] = v.z;
                b[4 * q + 3] = v.w;
            }
            float av[T::TM];
#pragma unroll
            for (int i = 0; i < T::TM; ++i)
                av[i] = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
            if (T::ORDER == 1) {
#pragma unroll
                for (int j = 0; j < T::TN; ++j)
#pragma unroll
                    for (int i = 0; i < T::TM; ++i) acc[i][j] = fmaf(av[i], b[j], acc[i][j]);
            } else if (T::ORDER == 2) {
#pragma unroll
                for (int i = 0; i < T::TM; i += 2)
#pragma unroll
                    for (int j = 0; j < T::TN; ++j) {
                        acc[i][j] = fmaf(av[i], b[j], acc[i][j]);
                        acc[i + 1][j] = fmaf(av[i + 1], b[j], acc[i + 1][j]);
                    }
            } else {
#pragma unroll
                for (int i = 0; i < T::TM; ++i)
#pragma unroll
                    for (int j = 0; j < T::TN; ++j) acc[i][j] = fmaf(av[i], b[j], acc[i][j]);
            }
            }  // scalar form
        }
    }
}

// The cluster split's exchange, after the k-loop of every CTA of a cluster of
// cs: each parks its packed partial sums in its own stage buffers (which every
// warp has finished reading), with a flag word saying whether it gave up on a
// wait; after a cluster barrier, rank r adds up its share of the rows -- rows
// i of each thread with i * cs / TM == r -- over ranks 0, 1, ..., cs - 1 in
// that order, reading the other ranks' shared memory; a second barrier keeps
// every CTA's shared memory in place until all ranks have read it.  Returns
// true when some rank gave up (then nothing may be stored).  Every thread of
// every CTA of the cluster must call it.
template <class T>
__device__ __forceinline__ bool cluster_reduce(uint64_t (&acc2)[T::PACKED ? T::TM : 1][T::PACKED ? T::TN / 2 : 1],
                                               uint32_t base, unsigned char *smem, int tid, int cs, int rank,
                                               bool failed) {
    // 16-byte chunk c = i * TN/4 + q (accumulator pairs 2q, 2q + 1 of row i) of
    // thread tid sits at (c * THREADS + tid) * 16; the flag word follows the chunks
    constexpr int CHUNKS = T::TM * T::TN / 4;
    const uint32_t flag = base + CHUNKS * T::THREADS * 16;
    if (!failed) {
#pragma unroll
        for (int i = 0; i < T::TM; ++i)
#pragma unroll
            for (int q = 0; q < T::TN / 4; ++q)
                *reinterpret_cast<ulonglong2 *>(smem + ((i * (T::TN / 4) + q) * T::THREADS + tid) * 16) =
                    make_ulonglong2(acc2[i][2 * q], acc2[i][2 * q + 1]);
    }
    if (tid == 0) *reinterpret_cast<volatile uint32_t *>(smem + CHUNKS * T::THREADS * 16) = failed;
    cluster_sync();
    uint32_t bad = 0;
    for (int r = 0; r < cs; ++r) bad |= dsmem_ld_u32(dsmem_map(flag, (uint32_t)r));
    if (!bad) {
        const uint64_t one2 = f32x2_dup(1.f);
#pragma unroll
        for (int i = 0; i < T::TM; ++i) {
            if ((i * cs) / T::TM != rank) continue;
#pragma unroll
            for (int q = 0; q < T::TN / 4; ++q) {
                const uint32_t off = base + ((i * (T::TN / 4) + q) * T::THREADS + tid) * 16;
                uint64_t s0 = acc2[i][2 * q], s1 = acc2[i][2 * q + 1];
                if (rank != 0) {
                    const ulonglong2 v = dsmem_ld_v2u64(dsmem_map(off, 0));
                    s0 = v.x;
                    s1 = v.y;
                }
                for (int r = 1; r < cs; ++r) {
                    uint64_t v0 = acc2[i][2 * q], v1 = acc2[i][2 * q + 1];
                    if (r != rank) {
                        const ulonglong2 v = dsmem_ld_v2u64(dsmem_map(off, (uint32_t)r));
                        v0 = v.x;
                        v1 = v.y;
                    }
                    f32x2_fma(s0, v0, one2);  // s + v, rounded once (v * 1 is exact)
                    f32x2_fma(s1, v1, one2);
                }
                acc2[i][2 * q] = s0;
                acc2[i][2 * q + 1] = s1;
            }
        }
    }
    cluster_sync();
    return bad != 0;
}

// Epilogue: this thread's rows r0 + 8 i and 16-byte column quads at c0 + 16 q
// (matrix coordinates); C = alpha * acc + beta * C, masked at the edges: rows
// below row_lo or from M on, and columns from N on, are not stored.  With the
// cluster split, only the rows this rank added up.
template <class T, bool VEC_C, bool CSPLIT>
__device__ __forceinline__ void store_tile(const float (&acc)[T::PACKED ? 1 : T::TM][T::PACKED ? 1 : T::TN],
                                           const uint64_t (&acc2)[T::PACKED ? T::TM : 1][T::PACKED ? T::TN / 2 : 1],
                                           float *C, int ldc, int M, int N, int r0, int c0, float alpha, float beta,
                                           int cs, int rank, int row_lo = 0) {
#pragma unroll
    for (int i = 0; i < T::TM; ++i) {
        const int row = r0 + 8 * i;
        if (row >= M || row < row_lo) continue;
        if (CSPLIT && (i * cs) / T::TM != rank) continue;
        float *crow = C + (int64_t)row * ldc;
#pragma unroll
        for (int q = 0; q < T::TN / 4; ++q) {
            const int col = c0 + 16 * q;
            float vp[4];
            if constexpr (T::PACKED) {
                const float2 lo = f32x2_unpack(acc2[i][2 * q]), hi = f32x2_unpack(acc2[i][2 * q + 1]);
                vp[0] = lo.x, vp[1] = lo.y, vp[2] = hi.x, vp[3] = hi.y;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) vp[j] = acc[i][4 * q + j];
            }
            store_quad<VEC_C>(crow, col, N, vp, alpha, beta);
        }
    }
}

// Quiet NaN in every accumulator: what a CTA that gave up writes to its
// split-K slab.
template <class T>
__device__ __forceinline__ void poison_tile(float (&acc)[T::PACKED ? 1 : T::TM][T::PACKED ? 1 : T::TN],
                                            uint64_t (&acc2)[T::PACKED ? T::TM : 1][T::PACKED ? T::TN / 2 : 1]) {
#pragma unroll
    for (int i = 0; i < (T::PACKED ? 1 : T::TM); ++i)
#pragma unroll
        for (int j = 0; j < (T::PACKED ? 1 : T::TN); ++j) acc[i][j] = __int_as_float(0x7fc00000);
#pragma unroll
    for (int i = 0; i < (T::PACKED ? T::TM : 1); ++i)
#pragma unroll
        for (int j = 0; j < (T::PACKED ? T::TN / 2 : 1); ++j) acc2[i][j] = 0x7fc000007fc00000ull;
}

// What a launch of the kernel does: a plain grid of tiles; the same, as the
// first of a plain + cluster-split pair (it lets the second grid start early);
// or the cluster-split grid.
enum : int { kRolePlain = 0, kRolePrimary = 1, kRoleSplit = 2 };

// Tile t of the launch is grouped tile tile_base + blockIdx.x (tile_base +
// cluster index for the split role), so one product can be covered by a plain
// launch over tiles [0, full) and a cluster-split launch over [full, tiles).
// PLAIN: alpha = 1 and beta = 0 known at compile time (C = A B, the
// arguments are not read); the general epilogue in the kernel cost the k-loop
// 0.5 % at 8192^3 and 1.2 % at 2048^3.
template <class T, bool VEC_C, int ROLE = kRolePlain, bool PLAIN = false>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
    sgemm_ffma_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M,
                          int N, int K, float alpha, float beta, float *__restrict__ C, int ldc,
                          float *__restrict__ partials, int ldp, int tile_base, int *__restrict__ err_word,
                          unsigned long long wait_limit_ns, int debug) {
    constexpr bool CSPLIT = ROLE == kRoleSplit;
    static_assert(!CSPLIT || T::CSPLIT_OK, "the cluster split exchanges packed accumulators through the stage buffers");
    // the cluster-split grid queued behind this one may start as soon as all of its CTAs run
    if constexpr (ROLE == kRolePrimary) griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);
    const uint32_t bars = base + T::STAGES * T::STAGE;  // STAGES mbarriers of 8 bytes

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    const int tiles_m = (M + T::BM - 1) / T::BM;
    const int tiles_n = (N + T::BN - 1) / T::BN;
    // cluster split: `cs` CTAs share a tile; this one is rank `rank`
    const int cs = CSPLIT ? (int)cluster_nctarank() : 1;
    const int rank = CSPLIT ? (int)cluster_ctarank() : 0;
    int tile_m, tile_n;
    grouped_tile<8>(tile_base + (CSPLIT ? (int)cluster_id_x() : (int)blockIdx.x), tiles_m, tiles_n, tile_m, tile_n);
    const int m0 = tile_m * T::BM;
    const int n0 = tile_n * T::BN;
    // split-K: CTA row blockIdx.y (or cluster rank) owns k-steps [kt_begin,
    // kt_begin + KT).  A grid with more than one row writes its partial sums to
    // its own M x N slab of `partials` (leading dimension ldp) instead of C.
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
        prefetch_tensor_map(&tmA);
        prefetch_tensor_map(&tmB);
#pragma unroll
        for (int s = 0; s < T::STAGES; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int kt, int s) {
        const uint32_t bar = bars + 8 * s;
        const uint32_t dst = base + s * T::STAGE;
        mbar_arrive_expect_tx(bar, T::STAGE);
        tma_load_2d(dst, &tmA, (kt_begin + kt) * T::BK, m0, bar);
        tma_load_2d(dst + T::A_STAGE, &tmB, n0, (kt_begin + kt) * T::BK, bar);
    };
    const bool copies = !(debug & kDebugSkipCopies);
    if (tid == 0 && copies) {
        const int pre = KT < T::STAGES ? KT : T::STAGES;
        for (int s = 0; s < pre; ++s) issue(s, s);
    }

    // lane -> (lm, ln): lm from lane bits {0, 1, 3}, ln from bits {2, 4}
    const int lm = (lane & 3) | (((lane >> 3) & 1) << 2);
    const int ln = ((lane >> 2) & 1) | (((lane >> 4) & 1) << 1);
    const int warp_m = warp / T::WARPS_N;
    const int warp_n = warp % T::WARPS_N;
    const int row0 = warp_m * T::WM + lm;          // thread rows: row0 + 8 i, i < TM
    const int col0 = warp_n * T::WN + ln * 4;      // thread cols: col0 + 16 q + (0..3), q < TN / 4

    // scalar accumulators, or column pairs for the packed form (one of the two is used)
    float acc[T::PACKED ? 1 : T::TM][T::PACKED ? 1 : T::TN];
    uint64_t acc2[T::PACKED ? T::TM : 1][T::PACKED ? T::TN / 2 : 1];
    if constexpr (T::PACKED) {
#pragma unroll
        for (int i = 0; i < T::TM; ++i)
#pragma unroll
            for (int j = 0; j < T::TN / 2; ++j) acc2[i][j] = 0ull;
    } else {
#pragma unroll
        for (int i = 0; i < T::TM; ++i)
#pragma unroll
            for (int j = 0; j < T::TN; ++j) acc[i][j] = 0.f;
    }

    int failed_kt = -1;
    for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % T::STAGES;
        const bool ok = mbar_wait_bounded(bars + 8 * s, (kt / T::STAGES) & 1, wait_limit_ns);
        if (ok) {
            const unsigned char *sa = smem + s * T::STAGE + row0 * 128;
            const unsigned char *sb = smem + s * T::STAGE + T::A_STAGE + col0 * 4;
            tile_fma<T>(acc, acc2, sa, sb, lm);
        }
        // every warp is done with stage s (or the CTA gives up together)
        if (__syncthreads_or(!ok)) {
            failed_kt = kt;
            break;
        }
        if (tid == 0 && copies && kt + T::STAGES < KT) issue(kt + T::STAGES, s);
    }

    if (failed_kt >= 0) {
        if (tid == 0) {
            atomicCAS(err_word, kDeviceErrNone, kDeviceErrTimeout);
            // let the copies already issued (k-steps failed_kt .. failed_kt + STAGES - 1)
            // land before the CTA's shared memory is released; bounded as well
            if (copies)
                for (int t = failed_kt; t < KT && t < failed_kt + T::STAGES; ++t)
                    (void)mbar_wait_bounded(bars + 8 * (t % T::STAGES), (t / T::STAGES) & 1, wait_limit_ns);
        }
        __syncthreads();
        // a cluster-split CTA still takes part in both cluster barriers below
        if constexpr (!CSPLIT) {
            if (!T::SLABS_OK || gridDim.y <= 1) return;
            // a split-K slab is filled with NaN instead, so that the reduction
            // cannot add stale partial sums into C
            if constexpr (T::SLABS_OK) poison_tile<T>(acc, acc2);
        }
    }

    if constexpr (CSPLIT) {
        if (cluster_reduce<T>(acc2, base, smem, tid, cs, rank, failed_kt >= 0)) {
            griddep_wait();
            return;
        }
    }
    store_tile<T, VEC_C, CSPLIT>(acc, acc2, C, ldc, M, N, m0 + row0, n0 + col0, PLAIN ? 1.f : alpha,
                                 PLAIN ? 0.f : beta, cs, rank);
    // a cluster-split grid overlapping a plain one completes after it
    if constexpr (CSPLIT) griddep_wait();
}

}  // namespace sgemm
