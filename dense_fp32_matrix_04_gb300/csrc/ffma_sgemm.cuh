// Register-tiled FP32 SGEMM for sm_103a: C = A * B, row-major, general shapes.
//
// Scheme (the pages' reuse steps, sized for a 152-SM GB300):
//  * Thread-block tiling: each CTA owns a BM x BN block of C and walks K in
//    BK-deep steps, staging a BM x BK slab of A and a BK x BN slab of B in
//    shared memory so that every element fetched from HBM is reused BN (resp.
//    BM) times ("Shared Memory Tiling", 'The reuse argument' and the tiled
//    kernel; "Memory hierarchy -- visual walkthrough", Steps 3-5).
//  * Software pipelining: STAGES slabs in flight through cp.async, so the copy
//    of step t + STAGES - 1 overlaps the arithmetic of step t, with one barrier
//    per step ("Shared Memory Tiling", 'What tiling does not fix').
//  * 2-D register tiling: each thread keeps an 8 x 8 block of C in registers
//    and, per k, loads a column vector of 8 A values and a row vector of 8 B
//    values (two 16-byte shared loads each) for 64 FFMAs -- 16 shared reads
//    per 64 multiply-adds ("SGEMM: 2D Register Tiling Visualizer", listing and
//    'Why this matters on real GPUs').  The fragments of k + 1 are loaded
//    while the FFMAs of k run.
//  * Bank-conflict-free layout: A is stored k-major (transposed) so a thread's
//    8 A values are contiguous; rows of that tile are padded by 4 words so the
//    transposing 4-byte stores of a warp (4 rows x 8 k) hit 32 distinct banks,
//    while the 16-byte fragment reads stay aligned.  B keeps its row-major
//    layout, whose row reads are conflict-free ("SGEMM: Shared Memory Tiling
//    Visualizer", 'Why no padding?'; "Memory hierarchy -- visual
//    walkthrough", Step 6).
//  * Boundary masking: slots outside A or B are zero-filled by the copy itself
//    (source size 0) and stores outside C are skipped ("SGEMM: Shared Memory
//    Tiling Visualizer", the masked tile loads; "Shared Memory Tiling", the
//    remark on boundary handling).
//  * Coalesced, vectorised access: B moves in 16-byte copies and C in 16-byte
//    stores whenever the pointer and leading dimension allow it
//    ("Shared Memory Tiling", opening paragraph).
#pragma once

#include <cstdint>

#include "epilogue.cuh"
#include "ptx.cuh"
#include "tile_map.cuh"

namespace sgemm {

template <int BM_, int BN_, int BK_, int STAGES_, int MIN_BLOCKS_>
struct FfmaTile {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_, MIN_BLOCKS = MIN_BLOCKS_;
    // warp tile 64 x 32: lanes as 8 (m) x 4 (n), each thread two 4-row and two
    // 4-column quads (8 x 8 outputs)
    static constexpr int WM = 64, WN = 32;
    static constexpr int LANES_M = 8, LANES_N = 4;
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int WARPS = WARPS_M * WARPS_N;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int A_PAD = 4;
    static constexpr int A_LD = BM + A_PAD;  // words per k-row of the k-major A slab
    static constexpr int B_LD = BN;          // words per k-row of the B slab
    static constexpr int A_STAGE = BK * A_LD;
    static constexpr int B_STAGE = BK * B_LD;
    static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    // A copies: a warp instruction covers 4 rows x 8 k
    static constexpr int KO = BK / 8;
    static constexpr int A_LOADS = BM * BK / THREADS;
    static constexpr int A_ROW_STEP = 4 * WARPS / KO;
    // B copies
    static constexpr int B_VEC_LOADS = BK * BN / (4 * THREADS);
    static constexpr int B_VEC_KSTEP = THREADS / (BN / 4);
    static constexpr int B_SCALAR_LOADS = BK * BN / THREADS;
    static constexpr int B_SCALAR_KSTEP = THREADS / BN;

    static_assert(BM % WM == 0 && BN % WN == 0, "block tile must be a whole number of warp tiles");
    static_assert(BK % 8 == 0 && WARPS % KO == 0, "A copy layout needs BK % 8 == 0 and WARPS % (BK/8) == 0");
    static_assert((BM * BK) % THREADS == 0 && A_LOADS * THREADS == BM * BK, "A slab must split evenly");
    static_assert(THREADS % (BN / 4) == 0 && (BK * BN) % (4 * THREADS) == 0, "B slab must split evenly");
    static_assert(THREADS % BN == 0 || BN > THREADS, "scalar B copy layout");
    static_assert(STAGES >= 2, "pipeline needs two stages");
};

template <class T, bool VEC_B, bool VEC_C>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
    sgemm_ffma_kernel(int M, int N, int K, float alpha, const float *__restrict__ A, int lda,
                      const float *__restrict__ B, int ldb, float beta, float *__restrict__ C, int ldc,
                      float *__restrict__ partials, int ldp) {
    extern __shared__ __align__(16) float smem[];
    float *sA = smem;                          // [STAGES][BK][A_LD]
    float *sB = smem + T::STAGES * T::A_STAGE;  // [STAGES][BK][B_LD]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    const int tiles_m = (M + T::BM - 1) / T::BM;
    const int tiles_n = (N + T::BN - 1) / T::BN;
    int tile_m, tile_n;
    grouped_tile<8>(blockIdx.x, tiles_m, tiles_n, tile_m, tile_n);
    const int m0 = tile_m * T::BM;
    const int n0 = tile_n * T::BN;

    // ---------------------------------------------------------------- copy roles
    // A: lane -> (row within quad, k within octet); warp/i -> (row quad, k octet)
    const int a_k = (warp % T::KO) * 8 + (lane & 7);
    const int a_row0 = (warp / T::KO) * 4 + (lane >> 3);
    uint32_t a_valid = 0;  // bit i: row of copy i lies inside A
#pragma unroll
    for (int i = 0; i < T::A_LOADS; ++i)
        if (m0 + a_row0 + i * T::A_ROW_STEP < M) a_valid |= 1u << i;
    const float *gA = A + (int64_t)(m0 + a_row0) * lda + a_k;
    const int64_t a_step = (int64_t)T::A_ROW_STEP * lda;
    const uint32_t sA_dst = smem_addr(sA + a_k * T::A_LD + a_row0);

    // B: vector copies move 4 consecutive columns, scalar copies one column
    int b_col, b_krow0, b_bytes;
    int64_t b_step;
    if (VEC_B) {
        b_col = (tid % (T::BN / 4)) * 4;
        b_krow0 = tid / (T::BN / 4);
        b_step = (int64_t)T::B_VEC_KSTEP * ldb;
        const int left = N - (n0 + b_col);
        b_bytes = left >= 4 ? 16 : (left > 0 ? left * 4 : 0);
    } else {
        b_col = tid % T::BN;
        b_krow0 = tid / T::BN;
        b_step = (int64_t)T::B_SCALAR_KSTEP * ldb;
        b_bytes = (n0 + b_col < N) ? 4 : 0;
    }
    const float *gB = B + (int64_t)b_krow0 * ldb + n0 + b_col;
    const uint32_t sB_dst = smem_addr(sB + b_krow0 * T::B_LD + b_col);

    // split-K: CTA row blockIdx.y owns k-steps [kt_begin, kt_begin + KT) and, when
    // the grid has more than one row, writes its partial sums to its own M x N
    // slab of `partials` (leading dimension ldp) instead of C
    const int KT_all = (K + T::BK - 1) / T::BK;
    const int per_split = (KT_all + gridDim.y - 1) / gridDim.y;
    const int kt_begin = blockIdx.y * per_split;
    const int KT = max(0, min(KT_all, kt_begin + per_split) - kt_begin);
    if (gridDim.y > 1) {
        C = partials + (int64_t)blockIdx.y * M * ldp;
        ldc = ldp;
    }

    // Issue the copies of k-step `kt` (counted from kt_begin) into pipeline slot `slot`.
    auto load_slab = [&](int kt, int slot) {
        const int k0 = (kt_begin + kt) * T::BK;
        const bool full_k = k0 + T::BK <= K;
        // A
        {
            const float *src = gA + k0;
            const bool k_ok = full_k || (k0 + a_k < K);
            const uint32_t dst = sA_dst + slot * (T::A_STAGE * 4);
#pragma unroll
            for (int i = 0; i < T::A_LOADS; ++i) {
                const bool ok = k_ok && ((a_valid >> i) & 1u);
                cp_async_4(dst + i * T::A_ROW_STEP * 4, ok ? (const void *)(src + i * a_step) : (const void *)A,
                           ok ? 4 : 0);
            }
        }
        // B
        {
            const float *src = gB + (int64_t)k0 * ldb;
            const uint32_t dst = sB_dst + slot * (T::B_STAGE * 4);
            if (VEC_B) {
#pragma unroll
                for (int i = 0; i < T::B_VEC_LOADS; ++i) {
                    const bool ok = full_k || (k0 + b_krow0 + i * T::B_VEC_KSTEP < K);
                    const int bytes = ok ? b_bytes : 0;
                    cp_async_16(dst + i * T::B_VEC_KSTEP * T::B_LD * 4,
                                bytes ? (const void *)(src + i * b_step) : (const void *)B, bytes);
                }
            } else {
#pragma unroll
                for (int i = 0; i < T::B_SCALAR_LOADS; ++i) {
                    const bool ok = full_k || (k0 + b_krow0 + i * T::B_SCALAR_KSTEP < K);
                    const int bytes = ok ? b_bytes : 0;
                    cp_async_4(dst + i * T::B_SCALAR_KSTEP * T::B_LD * 4,
                               bytes ? (const void *)(src + i * b_step) : (const void *)B, bytes);
                }
            }
        }
    };

    // ---------------------------------------------------------------- compute roles
    const int warp_m = warp / T::WARPS_N;
    const int warp_n = warp % T::WARPS_N;
    const int lm = lane >> 2;  // 0..7
    const int ln = lane & 3;   // 0..3
    const int frag_a = warp_m * T::WM + lm * 4;  // first A column (m) of quad 0; quad 1 at +32
    const int frag_b = warp_n * T::WN + ln * 4;  // first B column (n) of quad 0; quad 1 at +16

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    // prologue: fill STAGES - 1 slots
#pragma unroll
    for (int s = 0; s < T::STAGES - 1; ++s) {
        if (s < KT) load_slab(s, s);
        cp_async_commit();
    }

    int read_slot = 0;
    int write_slot = T::STAGES - 1;
    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<T::STAGES - 2>();
        __syncthreads();  // slab kt visible to all; slot of kt-1 free for reuse

        if (kt + T::STAGES - 1 < KT) load_slab(kt + T::STAGES - 1, write_slot);
        cp_async_commit();

        const float *As = sA + read_slot * T::A_STAGE + frag_a;
        const float *Bs = sB + read_slot * T::B_STAGE + frag_b;

        float4 a[2][2], b[2][2];
        a[0][0] = *reinterpret_cast<const float4 *>(As);
        a[0][1] = *reinterpret_cast<const float4 *>(As + 32);
        b[0][0] = *reinterpret_cast<const float4 *>(Bs);
        b[0][1] = *reinterpret_cast<const float4 *>(Bs + 16);
#pragma unroll
        for (int k = 0; k < T::BK; ++k) {
            const int cur = k & 1;
            if (k + 1 < T::BK) {
                const int nxt = cur ^ 1;
                a[nxt][0] = *reinterpret_cast<const float4 *>(As + (k + 1) * T::A_LD);
                a[nxt][1] = *reinterpret_cast<const float4 *>(As + (k + 1) * T::A_LD + 32);
                b[nxt][0] = *reinterpret_cast<const float4 *>(Bs + (k + 1) * T::B_LD);
                b[nxt][1] = *reinterpret_cast<const float4 *>(Bs + (k + 1) * T::B_LD + 16);
            }
            const float av[8] = {a[cur][0].x, a[cur][0].y, a[cur][0].z, a[cur][0].w,
                                 a[cur][1].x, a[cur][1].y, a[cur][1].z, a[cur][1].w};
            const float bv[8] = {b[cur][0].x, b[cur][0].y, b[cur][0].z, b[cur][0].w,
                                 b[cur][1].x, b[cur][1].y, b[cur][1].z, b[cur][1].w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        read_slot = (read_slot + 1 == T::STAGES) ? 0 : read_slot + 1;
        write_slot = (write_slot + 1 == T::STAGES) ? 0 : write_slot + 1;
    }
    cp_async_wait<0>();

    // ---------------------------------------------------------------- epilogue
#pragma unroll
    for (int qm = 0; qm < 2; ++qm) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = m0 + frag_a + qm * 32 + i;
            if (row >= M) continue;
            float *crow = C + (int64_t)row * ldc;
#pragma unroll
            for (int qn = 0; qn < 2; ++qn) {
                const int col = n0 + frag_b + qn * 16;
                const float v[4] = {acc[qm * 4 + i][qn * 4], acc[qm * 4 + i][qn * 4 + 1], acc[qm * 4 + i][qn * 4 + 2],
                                    acc[qm * 4 + i][qn * 4 + 3]};
                store_quad<VEC_C>(crow, col, N, v, alpha, beta);
            }
        }
    }
}

}  // namespace sgemm
