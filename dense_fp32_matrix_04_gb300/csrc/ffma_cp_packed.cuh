// Register-tiled FP32 SGEMM for operands the tensor memory accelerator cannot
// address (a base or leading dimension that is not a multiple of 16 bytes,
// e.g. lda = 2047): the TMA kernel's tile, fragment reads, packed two-wide
// FMAs, epilogue and cluster split, fed by cp.async copies that every thread
// issues instead of TMA boxes.
//
//  * Copies: per k-step, the 128 x 32 slab of A and the 32 x BN slab of B
//    (BN = 128, or 64 for the narrow tile) move by cp.async into the same
//    shared-memory layout the TMA writes (A in 128-byte rows with the 128-byte
//    swizzle, chunk c of row r at c ^ (r % 8); B dense), so the arithmetic is
//    the TMA kernel's own (tile_fma).  A warp copies one row of 32 consecutive
//    k of A, or 32 consecutive columns of a row of B, with 4-byte copies
//    (coalesced 128-byte requests); when an operand's rows are 16-byte aligned
//    it uses 16-byte copies instead.
//  * Masking: slots outside A or B are zero-filled by the copy itself (source
//    size 0, no global read) -- the pages' masked tile loads ("SGEMM: Shared
//    Memory Tiling Visualizer", the tiled kernel listing).  Most copies need
//    no mask at all: a last, partial row tile reads the 128 rows that end at
//    row M (and stores only its own), and B's right edge is a per-thread copy
//    size, so only the last, partial k-step and products with M < 128 take
//    the masked path.
//  * Pipeline: STAGES slabs in flight as cp.async groups, one CTA barrier per
//    k-step; the copy of step t + STAGES - 1 overlaps the FMAs of step t
//    ("Shared Memory Tiling", 'What tiling does not fix').  With 4-byte
//    copies of A, the unmasked copies go out an eighth at a time between the
//    groups of FMAs instead of in one burst.
//  * No bounded waits are needed: cp.async groups complete on their own.
#pragma once

#include <cstdint>
#include <type_traits>

#include "ffma_tma_sgemm.cuh"

namespace sgemm {

// VEC_A / VEC_B: that operand's base and leading dimension are multiples of 16
// bytes (16-byte copies); otherwise 4-byte copies.
// vec_c: C's base and leading dimension allow 16-byte stores (a run-time flag
// here, to halve the number of instances).
template <class T, bool VEC_A, bool VEC_B, int ROLE = kRolePlain>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
    sgemm_ffma_cp_kernel(int M, int N, int K, float alpha, const float *__restrict__ A, int lda,
                         const float *__restrict__ B, int ldb, float beta, float *__restrict__ C, int ldc,
                         int vec_c, float *__restrict__ partials, int ldp, int tile_base) {
    constexpr bool CSPLIT = ROLE == kRoleSplit;
    // 4-byte copies of A are spread through the FMAs of the step before (32 per
    // thread and step otherwise come in one burst).  16-byte copies of A, and
    // the cluster split's short k-ranges (a quarter of whose steps issue no
    // copy, so both loop bodies would be live in the SM's instruction cache),
    // measured faster in one burst.
    constexpr bool SPREAD = !VEC_A && ROLE != kRoleSplit;
    static_assert(T::PACKED && T::THREADS == 128 && T::BM == 128 && (T::BN == 128 || T::BN == 64) && T::BK == 32,
                  "the copy roles below are laid out for 128 threads and 128 x 128 x 32 or 128 x 64 x 32 tiles");
    static_assert(T::STAGES >= 2, "the cp.async pipeline needs two stages");
    static_assert(!CSPLIT || T::CSPLIT_OK, "the cluster split exchanges packed accumulators through the stage buffers");
    if constexpr (ROLE == kRolePrimary) griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment: the swizzle pattern repeats every 8 rows of 128 bytes
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);

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
    // The copies read rows m0c .. m0c + BM - 1 of A: a last, partial row tile is
    // moved up to end at row M (when M >= BM), so that none of its copies needs
    // a row mask; the rows it then covers twice are left to the tile above.
    const bool shift_m = M >= T::BM;
    const int m0c = shift_m ? min(m0, M - T::BM) : m0;
    // split-K by CTA row (partial slabs) or by cluster rank, as in the TMA kernel
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

    // ---------------------------------------------------------------- copy roles
    // A, 4-byte: warp w copies rows w + 4 j (j < 32), lane = k within the step.
    // A, 16-byte: rows 16 j + 4 w + lane / 8 (j < 8), 16-byte chunk lane % 8.
    // Shared address of (row r, k) = r * 128 + ((k / 4) ^ (r % 8)) * 16 + (k % 4) * 4;
    // r % 8 takes two values over a thread's 4-byte copies (rows w + 4 j) and one
    // over its 16-byte copies (rows 4 w + lane / 8 + 16 j), so the shared
    // addresses are a per-thread base plus a constant per copy.
    constexpr int A_COPIES = VEC_A ? 8 : 32;
    const int a_row0 = VEC_A ? 4 * warp + (lane >> 3) : warp;
    constexpr int A_ROW_STEP = VEC_A ? 16 : 4;
    const int a_k = VEC_A ? (lane & 7) * 4 : lane;
    const float *gA = A + (int64_t)(m0c + a_row0) * lda + a_k;
    const int a_step = A_ROW_STEP * lda;  // fits an int: the host checks A_ROW_STEP * lda
    // shared offsets of copy 0 and (4-byte copies) copy 1; copy j adds
    // (j / 2) * 1024 (4-byte) or j * 2048 (16-byte) to the one of its parity
    auto a_off = [&](int r) { return (uint32_t)(r * 128 + ((((a_k >> 2) ^ (r & 7))) << 4) + (VEC_A ? 0 : (a_k & 3) * 4)); };
    const uint32_t a_off0 = a_off(a_row0), a_off1 = a_off(a_row0 + A_ROW_STEP);
    // B, 4-byte: a warp copies 32 consecutive columns of one k-row per copy;
    // the BN / 32 warps of a k-row (W) take columns 32 (w % W) + lane of k-rows
    // w / W + (4 / W) j.  16-byte: a warp copies 32 / (BN / 4) k-rows of BN
    // columns per copy, lane l taking the 16-byte chunk l % (BN / 4) of its row.
    // A thread's columns are the same in every k-step, so the right edge is a
    // per-thread copy size (zero past column N, from a column inside B).
    constexpr int B_WARPS_PER_ROW = T::BN / 32;
    constexpr int B_CHUNKS_PER_ROW = T::BN / 4;
    constexpr int B_KROW_STEP = VEC_B ? 4 * (32 / B_CHUNKS_PER_ROW) : 4 / B_WARPS_PER_ROW;
    constexpr int B_COPIES = 32 / B_KROW_STEP;
    const int b_col = VEC_B ? 4 * (lane % B_CHUNKS_PER_ROW) : 32 * (warp % B_WARPS_PER_ROW) + lane;
    const int b_krow0 = VEC_B ? lane / B_CHUNKS_PER_ROW + (32 / B_CHUNKS_PER_ROW) * warp : warp / B_WARPS_PER_ROW;
    const int b_left = N - (n0 + b_col);
    const int b_bytes = VEC_B ? (b_left >= 4 ? 16 : (b_left > 0 ? 4 * b_left : 0)) : (b_left > 0 ? 4 : 0);
    const float *gB = B + (int64_t)b_krow0 * ldb + (b_left > 0 ? n0 + b_col : 0);
    const int b_step = B_KROW_STEP * ldb;  // likewise
    const uint32_t b_off0 = (uint32_t)(T::A_STAGE + b_krow0 * (T::BN * 4) + b_col * 4);

    // Issue copies of k-step kt (counted from kt_begin) into stage s: group grp
    // of NG equal groups.  FULL: the step's 32 k lie inside K and the rows of A
    // inside M, so only B's per-thread size masks anything.
    auto issue_impl = [&](auto full_tag, auto ng_tag, int kt, int s, int grp) {
        constexpr bool FULL = decltype(full_tag)::value;
        constexpr int NG = decltype(ng_tag)::value;
        const int k0 = (kt_begin + kt) * T::BK;
        const uint32_t st = base + s * T::STAGE;
        {
            const float *src = gA + k0;
            int a_bytes = VEC_A ? 16 : 4;
            if constexpr (!FULL) {
                if constexpr (VEC_A) {
                    const int left = K - (k0 + a_k);
                    a_bytes = left >= 4 ? 16 : (left > 0 ? 4 * left : 0);
                } else {
                    a_bytes = k0 + a_k < K ? 4 : 0;
                }
            }
#pragma unroll
            for (int jj = 0; jj < A_COPIES / NG; ++jj) {
                const int j = grp * (A_COPIES / NG) + jj;
                const uint32_t dst =
                    st + (VEC_A ? a_off0 + j * 2048 : ((jj & 1) ? a_off1 : a_off0) + (j >> 1) * 1024);
                const float *g = src + (int64_t)j * a_step;
                if constexpr (FULL) {
                    if constexpr (VEC_A) cp_async_16(dst, g, 16);
                    else cp_async_4(dst, g, 4);
                } else {
                    const int bytes = m0c + a_row0 + j * A_ROW_STEP < M ? a_bytes : 0;
                    const void *gg = bytes ? (const void *)g : (const void *)A;
                    if constexpr (VEC_A) cp_async_16(dst, gg, bytes);
                    else cp_async_4(dst, gg, bytes);
                }
            }
        }
        {
            const float *src = gB + (int64_t)k0 * ldb;
            // with fewer copies than groups, group g < B_COPIES takes copy g
            constexpr int BPG = B_COPIES >= NG ? B_COPIES / NG : 1;
#pragma unroll
            for (int jj = 0; jj < BPG; ++jj) {
                const int j = grp * BPG + jj;
                if (B_COPIES < NG && j >= B_COPIES) break;
                const uint32_t dst = st + b_off0 + j * B_KROW_STEP * (T::BN * 4);
                const float *g = src + (int64_t)j * b_step;
                if constexpr (FULL) {
                    if constexpr (VEC_B) cp_async_16(dst, g, b_bytes);
                    else cp_async_4(dst, g, b_bytes);
                } else {
                    const int kr = b_krow0 + j * B_KROW_STEP;
                    const int bytes = k0 + kr < K ? b_bytes : 0;
                    const void *gg = bytes ? (const void *)g : (const void *)B;
                    if constexpr (VEC_B) cp_async_16(dst, gg, bytes);
                    else cp_async_4(dst, gg, bytes);
                }
            }
        }
    };
    // steps 0 .. kt_full - 1 are FULL
    const int kt_full = shift_m ? min(KT, K / T::BK - kt_begin) : 0;
    auto full_step = [&](int kt) { return kt < kt_full; };
    auto issue = [&](int kt, int s) {
        if (full_step(kt)) issue_impl(std::true_type{}, std::integral_constant<int, 1>{}, kt, s, 0);
        else issue_impl(std::false_type{}, std::integral_constant<int, 1>{}, kt, s, 0);
    };

    // ---------------------------------------------------------------- compute roles (as the TMA kernel)
    const int lm = (lane & 3) | (((lane >> 3) & 1) << 2);
    const int ln = ((lane >> 2) & 1) | (((lane >> 4) & 1) << 1);
    const int warp_m = warp / T::WARPS_N;
    const int warp_n = warp % T::WARPS_N;
    const int row0 = warp_m * T::WM + lm;
    const int col0 = warp_n * T::WN + ln * 4;

    float acc[1][1];
    uint64_t acc2[T::TM][T::TN / 2];
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
#pragma unroll
        for (int j = 0; j < T::TN / 2; ++j) acc2[i][j] = 0ull;

    // prologue: STAGES - 1 steps in flight (empty groups past the end keep the count)
#pragma unroll
    for (int s = 0; s < T::STAGES - 1; ++s) {
        if (s < KT) issue(s, s);
        cp_async_commit();
    }
    for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % T::STAGES;
        // step kt has landed for this thread; the barrier makes it every thread's,
        // and frees the stage read in step kt - 1 for the copies issued below
        cp_async_wait<T::STAGES - 2>();
        __syncthreads();
        const int next = kt + T::STAGES - 1;
        const int sn = next % T::STAGES;
        const unsigned char *sa = smem + s * T::STAGE + row0 * 128;
        const unsigned char *sb = smem + s * T::STAGE + T::A_STAGE + col0 * 4;
        if (SPREAD && next < KT && full_step(next)) {
            // the copies of step `next`, an eighth before each group of four k
            tile_fma<T>(acc, acc2, sa, sb, lm, [&](int g) {
                issue_impl(std::true_type{}, std::integral_constant<int, 8>{}, next, sn, g);
            });
        } else {
            if (next < KT) issue(next, sn);
            tile_fma<T>(acc, acc2, sa, sb, lm);
        }
        cp_async_commit();
    }
    // no copy in flight, every warp done with the stage buffers
    cp_async_wait<0>();
    __syncthreads();

    if constexpr (CSPLIT) {
        if (cluster_reduce<T>(acc2, base, smem, tid, cs, rank, false)) {
            griddep_wait();
            return;
        }
    }
    // rows m0c .. m0 - 1 of a moved-up tile belong to the tile above
    if (vec_c) store_tile<T, true, CSPLIT>(acc, acc2, C, ldc, M, N, m0c + row0, n0 + col0, alpha, beta, cs, rank, m0);
    else store_tile<T, false, CSPLIT>(acc, acc2, C, ldc, M, N, m0c + row0, n0 + col0, alpha, beta, cs, rank, m0);
    if constexpr (CSPLIT) griddep_wait();
}

}  // namespace sgemm
