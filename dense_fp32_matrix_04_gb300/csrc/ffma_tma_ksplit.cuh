// A single round of 128 x 64 tiles, one CTA per SM, each tile computed by two
// groups of warps that take alternate k-steps.
//
// Products whose 128 x 64 tiles number a little below the SM count (1024^3:
// 128 tiles for 152 SMs) fill the SMs in a single round of tiles, the case of
// "Shared Memory Tiling" ('What tiling does not fix') where the grid, not the
// tile, decides how busy the SMs are.  Splitting each tile's k-steps over a
// cluster costs more than it gains there (the exchange and a short k-loop per
// CTA), and a plain grid of two-warp CTAs keeps too few warps on each SM to
// cover the latencies of the outer-product loop.  Here each tile is one CTA of two
// groups of two warps that share the TMA ring of the other kernels: of every
// 32-deep k-step, group 0 takes k-values 0-15 and group 1 k-values 16-31,
// each with the packed 8 x 16 outer product of the other TMA kernels.  After
// the k-loop group 1 parks its sums in the (idle) stage buffers and group 0
// adds them to its own, so every element is (sum over the first halves) +
// (sum over the second halves), in a fixed order, and stores the tile with
// the alpha / beta epilogue.  Every wait is bounded; on a timeout the CTA
// records an error code, lets its copies land and writes nothing.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "epilogue.cuh"
#include "ffma_tma_sgemm.cuh"
#include "ptx.cuh"
#include "tile_map.cuh"

namespace sgemm {

// The tile T seen by one group: half of each 32-deep k-step, four groups of
// four k-values (tile_fma walks BK / 4 of them, all unrolled).  The second
// half starts 16 rows into the B stage, and its A chunks 4..7 of a row sit at
// chunk (4 + g) ^ (r % 8) = g ^ ((r % 8) ^ 4) of the 128-byte swizzle, so that
// group passes lm ^ 4 where the first passes lm.
template <class T>
struct HalfK : T {
    static constexpr int BK = T::BK / 2, G_UNROLL = T::BK / 8;
};

// T: the per-group tile (two warps, 128 x 64, packed); the CTA runs 2 * T::THREADS threads.
// PLAIN: alpha = 1 and beta = 0 (C = A B, the arguments are not read), known
// at compile time: with the general epilogue in the kernel the k-loop ran
// 3.4 % slower at 1024^3 (51.6 against 49.9 us, ncu).
template <class T, bool VEC_C, bool PLAIN>
__global__ void __launch_bounds__(2 * T::THREADS, 1)
    sgemm_ffma_tma_ksplit_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                 int M, int N, int K, float alpha, float beta, float *__restrict__ C, int ldc,
                                 int *__restrict__ err_word, unsigned long long wait_limit_ns, int debug) {
    static_assert(T::PACKED, "group 1 hands over packed accumulators");
    static_assert(T::BK == 32, "two halves of four 4-deep k-groups; chunks 4..7 of a 128-byte row");
    static_assert(T::TM * T::TN * T::THREADS * 4 <= T::STAGES * T::STAGE, "group 1 parks its sums in the stages");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the 128-byte swizzle pattern repeats every 1024 bytes
    unsigned char *smem = smem_raw + (base - raw);
    const uint32_t bars = base + T::STAGES * T::STAGE;

    const int tid = threadIdx.x;
    const int group = tid / T::THREADS;  // 0 or 1: which k-steps
    const int t = tid - group * T::THREADS;
    const int lane = t & 31;
    const int warp = t >> 5;

    const int tiles_m = (M + T::BM - 1) / T::BM;
    const int tiles_n = (N + T::BN - 1) / T::BN;
    int tile_m, tile_n;
    grouped_tile<8>((int)blockIdx.x, tiles_m, tiles_n, tile_m, tile_n);
    const int m0 = tile_m * T::BM;
    const int n0 = tile_n * T::BN;
    const int KT = (K + T::BK - 1) / T::BK;

    if (tid == 0) {
        prefetch_tensor_map(&tmA);
        prefetch_tensor_map(&tmB);
#pragma unroll
        for (int s = 0; s < T::STAGES; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // k-step kt into stage kt % STAGES
    auto issue = [&](int kt) {
        const int s = kt % T::STAGES;
        const uint32_t bar = bars + 8 * s;
        const uint32_t dst = base + s * T::STAGE;
        mbar_arrive_expect_tx(bar, T::STAGE);
        tma_load_2d(dst, &tmA, kt * T::BK, m0, bar);
        tma_load_2d(dst + T::A_STAGE, &tmB, n0, kt * T::BK, bar);
    };
    const bool copies = !(debug & kDebugSkipCopies);
    if (tid == 0 && copies)
        for (int kt = 0; kt < KT && kt < T::STAGES; ++kt) issue(kt);

    const int lm = (lane & 3) | (((lane >> 3) & 1) << 2);
    const int ln = ((lane >> 2) & 1) | (((lane >> 4) & 1) << 1);
    const int row0 = (warp / T::WARPS_N) * T::WM + lm;
    const int col0 = (warp % T::WARPS_N) * T::WN + ln * 4;

    float acc[1][1];  // unused: the packed form keeps acc2
    uint64_t acc2[T::TM][T::TN / 2];
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
#pragma unroll
        for (int j = 0; j < T::TN / 2; ++j) acc2[i][j] = 0ull;

    // this group's half of every k-step: B rows 16 * group on, A chunks through lm ^ (4 * group)
    const int lm_half = lm ^ (4 * group);
    const int b_half = group * (T::BK / 2) * (T::BN * 4);
    int failed_k0 = -1;
    for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % T::STAGES;
        const bool ok = mbar_wait_bounded(bars + 8 * s, (kt / T::STAGES) & 1, wait_limit_ns);
        if (ok) {
            const unsigned char *stage = smem + s * T::STAGE;
            tile_fma<HalfK<T>>(acc, acc2, stage + row0 * 128, stage + T::A_STAGE + b_half + col0 * 4, lm_half);
        }
        // both groups are done with stage s (or give up together)
        if (__syncthreads_or(!ok)) {
            failed_k0 = kt;
            break;
        }
        if (tid == 0 && copies && kt + T::STAGES < KT) issue(kt + T::STAGES);
    }

    if (failed_k0 >= 0) {
        if (tid == 0) {
            atomicCAS(err_word, kDeviceErrNone, kDeviceErrTimeout);
            // let the copies already issued (k-steps failed_k0 .. failed_k0 + STAGES - 1)
            // land before the CTA's shared memory is released; bounded as well
            if (copies)
                for (int kt = failed_k0; kt < KT && kt < failed_k0 + T::STAGES; ++kt)
                    (void)mbar_wait_bounded(bars + 8 * (kt % T::STAGES), (kt / T::STAGES) & 1, wait_limit_ns);
        }
        return;
    }

    // 16-byte chunk (i, q) of thread t at ((i * TN/4 + q) * THREADS + t) * 16
    if (group == 1) {
#pragma unroll
        for (int i = 0; i < T::TM; ++i)
#pragma unroll
            for (int q = 0; q < T::TN / 4; ++q)
                *reinterpret_cast<ulonglong2 *>(smem + ((i * (T::TN / 4) + q) * T::THREADS + t) * 16) =
                    make_ulonglong2(acc2[i][2 * q], acc2[i][2 * q + 1]);
    }
    __syncthreads();
    if (group == 1) return;
    const uint64_t one2 = f32x2_dup(1.f);
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
#pragma unroll
        for (int q = 0; q < T::TN / 4; ++q) {
            const ulonglong2 v =
                *reinterpret_cast<const ulonglong2 *>(smem + ((i * (T::TN / 4) + q) * T::THREADS + t) * 16);
            f32x2_fma(acc2[i][2 * q], v.x, one2);  // s + v, rounded once (v * 1 is exact)
            f32x2_fma(acc2[i][2 * q + 1], v.y, one2);
        }
    store_tile<T, VEC_C, false>(acc, acc2, C, ldc, M, N, m0 + row0, n0 + col0, PLAIN ? 1.f : alpha, PLAIN ? 0.f : beta,
                                1, 0);
}

}  // namespace sgemm
