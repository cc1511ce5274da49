// Single-k-step FP32 SGEMM (K <= 32) with the tile of C written by the TMA.
//
// A product with one k-step (e.g. 16384 x 16384 x 32) loads each block's A and
// B tiles once, computes briefly and then writes a tile of C that is larger
// than both operand tiles together: the write of C is most of its memory
// traffic ("Shared Memory Tiling": tiling divides the reads of A and B by the
// tile size, but every element of C is written once whatever the tile).
// This kernel keeps the reuse scheme of the TMA-fed kernel -- TMA boxes of A
// and B with hardware zero-fill at the edges, register outer products as
// packed two-wide FMAs -- and changes the end of the block:
//  * 64 threads (two warps of 64 x 64) hold 8 x 16 outputs each, the
//    per-thread tile of the main kernel, in 128 x 64 block tiles;
//  * after the FMAs every thread writes its outputs (times alpha) into a
//    shared tile laid out as two 128-row x 32-column boxes with the TMA's
//    128-byte swizzle, and one thread hands both boxes to the TMA as a bulk
//    tensor store.  The block then only waits until the TMA has read shared
//    memory, not until C reaches memory, so the next block on the SM starts
//    while this block's C is still being written; the TMA store skips the
//    parts of a box outside the M x N matrix, which is the boundary masking of
//    the store.  It clips a row's right edge in 16-byte units (measured: with
//    N = 70 and ldc = 72 it wrote columns 70 and 71 too), so the kernel is
//    used only when N is a multiple of 4.
// Measured on GB300 at 16384 x 16384 x 32 (one product 0.330 ms against
// 0.342 ms with per-thread stores of the same tile and 0.345-0.350 ms for the
// 8 x 8 small-K tile); with no C write at all the same FMAs take 0.281 ms, and
// C's write alone 0.158 ms.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ffma_tma_sgemm.cuh"
#include "ptx.cuh"
#include "tile_map.cuh"

namespace sgemm {

// Make this thread's shared-memory writes visible to the async proxy (a TMA
// store that reads them next).
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// 2-D tiled TMA store of the shared-memory box at `src` to the box at (x, y)
// (x innermost) of the tensor; elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void *tensor_map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];\n" ::"l"(tensor_map),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Wait until every bulk store this thread committed has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }

template <class T>
struct SmallKStore {
    static constexpr int C_BYTES = T::BM * T::BN * 4;           // the C tile, as BN / 32 boxes of BM x 32
    static constexpr int BUF = T::STAGE > C_BYTES ? T::STAGE : C_BYTES;  // operands, then C
    static constexpr int SMEM_BYTES = BUF + 1024 /* alignment */ + 8 /* barrier */;
    static_assert(T::PACKED && T::STAGES == 1 && T::BN % 32 == 0, "one stage, 32-column boxes of C");
    static_assert(T::BM <= 256, "a TMA box spans at most 256 rows");
};

// C = alpha * A B for K <= 32 (one k-step).  tmC: C (N columns x M rows, pitch
// ldc, 16-byte aligned, N a multiple of 4), boxes of 32 x BM with the 128-byte
// swizzle.
template <class T>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
    sgemm_ffma_tma_smallk_store_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                       const __grid_constant__ CUtensorMap tmC, int M, int N, int K, float alpha,
                                       int *__restrict__ err_word, unsigned long long wait_limit_ns, int debug) {
    using S = SmallKStore<T>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 bytes
    unsigned char *smem = smem_raw + (base - raw);
    const uint32_t bar = base + S::BUF;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tiles_m = (M + T::BM - 1) / T::BM, tiles_n = (N + T::BN - 1) / T::BN;
    int tile_m, tile_n;
    grouped_tile<8>(blockIdx.x, tiles_m, tiles_n, tile_m, tile_n);
    const int m0 = tile_m * T::BM, n0 = tile_n * T::BN;

    const bool copies = !(debug & kDebugSkipCopies);
    if (tid == 0) {
        prefetch_tensor_map(&tmA);
        prefetch_tensor_map(&tmB);
        prefetch_tensor_map(&tmC);
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0 && copies) {
        mbar_arrive_expect_tx(bar, T::STAGE);
        tma_load_2d(base, &tmA, 0, m0, bar);
        tma_load_2d(base + T::A_STAGE, &tmB, n0, 0, bar);
    }

    // lane -> (lm, ln) as in the TMA kernel: lm from lane bits {0, 1, 3}, ln from {2, 4}
    const int lm = (lane & 3) | (((lane >> 3) & 1) << 2);
    const int ln = ((lane >> 2) & 1) | (((lane >> 4) & 1) << 1);
    const int row0 = (warp / T::WARPS_N) * T::WM + lm;
    const int col0 = (warp % T::WARPS_N) * T::WN + ln * 4;

    float acc[1][1];
    uint64_t acc2[T::TM][T::TN / 2];
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
#pragma unroll
        for (int j = 0; j < T::TN / 2; ++j) acc2[i][j] = 0ull;

    const bool ok = mbar_wait_bounded(bar, 0, wait_limit_ns);
    if (ok) tile_fma<T>(acc, acc2, smem + row0 * 128, smem + T::A_STAGE + col0 * 4, lm);
    // every warp is done with A and B (or the block gives up together)
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            atomicCAS(err_word, kDeviceErrNone, kDeviceErrTimeout);
            // let the copy land before the block's shared memory is released (bounded)
            if (copies) (void)mbar_wait_bounded(bar, 0, wait_limit_ns);
        }
        __syncthreads();
        return;
    }

    // C tile into shared memory: box b holds columns 32 b .. 32 b + 31 of the
    // tile; 16-byte chunk c of row r sits at chunk c ^ (r % 8) of the row's 128
    // bytes (r % 8 == lm for every row of this thread)
    // alpha * acc + (-0): the product rounded once, with the sign of a zero product kept
    const uint64_t alpha2 = f32x2_dup(alpha), zero2 = 0x8000000080000000ull;
#pragma unroll
    for (int i = 0; i < T::TM; ++i) {
        const int r = row0 + 8 * i;
#pragma unroll
        for (int q = 0; q < T::TN / 4; ++q) {
            const int col = col0 + 16 * q;
            const int c = (col & 31) >> 2;
            uint64_t v0 = zero2, v1 = zero2;
            f32x2_fma(v0, acc2[i][2 * q], alpha2);
            f32x2_fma(v1, acc2[i][2 * q + 1], alpha2);
            *reinterpret_cast<ulonglong2 *>(smem + (col >> 5) * (T::BM * 128) + r * 128 + ((c ^ (r & 7)) << 4)) =
                make_ulonglong2(v0, v1);
        }
    }
    fence_async_shared();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
        for (int b = 0; b < T::BN / 32; ++b)
            if (n0 + 32 * b < N) tma_store_2d(&tmC, base + b * (T::BM * 128), n0 + 32 * b, m0);  // a box past N is skipped
        bulk_commit();
        bulk_wait_read_all();  // shared memory stays in place until the TMA has read it
    }
}

}  // namespace sgemm
