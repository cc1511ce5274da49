// Stream-K form of the TMA-fed FFMA kernel, for products whose tiles would
// leave SMs idle (e.g. 256 x 256 x 65536: 4 tiles of 128 x 128 for 152 SMs).
//
// "Shared Memory Tiling" ('What tiling does not fix') names the load
// imbalance left when the tiles do not divide evenly over the SMs.  Here the
// work is not dealt out in tiles but in k-steps: the product is the linear
// sequence of units (tile t, k-step k), tile-major over the grouped tile
// raster, and the grid -- exactly the CTAs that are resident at once, so that
// every SM gets the same share -- gives CTA c the units
// [floor(U c / G), floor(U (c + 1) / G)) of the U units.  A CTA walks its
// units through the same TMA pipeline and packed FFMA loop as the plain kernel,
// prefetching across tile boundaries, and at the end of each run of units
// that share a tile (a segment):
//  * a segment covering the whole tile stores it (alpha, beta epilogue);
//  * otherwise the CTA writes its partial tile to its own slot of the
//    workspace and counts itself in on the tile's counter.
// When its run is done, a CTA waits (bounded) until every contributor of each
// tile it shares has counted in, then adds up its own slice of that tile:
// contributor j of n takes the 16-byte chunks [4096 j / n, 4096 (j + 1) / n)
// and sums them over the n partial tiles in a fixed order -- k order, or, when
// the slice is narrower than the CTA, k order within P groups of consecutive
// contributors and then the P group sums in order -- and stores them.  The
// order depends only on the shape, so every run gives the same bits, and the
// whole grid shares the fix-up instead of one CTA per tile.  A CTA writes all
// of its partial tiles before it waits on anything, and the grid is launched
// cooperatively (every CTA resident at once), so every wait ends.
// Each CTA has at most two partial segments (its first and its last), so the
// workspace holds two partial tiles per CTA, plus one counter per tile that
// the host zeroes before the launch.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "epilogue.cuh"
#include "ffma_tma_sgemm.cuh"
#include "ptx.cuh"
#include "tile_map.cuh"

namespace sgemm {

// CTA that owns unit u when U units are dealt to G CTAs in contiguous runs
// [floor(U c / G), floor(U (c + 1) / G)).
__device__ __forceinline__ int64_t streamk_cta_of(int64_t u, int64_t U, int64_t G) { return ((u + 1) * G - 1) / U; }

__device__ __forceinline__ int64_t streamk_begin(int64_t c, int64_t U, int64_t G) { return U * c / G; }

// Byte offset of accumulator chunk (i, q) of thread tid inside a partial
// tile: each 16-byte chunk (pairs 2q, 2q + 1 of row i) of all threads lies
// together, so a warp's store or load is 512 contiguous bytes.
template <class T>
__device__ __forceinline__ int64_t streamk_chunk(int i, int q, int tid) {
    return ((int64_t)(i * (T::TN / 4) + q) * T::THREADS + tid) * 16;
}

// Thread 0 of a CTA: wait until *count reaches n (every contributor of a
// shared tile has counted in), at most limit_ns; true if it did.  The load
// after the count has been seen is ordered before the CTA's reads of the
// partial tiles by the fence and the CTA barrier that follow.
__device__ __forceinline__ bool wait_count_bounded(const int *count, int n, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(count) : "memory");
        if (v >= n) {
            __threadfence();
            return v == n;
        }
        if (global_timer_ns() - t0 > limit_ns) return false;
        __nanosleep(64);
    }
}

// Contributor j of the n CTAs that share a tile: add up its slice of the
// tile's 16-byte accumulator chunks over the n partial tiles (the first at
// slot slot0, then the first slots of CTAs cf + 1, ..., cf + n - 1, in k
// order) and store C = alpha * sum + beta * C there.  With fewer chunks in
// the slice (m) than threads, P = THREADS / m groups of consecutive partial
// tiles are summed side by side (each in k order) and the P sums are then
// added in group order through `red` (P * m <= THREADS float4s); the order
// depends only on (n, j), never on timing.  (tile_r, tile_c) is the tile's
// corner in C.
template <class T, bool VEC_C>
__device__ __forceinline__ void streamk_fixup(const unsigned char *__restrict__ slots, int slot0, int cf, int n, int j,
                                              float4 *red, int tile_r, int tile_c, float *__restrict__ C, int ldc,
                                              int M, int N, float alpha, float beta) {
    constexpr int64_t SLOT = (int64_t)T::BM * T::BN * 4;
    constexpr int CHUNKS = T::TM * (T::TN / 4) * T::THREADS;
    const int lo = (int)((int64_t)CHUNKS * j / n), hi = (int)((int64_t)CHUNKS * (j + 1) / n);
    const int m = hi - lo;
    if (m <= 0) return;
    const int tid = threadIdx.x;
    int P = m >= T::THREADS ? 1 : T::THREADS / m;
    if (P > n) P = n;
    // chunk g of a partial tile: accumulator chunk (i, q) of thread g % THREADS
    auto part = [&](int r, int g) -> float4 {
        const int64_t slot = r == 0 ? slot0 : 2 * (int64_t)(cf + r);
        return __ldcg(reinterpret_cast<const float4 *>(slots + slot * SLOT + (int64_t)g * 16));
    };
    auto store = [&](int g, float4 v) {
        const int th = g % T::THREADS, iq = g / T::THREADS;
        const int i = iq / (T::TN / 4), q = iq % (T::TN / 4);
        const int lane = th & 31, warp = th >> 5;
        const int lm = (lane & 3) | (((lane >> 3) & 1) << 2);
        const int ln = ((lane >> 2) & 1) | (((lane >> 4) & 1) << 1);
        const int row = tile_r + (warp / T::WARPS_N) * T::WM + lm + 8 * i;
        const int col = tile_c + (warp % T::WARPS_N) * T::WN + ln * 4 + 16 * q;
        if (row >= M) return;
        const float vp[4] = {v.x, v.y, v.z, v.w};
        store_quad<VEC_C>(C + (int64_t)row * ldc, col, N, vp, alpha, beta);
    };
    auto add = [](float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); };
    if (P == 1) {
        for (int g = lo + tid; g < hi; g += T::THREADS) {
            float4 v = part(0, g);
#pragma unroll 8
            for (int r = 1; r < n; ++r) v = add(v, part(r, g));
            store(g, v);
        }
        return;
    }
    if (tid < P * m) {
        const int g = lo + tid % m, p = tid / m;
        const int r0 = n * p / P, r1 = n * (p + 1) / P;
        float4 v = part(r0, g);
#pragma unroll 8
        for (int r = r0 + 1; r < r1; ++r) v = add(v, part(r, g));
        red[p * m + tid % m] = v;
    }
    __syncthreads();
    if (tid < m) {
        float4 v = red[tid];
        for (int p = 1; p < P; ++p) v = add(v, red[p * m + tid]);
        store(lo + tid, v);
    }
}

template <class T, bool VEC_C>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
    sgemm_ffma_tma_streamk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                  int M, int N, int K, float alpha, float beta, float *__restrict__ C, int ldc,
                                  int *__restrict__ counters, unsigned char *__restrict__ slots, int *__restrict__ err_word,
                                  unsigned long long wait_limit_ns, int debug) {
    static_assert(T::PACKED, "the partial tiles are the packed accumulators");
    constexpr int64_t SLOT = (int64_t)T::BM * T::BN * 4;
    extern __shared__ unsigned char smem_raw[];
    // values the k-loop does not need, kept out of its registers: the wait's
    // outcome, the partial tiles' bookkeeping, and thread 0's copy cursor
    __shared__ int last_flag;
    __shared__ int info[4];        // cf_a, nseg_a, slot_a, nseg_b
    __shared__ int cursor[4];      // t_iss, k_iss, tm_iss, tn_iss
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);
    const uint32_t bars = base + T::STAGES * T::STAGE;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int tiles_m = (M + T::BM - 1) / T::BM;
    const int tiles_n = (N + T::BN - 1) / T::BN;
    const int kt = (K + T::BK - 1) / T::BK;
    const int64_t G = gridDim.x;
    const int64_t U = (int64_t)tiles_m * tiles_n * kt;
    const int64_t c = blockIdx.x;
    const int64_t u0 = streamk_begin(c, U, G), u1 = streamk_begin(c + 1, U, G);
    if (u0 >= u1) return;
    const int n_units = (int)(u1 - u0);
    // Where this CTA's run starts and ends, and what the (at most two) partial
    // tiles it shares need at the end: the first contributing CTA, the number
    // of segments, and the slot of the first segment.  All the 64-bit
    // divisions happen here, once.
    const int t_first = (int)(u0 / kt), k_first = (int)(u0 - (int64_t)t_first * kt);
    const int t_last = (int)((u1 - 1) / kt);
    if (tid == 0) {
        const int64_t tb = (int64_t)t_first * kt;
        const int64_t cf = k_first == 0 ? c : streamk_cta_of(tb, U, G);
        info[0] = (int)cf;
        info[1] = (int)(streamk_cta_of(tb + kt - 1, U, G) - cf + 1);
        info[2] = (int)(2 * cf + (streamk_begin(cf, U, G) < tb ? 1 : 0));
        // the last tile, when another: this CTA is its first contributor (from its k = 0)
        info[3] = t_last != t_first ? (int)(streamk_cta_of((int64_t)(t_last + 1) * kt - 1, U, G) - c + 1) : 0;
        cursor[0] = t_first;
        cursor[1] = k_first;
        grouped_tile<8>(t_first, tiles_m, tiles_n, cursor[2], cursor[3]);
        prefetch_tensor_map(&tmA);
        prefetch_tensor_map(&tmB);
#pragma unroll
        for (int s = 0; s < T::STAGES; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // thread 0's copy cursor: the next unit to load is k-step cursor[1] of
    // tile cursor[0], at tile coordinates (cursor[2], cursor[3])
    auto issue = [&](int s) {
        const uint32_t bar = bars + 8 * s;
        const uint32_t dst = base + s * T::STAGE;
        const int k_iss = cursor[1];
        mbar_arrive_expect_tx(bar, T::STAGE);
        tma_load_2d(dst, &tmA, k_iss * T::BK, cursor[2] * T::BM, bar);
        tma_load_2d(dst + T::A_STAGE, &tmB, cursor[3] * T::BN, k_iss * T::BK, bar);
        if (k_iss + 1 == kt) {
            cursor[1] = 0;
            const int t_iss = ++cursor[0];
            grouped_tile<8>(t_iss, tiles_m, tiles_n, cursor[2], cursor[3]);
        } else {
            cursor[1] = k_iss + 1;
        }
    };
    const bool copies = !(debug & kDebugSkipCopies);
    if (tid == 0 && copies) {
        const int pre = n_units < T::STAGES ? n_units : T::STAGES;
        for (int s = 0; s < pre; ++s) issue(s);
    }

    const int lm = (lane & 3) | (((lane >> 3) & 1) << 2);
    const int ln = ((lane >> 2) & 1) | (((lane >> 4) & 1) << 1);
    const int warp_m = warp / T::WARPS_N;
    const int warp_n = warp % T::WARPS_N;
    const int row0 = warp_m * T::WM + lm;
    const int col0 = warp_n * T::WN + ln * 4;

    float acc[1][1];
    uint64_t acc2[T::TM][T::TN / 2];
    int it = 0;
    int failed_it = -1;
    int t = t_first, k = k_first;
    int parts = 0;  // bit 0: the first tile is shared (written, counted); bit 1: the last one
    while (it < n_units) {
        const int seg = min(kt - k, n_units - it);
#pragma unroll
        for (int i = 0; i < T::TM; ++i)
#pragma unroll
            for (int j = 0; j < T::TN / 2; ++j) acc2[i][j] = 0ull;
        for (int e = it + seg; it < e; ++it) {
            const int s = it % T::STAGES;
            const bool ok = mbar_wait_bounded(bars + 8 * s, (it / T::STAGES) & 1, wait_limit_ns);
            if (ok) {
                const unsigned char *sa = smem + s * T::STAGE + row0 * 128;
                const unsigned char *sb = smem + s * T::STAGE + T::A_STAGE + col0 * 4;
                tile_fma<T>(acc, acc2, sa, sb, lm);
            }
            if (__syncthreads_or(!ok)) {
                failed_it = it;
                break;
            }
            if (tid == 0 && copies && it + T::STAGES < n_units) issue(s);
        }
        if (failed_it >= 0) break;

        int tm, tn;
        grouped_tile<8>(t, tiles_m, tiles_n, tm, tn);
        const int r0 = tm * T::BM + row0, c0 = tn * T::BN + col0;
        const bool whole = seg == kt;
        const bool first_seg = t == t_first;
        ++t;
        k = 0;
        if (whole) {
            store_tile<T, VEC_C, false>(acc, acc2, C, ldc, M, N, r0, c0, alpha, beta, 1, 0);
            continue;
        }
        // a partial tile: into this CTA's slot (its first segment: slot 2c; its last: 2c + 1)
        unsigned char *mine = slots + (2 * c + (first_seg ? 0 : 1)) * SLOT + tid * 16;
#pragma unroll
        for (int i = 0; i < T::TM; ++i)
#pragma unroll
            for (int q = 0; q < T::TN / 4; ++q)
                __stcg(reinterpret_cast<ulonglong2 *>(mine + (i * (T::TN / 4) + q) * T::THREADS * 16),
                       make_ulonglong2(acc2[i][2 * q], acc2[i][2 * q + 1]));
        __threadfence();
        __syncthreads();
        if (tid == 0) atomicAdd(counters + (t - 1), 1);
        parts |= first_seg ? 1 : 2;
    }

    // every partial tile of this CTA is written and counted: add up this
    // CTA's slice of each, once all of the tile's contributors have counted in
    bool gave_up = false;
    if (failed_it < 0) {
        float4 *red = reinterpret_cast<float4 *>(smem);  // the stage buffers are idle now
        for (int which = 0; which < 2; ++which) {
            if (!(parts & (1 << which))) continue;
            const int tt = which == 0 ? t_first : t_last;
            const int cf = which == 0 ? info[0] : (int)c;
            const int n_seg = which == 0 ? info[1] : info[3];
            const int slot0 = which == 0 ? info[2] : (int)(2 * c + 1);
            if (tid == 0) last_flag = wait_count_bounded(counters + tt, n_seg, wait_limit_ns);
            __syncthreads();
            if (!last_flag) {
                gave_up = true;
                break;
            }
            int tm, tn;
            grouped_tile<8>(tt, tiles_m, tiles_n, tm, tn);
            streamk_fixup<T, VEC_C>(slots, slot0, cf, n_seg, (int)c - cf, red, tm * T::BM, tn * T::BN, C, ldc, M, N,
                                    alpha, beta);
            __syncthreads();  // red is reused for the second tile
        }
    }
    if (gave_up && tid == 0) atomicCAS(err_word, kDeviceErrNone, kDeviceErrTimeout);

    if (failed_it >= 0 && tid == 0) {
        atomicCAS(err_word, kDeviceErrNone, kDeviceErrTimeout);
        // let the copies already issued land before the CTA's shared memory is released
        if (copies)
            for (int i = failed_it; i < n_units && i < failed_it + T::STAGES; ++i)
                (void)mbar_wait_bounded(bars + 8 * (i % T::STAGES), (i / T::STAGES) & 1, wait_limit_ns);
    }
}

}  // namespace sgemm
