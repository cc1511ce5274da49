// The pages' own kernel ladder, on the GPU: the naive kernel, the shared-memory
// tiled kernel (unpadded and padded tiles) and the 2-D register-tiled kernel,
// each generalised to M x N x K with strides and boundary masks.  They are the
// reference points the tuned kernels are measured against, and their executed
// global loads are the read counts the pages derive (2MNK naive, 2MNK/T
// tiled), which the counting simulator predicts.
#pragma once

#include <cstdint>

namespace sgemm {

// One thread per output element, K-long dot product straight from global
// memory ("Shared Memory Tiling", 'The naive kernel'; "SGEMM: Shared Memory
// Tiling Visualizer", 'Why exactly 2 x M x N x K for the naive approach?').
__global__ void ladder_naive_kernel(int M, int N, int K, const float *__restrict__ A, int lda,
                                    const float *__restrict__ B, int ldb, float *__restrict__ C, int ldc) {
    const int row = blockIdx.y * blockDim.y + threadIdx.y;
    const int col = blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= M || col >= N) return;
    const float *a = A + (int64_t)row * lda;
    const float *b = B + col;
    float acc = 0.f;
#pragma unroll 1
    for (int k = 0; k < K; ++k) acc = fmaf(a[k], b[(int64_t)k * ldb], acc);
    C[(int64_t)row * ldc + col] = acc;
}

// T x T thread blocks; per tile step each thread loads one element of A and
// one of B into shared memory (zero outside the matrices), then accumulates T
// products; the store is masked ("SGEMM: Shared Memory Tiling Visualizer",
// the tiled kernel; "Shared Memory Tiling", 'The tiled kernel').  PAD = 1
// gives the [T][T + 1] layout of 'Conflict-free layout'.
template <int T, int PAD>
__global__ void __launch_bounds__(T *T) ladder_tiled_kernel(int M, int N, int K, const float *__restrict__ A, int lda,
                                                             const float *__restrict__ B, int ldb,
                                                             float *__restrict__ C, int ldc) {
    __shared__ float tileA[T][T + PAD];
    __shared__ float tileB[T][T + PAD];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int row = blockIdx.y * T + ty;
    const int col = blockIdx.x * T + tx;
    float acc = 0.f;
    const int steps = (K + T - 1) / T;
    for (int t = 0; t < steps; ++t) {
        const int ka = t * T + tx, kb = t * T + ty;
        tileA[ty][tx] = (row < M && ka < K) ? A[(int64_t)row * lda + ka] : 0.f;
        tileB[ty][tx] = (kb < K && col < N) ? B[(int64_t)kb * ldb + col] : 0.f;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < T; ++k) acc = fmaf(tileA[ty][k], tileB[k][tx], acc);
        __syncthreads();
    }
    if (row < M && col < N) C[(int64_t)row * ldc + col] = acc;
}

// The 2-D register-tiled kernel: BM x BN block tiles, BK-deep steps, each of
// the (BM/TM) x (BN/TN) threads keeping a TM x TN block of C and, per k,
// loading TM values of A and TN of B into registers for TM * TN FFMAs
// ("SGEMM: 2D Register Tiling Visualizer", the listing).  Plain loads and
// stores, one barrier pair per step, masks at every edge.
template <int BM, int BN, int BK, int TM, int TN>
__global__ void __launch_bounds__((BM / TM) * (BN / TN))
    ladder_register_kernel(int M, int N, int K, const float *__restrict__ A, int lda, const float *__restrict__ B,
                           int ldb, float *__restrict__ C, int ldc) {
    constexpr int THREADS = (BM / TM) * (BN / TN);
    __shared__ float As[BM][BK];
    __shared__ float Bs[BK][BN];
    const int tid = threadIdx.x;
    const int tm = tid / (BN / TN), tn = tid % (BN / TN);
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int e = tid; e < BM * BK; e += THREADS) {
            const int r = e / BK, c = e % BK;
            As[r][c] = (m0 + r < M && k0 + c < K) ? A[(int64_t)(m0 + r) * lda + k0 + c] : 0.f;
        }
        for (int e = tid; e < BK * BN; e += THREADS) {
            const int r = e / BN, c = e % BN;
            Bs[r][c] = (k0 + r < K && n0 + c < N) ? B[(int64_t)(k0 + r) * ldb + n0 + c] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float regM[TM], regN[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) regM[i] = As[tm * TM + i][k];
#pragma unroll
            for (int j = 0; j < TN; ++j) regN[j] = Bs[k][tn * TN + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(regM[i], regN[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + tm * TM + i;
        if (row >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int col = n0 + tn * TN + j;
            if (col < N) C[(int64_t)row * ldc + col] = acc[i][j];
        }
    }
}

}  // namespace sgemm
