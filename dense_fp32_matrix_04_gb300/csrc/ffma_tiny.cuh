// Products too small for block tiling to pay (a few hundred outputs, short
// k): one thread per element of C with its K-long dot product read straight
// from memory -- the pages' naive kernel ("Shared Memory Tiling", 'The naive
// kernel') -- with alpha and beta.  The tiled kernels spend several
// microseconds per launch on barrier set-up, tensor-map fetches and a copy
// round trip before their first FMA; here the whole product is one short
// launch.  The k terms are added in order with one round-to-nearest FMA each,
// the same per-element arithmetic as every other product kernel, so the bits
// equal theirs whenever no k-split divides the sum.
#pragma once

#include <cstdint>

#include "epilogue.cuh"

namespace sgemm {

// Outputs per block of the tiny kernel (one per thread).
constexpr int kTinyThreads = 256;

// C = alpha * A B + beta * C over M x N (beta == 0 never reads C); element
// e = blockIdx.x * 256 + threadIdx.x is (e / N, e % N).
__global__ void __launch_bounds__(kTinyThreads)
    sgemm_ffma_tiny_kernel(int M, int N, int K, const float *__restrict__ A, int lda, const float *__restrict__ B,
                           int ldb, float *__restrict__ C, int ldc, float alpha, float beta) {
    const int e = blockIdx.x * kTinyThreads + threadIdx.x;
    if (e >= M * N) return;
    const int i = e / N, j = e - (e / N) * N;
    const float *a = A + (int64_t)i * lda;
    const float *b = B + j;
    float acc = 0.f;
#pragma unroll 4
    for (int k = 0; k < K; ++k) acc = fmaf(a[k], b[(int64_t)k * ldb], acc);
    store_one(C + (int64_t)i * ldc + j, acc, alpha, beta);
}

}  // namespace sgemm
