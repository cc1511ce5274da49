// Split-K reduction: C = alpha * (sum over s of the partial products P[s]) +
// beta * C, the sum in increasing s (a fixed order, so the result is the same
// on every run).
//
// P holds S slabs of M rows with leading dimension ldp (a multiple of 4, 16-byte
// aligned base), written by the split-K product kernels.  Memory-bound: it
// reads S * M * N floats and writes M * N.  Each thread sums one 4-column quad
// of one row with 16-byte loads and stores the quad with one 16-byte store
// when C allows it.
#pragma once

#include <cstdint>

#include "epilogue.cuh"

namespace sgemm {

template <bool VEC_C>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(int M, int N, int S, const float *__restrict__ P, int ldp,
                                                            float alpha, float beta, float *__restrict__ C, int ldc) {
    const int64_t quads = (N + 3) / 4;
    const int64_t total = (int64_t)M * quads;
    const int64_t slab = (int64_t)M * ldp;
    for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = q / quads;
        const int j = (int)(q - i * quads) * 4;
        const float *p = P + i * ldp + j;
        float4 acc = *reinterpret_cast<const float4 *>(p);
        for (int s = 1; s < S; ++s) {
            const float4 v = *reinterpret_cast<const float4 *>(p + s * slab);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float v[4] = {acc.x, acc.y, acc.z, acc.w};
        store_quad<VEC_C>(C + i * ldc, j, N, v, alpha, beta);
    }
}

}  // namespace sgemm
