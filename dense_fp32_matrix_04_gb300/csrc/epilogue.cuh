// Output stage shared by the product kernels: C = alpha * acc + beta * C for
// one 4-column quad of one row, masked at the right edge.  beta == 0 never
// reads C (its old contents, NaN included, do not matter); alpha = 1 and
// beta = 0 store the accumulators unchanged.
#pragma once

#include "ptx.cuh"

namespace sgemm {

template <bool VEC_C>
__device__ __forceinline__ void store_quad(float *crow, int col, int N, const float (&v)[4], float alpha, float beta) {
    float o[4];
    if (beta == 0.f) {
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = alpha * v[j];
    } else {
        float c[4];
        if (VEC_C && col + 3 < N) {
            const float4 q = *reinterpret_cast<const float4 *>(crow + col);
            c[0] = q.x, c[1] = q.y, c[2] = q.z, c[3] = q.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) c[j] = col + j < N ? crow[col + j] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = fmaf(alpha, v[j], beta * c[j]);
    }
    if (VEC_C && col + 3 < N) {
        stg128(crow + col, o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (col + j < N) crow[col + j] = o[j];
    }
}

// The same arithmetic for one element: C = alpha * v (beta == 0, C not read)
// or alpha * v + beta * C rounded once.
__device__ __forceinline__ void store_one(float *c, float v, float alpha, float beta) {
    *c = beta == 0.f ? alpha * v : fmaf(alpha, v, beta * *c);
}

// C = beta * C over an M x N block (C = 0 when beta == 0, without reading C):
// the whole product when alpha == 0 or K == 0 leaves nothing to multiply.
__global__ void __launch_bounds__(256) scale_kernel(int M, int N, float beta, float *__restrict__ C, int ldc) {
    const int64_t total = (int64_t)M * N;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = t / N, j = t - i * N;
        float *c = C + i * ldc + j;
        *c = beta == 0.f ? 0.f : beta * *c;
    }
}

// dst[j][i] = src[i][j] for a rows x cols matrix (a plain tiled transpose
// through a padded 32 x 33 shared tile; 32 x 8 threads per block).
__global__ void __launch_bounds__(256) transpose_kernel(int rows, int cols, const float *__restrict__ src, int lds,
                                                        float *__restrict__ dst, int ldd) {
    __shared__ float tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int rr = ty + 8 * r;
        if (r0 + rr < rows && c0 + tx < cols) tile[rr][tx] = src[(int64_t)(r0 + rr) * lds + c0 + tx];
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int cc = ty + 8 * r;
        if (c0 + cc < cols && r0 + tx < rows) dst[(int64_t)(c0 + cc) * ldd + r0 + tx] = tile[tx][cc];
    }
}

}  // namespace sgemm
