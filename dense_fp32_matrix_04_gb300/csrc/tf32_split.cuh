// The operand split of the 3xTF32 product (memory-bound): each FP32 operand
// becomes a TF32 "high" part and a TF32 "low" part, a_hi = rna_tf32(a) and
// a_lo = rna_tf32(a - a_hi), written K-major for the tensor-core kernel.
#pragma once

#include <cstdint>

#include "tcgen05.cuh"

namespace sgemm {

// One launch splits both operands (A into A_hi, A_lo as M x K rows; B into
// B_hi^T, B_lo^T as N x K rows): its first blocks run A's job, the rest B's.
// A job is a row split of an operand already stored with K along its rows
// (A, or B^T stored N x K) or a transposing split (B, or A^T stored K x M), so
// transposed operands cost no extra pass.
struct SplitJob {
    const float *src;
    int ld;                 // leading dimension of src
    int rows, cols;         // output rows (M or N) and K
    float *hi, *lo;         // outputs, leading dimension ldo (a multiple of 4, 16-byte aligned rows)
    int ldo;
    int transpose;          // 0: src is rows x cols; 1: src is cols x rows
    int vec;                // row split: src rows 16-byte aligned (16-byte loads)
    int gx, gy;             // the job's blocks: gx x gy, block b = (b % gx, b / gx)
};

// Row split, block (bx, by): each thread splits a quad of 4 columns of rows
// by, by + gy, ...: one 16-byte load when the rows allow it, 4-byte loads
// otherwise, and one 16-byte store of each part; columns K .. ldo-1 of the
// output are written as zeros.
__device__ __forceinline__ void split_rows_block(const SplitJob &j, int bx, int by) {
    const int k = 4 * (bx * 256 + (int)threadIdx.x);
    if (k >= j.cols) return;
    for (int i = by; i < j.rows; i += j.gy) {
        const float *a = j.src + (int64_t)i * j.ld + k;
        float v[4];
        if (j.vec && k + 3 < j.cols) {
            const float4 q = *reinterpret_cast<const float4 *>(a);
            v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
        } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) v[t] = k + t < j.cols ? a[t] : 0.f;
        }
        float h[4], l[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            h[t] = to_tf32_rna(v[t]);
            l[t] = to_tf32_rna(v[t] - h[t]);
        }
        *reinterpret_cast<float4 *>(j.hi + (int64_t)i * j.ldo + k) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4 *>(j.lo + (int64_t)i * j.ldo + k) = make_float4(l[0], l[1], l[2], l[3]);
    }
}

// Transposing split, block (bx, by): a 32 x 32 piece of the cols x rows source
// (K x N for B) through a padded 32 x 33 shared tile, written as rows x cols.
__device__ __forceinline__ void split_transpose_block(const SplitJob &j, int bx, int by, float (&th)[32][33],
                                                      float (&tl)[32][33]) {
    const int n0 = bx * 32, k0 = by * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int kk = ty + 8 * r;
        if (k0 + kk < j.cols && n0 + tx < j.rows) {
            const float b = j.src[(int64_t)(k0 + kk) * j.ld + n0 + tx];
            const float h = to_tf32_rna(b);
            th[kk][tx] = h;
            tl[kk][tx] = to_tf32_rna(b - h);
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int nn = ty + 8 * r;
        if (n0 + nn < j.rows && k0 + tx < j.cols) {
            j.hi[(int64_t)(n0 + nn) * j.ldo + k0 + tx] = th[tx][nn];
            j.lo[(int64_t)(n0 + nn) * j.ldo + k0 + tx] = tl[tx][nn];
        }
    }
}

// Blocks [0, ja.gx * ja.gy) run job ja, the next jb.gx * jb.gy blocks job jb
// (256 threads each).
__global__ void __launch_bounds__(256) split_tf32_kernel(const SplitJob ja, const SplitJob jb) {
    __shared__ float th[32][33];
    __shared__ float tl[32][33];
    const int na = ja.gx * ja.gy;
    const bool first = (int)blockIdx.x < na;
    const SplitJob &j = first ? ja : jb;
    const int b = first ? (int)blockIdx.x : (int)blockIdx.x - na;
    const int bx = b % j.gx, by = b / j.gx;
    if (j.transpose) split_transpose_block(j, bx, by, th, tl);
    else split_rows_block(j, bx, by);
}

}  // namespace sgemm
