/*
 * CPU oracle for C = A * B (FP32 row-major operands), test infrastructure only.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
 * file; the GPU library never links or calls it, and it shares no code with it.
 *
 * Definition followed: the output element is the length-K dot product of row i
 * of A with column j of B ("SGEMM: Shared Memory Tiling Visualizer", the
 * per-thread partialSum of the tiled kernel; "Shared Memory Tiling", the
 * naive kernel's acc loop), with row-major indexing A[i*lda + k],
 * B[k*ldb + j], C[i*ldc + j].
 *
 * Arithmetic: every FP32 x FP32 product is exact in FP64 (24 + 24 significant
 * bits fit in 53), so the only rounding is the sequential FP64 sum over k,
 * whose error is at most about K * 2^-53 * S[i][j], where
 * S[i][j] = sum_k |A[i][k]| * |B[k][j]| is returned beside the result.  A
 * fused multiply-add in place of the product-then-add gives the same result
 * here, because the product is exact either way.
 *
 * Loop order: i (parallel over rows) then k then j, accumulating into an FP64
 * output row.  Each element still sums its k terms in increasing k.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * C64[i*ldc + j] = sum_k A[i*lda + k] * B[k*ldb + j] in FP64, and, when S is
 * not NULL, S[i*ldc + j] = sum_k |A[i*lda + k]| * |B[k*ldb + j]|.
 * M, N, K >= 0.  C64 and S are M x N with leading dimension ldc.
 */
void oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     double *C64, double *S, int64_t ldc) {
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < M; ++i) {
        double *c = C64 + i * ldc;
        double *s = S ? S + i * ldc : 0;
        int64_t j, k;
        for (j = 0; j < N; ++j) c[j] = 0.0;
        if (s)
            for (j = 0; j < N; ++j) s[j] = 0.0;
        for (k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const float *b = B + k * ldb;
            for (j = 0; j < N; ++j) c[j] += a * (double)b[j];
            if (s) {
                const double aa = fabs(a);
                for (j = 0; j < N; ++j) s[j] += aa * fabs((double)b[j]);
            }
        }
    }
}

/*
 * The same definition for a list of single output elements (rows[t], cols[t]),
 * t < count, for spot checks of products too large to compute in full.
 */
void oracle_gemm_entries(int64_t K,
                         const float *A, int64_t lda,
                         const float *B, int64_t ldb,
                         int64_t count, const int64_t *rows, const int64_t *cols,
                         double *out_c, double *out_s) {
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < count; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double c = 0.0, s = 0.0;
        int64_t k;
        for (k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const double b = (double)B[k * ldb + j];
            c += a * b;
            s += fabs(a) * fabs(b);
        }
        out_c[t] = c;
        if (out_s) out_s[t] = s;
    }
}
