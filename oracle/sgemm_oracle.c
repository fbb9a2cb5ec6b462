/*
 * FP64 reference for single-precision GEMM — TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline / reference
 * arm may call this file. The GPU library never links it, and it shares no
 * code, header or table with the GPU library.
 *
 * What it computes is the problem statement itself:
 *
 *     C_out = alpha * A * B + beta * C_in
 *
 * with A (M x K), B (K x N), C (M x N), all row-major, element (i, j) of a
 * matrix with leading dimension ld at offset i*ld + j
 *   - "SGEMM CUDA kernel (First Half)", opening definition (S = single
 *     precision, GEMM: C = alpha AB + beta C; A is M x K, B is K x N);
 *   - same page, "Part 1: CPU version" (row-major OFFSET(row, col) =
 *     row * ncols + col, one dot product of length K per output);
 *   - "Optimizing Matrix Multiplication in CUDA", "Baseline CPU
 *     Implementation" (c[i*n + j] accumulates a[i*k + p] * b[p*n + j]).
 *
 * The pages accumulate in FP32. Here every product of two floats is formed in
 * double (exact: 24 + 24 significant bits fit in 53), and the K products of an
 * output are summed in double in ascending k, so the only error left is the
 * double summation (relative ≤ K * 2^-53), far below the FP32 error bound the
 * GPU result is held to.
 *
 * Loop order is i-k-j (the outer-product order of "SGEMM CUDA kernel (First
 * Half)", Part 4): for each row i, a double row accumulator s[0..N) and a
 * magnitude row t[0..N) = sum_k |a_ik| |b_kj| are updated for k = 0..K-1.
 * Per output the additions still run in ascending k, exactly as in the
 * page's i-j-k loop; only the interleaving across j differs.
 *
 * Readings where the pages are silent (also listed in the design notes):
 *   - beta == 0: C_in is never read (the FP32 page kernel skips the read when
 *     beta is zero; BLAS convention), so NaN in C_in does not propagate.
 *   - alpha == 0: A and B are not read; C_out = beta * C_in.
 *   - K == 0: the sum is empty, C_out = beta * C_in.
 *
 * Build with -ffp-contract=off so no multiply-add is fused and the result is
 * identical on every host. OpenMP (optional) only splits rows across threads;
 * each row is computed by one thread in the order above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * out[r*N + j]  = alpha * sum_k A[i,k] * B[k,j] + beta * C[i,j]      (double)
 * mag[r*N + j]  = |alpha| * sum_k |A[i,k]| |B[k,j]| + |beta| |C[i,j]| (double)
 * for i = rows[r] (r < nrows), or i = r for all M rows when rows == NULL.
 * mag may be NULL. Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_sgemm_f64(int M, int N, int K, float alpha,
                     const float *A, long long lda,
                     const float *B, long long ldb,
                     float beta, const float *C, long long ldc,
                     const int *rows, int nrows,
                     double *out, double *mag, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || out == NULL) return -1;
    int R = rows ? nrows : M;
    if (R < 0) return -1;
    if (N == 0 || R == 0) return 0;
    const double da = (double)alpha, db = (double)beta;
    int bad = 0;
    int nt = nthreads > 0 ? nthreads : oracle_max_threads();
    (void)nt;

#pragma omp parallel num_threads(nt) reduction(|: bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        double *t = (double *)malloc(sizeof(double) * (size_t)N);
        if (s == NULL || t == NULL) {
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < R; ++r) {
                int i = rows ? rows[r] : r;
                if (i < 0 || i >= M) { bad = 1; continue; }
                for (int j = 0; j < N; ++j) { s[j] = 0.0; t[j] = 0.0; }
                if (alpha != 0.0f) {
                    for (int k = 0; k < K; ++k) {
                        const double a = (double)A[(long long)i * lda + k];
                        const double aa = fabs(a);
                        const float *brow = B + (long long)k * ldb;
                        for (int j = 0; j < N; ++j) {
                            const double b = (double)brow[j];
                            s[j] += a * b;
                            t[j] += aa * fabs(b);
                        }
                    }
                }
                double *o = out + (size_t)r * (size_t)N;
                double *m = mag ? mag + (size_t)r * (size_t)N : NULL;
                for (int j = 0; j < N; ++j) {
                    double v = (alpha != 0.0f) ? da * s[j] : 0.0;
                    double w = fabs(da) * t[j];
                    if (beta != 0.0f) {
                        const double c = (double)C[(long long)i * ldc + j];
                        v += db * c;
                        w += fabs(db) * fabs(c);
                    }
                    o[j] = v;
                    if (m) m[j] = w;
                }
            }
        }
        free(s);
        free(t);
    }
    return bad ? -1 : 0;
}

/*
 * The pages' own FP32 ground truth, generalised to alpha/beta: one float
 * accumulator per output, products and sums rounded to float in i-j-k order
 * ("SGEMM CUDA kernel (First Half)", Part 1: CPU version). Used only to check
 * that the FP32 error bound is neither vacuous nor too tight. out is M x N.
 */
int oracle_sgemm_f32_ijk(int M, int N, int K, float alpha,
                         const float *A, long long lda,
                         const float *B, long long ldb,
                         float beta, const float *C, long long ldc,
                         float *out)
{
    if (M < 0 || N < 0 || K < 0 || out == NULL) return -1;
    for (int i = 0; i < M; ++i) {
        for (int j = 0; j < N; ++j) {
            float sum = 0.0f;
            for (int k = 0; k < K; ++k) {
                float p = A[(long long)i * lda + k] * B[(long long)k * ldb + j];
                sum = sum + p;
            }
            float v = alpha * sum;
            if (beta != 0.0f) {
                float c = beta * C[(long long)i * ldc + j];
                v = v + c;
            }
            out[(size_t)i * (size_t)N + j] = v;
        }
    }
    return 0;
}
