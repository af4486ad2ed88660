/*
 * sgemm_oracle.c — the CPU oracle for strict-FP32 SGEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference legs use it. It shares no code, header, helper
 * or constant with the CUDA library.
 *
 * What it computes is the plain definition of SGEMM as the pages state it
 * ("Optimizing SGEMM in CUDA", section "What is a SGEMM?"; "The road to a
 * fast GEMM", section "The problem and the ceiling"):
 *
 *     C[i][j] = alpha * sum_{k<K} A[i][k] * B[k][j] + beta * C0[i][j]
 *
 * with row-major A (M x K, row stride lda), B (K x N, row stride ldb) and
 * C (M x N, row stride ldc). Every float is promoted to double before any
 * arithmetic; the product of two floats is exact in double (24+24 < 53
 * significand bits), so the only rounding left is that of the double sum.
 * The loop order is i-k-j (the order of the CPU reference on "The road to a
 * fast GEMM", section "The complete code"), with a double accumulator row.
 *
 * Alongside the value it returns the magnitude sum
 *     S[i][j] = |alpha| * sum_k |A[i][k] * B[k][j]| + |beta * C0[i][j]|
 * that scales the floating-point error bound the GPU result is checked
 * against.
 *
 * Readings where the pages are silent (BLAS conventions):
 *   - beta == 0: C0 is not read (a NaN in C0 does not propagate).
 *   - alpha == 0 or K == 0: A and B are not read; C = beta * C0.
 *   - padding between rows (ld > width) is never read.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Returns 0 on success, -1 on invalid arguments. */
static int oracle_args_ok(int64_t M, int64_t N, int64_t K, int64_t lda,
                          int64_t ldb, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return 0;
    if (lda < (K > 1 ? K : 1)) return 0;
    if (ldb < (N > 1 ? N : 1)) return 0;
    if (ldc < (N > 1 ? N : 1)) return 0;
    return 1;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full oracle. ref and S are dense M x N double arrays (row stride N).
 * nthreads <= 0 uses every thread OpenMP offers.
 */
int oracle_sgemm(int64_t M, int64_t N, int64_t K, float alpha,
                 const float *A, int64_t lda, const float *B, int64_t ldb,
                 float beta, const float *C0, int64_t ldc,
                 double *ref, double *S, int nthreads) {
    if (!oracle_args_ok(M, N, K, lda, ldb, ldc)) return -1;
    if (M == 0 || N == 0) return 0;
    const double da = (double)alpha, db = (double)beta;
    const int use_ab = (alpha != 0.0f) && (K > 0);
    const int use_c = (beta != 0.0f);
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        double *mag = (double *)malloc(sizeof(double) * (size_t)N);
        if (acc == NULL || mag == NULL) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < M; ++i) {
                for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; mag[j] = 0.0; }
                if (use_ab) {
                    for (int64_t k = 0; k < K; ++k) {
                        const double a = (double)A[i * lda + k];
                        const float *brow = B + k * ldb;
                        for (int64_t j = 0; j < N; ++j) {
                            const double p = a * (double)brow[j];
                            acc[j] += p;
                            mag[j] += fabs(p);
                        }
                    }
                }
                for (int64_t j = 0; j < N; ++j) {
                    double v = use_ab ? da * acc[j] : 0.0;
                    double s = use_ab ? fabs(da) * mag[j] : 0.0;
                    if (use_c) {
                        const double c = db * (double)C0[i * ldc + j];
                        v += c;
                        s += fabs(c);
                    }
                    ref[i * N + j] = v;
                    S[i * N + j] = s;
                }
            }
        }
        free(acc);
        free(mag);
    }
    return failed ? -2 : 0;
}

/*
 * Sampled oracle: the same definition evaluated only at the n entries
 * (rows[e], cols[e]); ref[e] and S[e] receive the value and the magnitude
 * sum. Used where the full product would take the CPU too long.
 */
int oracle_sgemm_sampled(int64_t M, int64_t N, int64_t K, float alpha,
                         const float *A, int64_t lda, const float *B,
                         int64_t ldb, float beta, const float *C0, int64_t ldc,
                         int64_t n, const int64_t *rows, const int64_t *cols,
                         double *ref, double *S, int nthreads) {
    if (!oracle_args_ok(M, N, K, lda, ldb, ldc) || n < 0) return -1;
    for (int64_t e = 0; e < n; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -1;
    const double da = (double)alpha, db = (double)beta;
    const int use_ab = (alpha != 0.0f) && (K > 0);
    const int use_c = (beta != 0.0f);
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 64)
    for (int64_t e = 0; e < n; ++e) {
        const int64_t i = rows[e], j = cols[e];
        double acc = 0.0, mag = 0.0;
        if (use_ab) {
            for (int64_t k = 0; k < K; ++k) {
                const double p = (double)A[i * lda + k] * (double)B[k * ldb + j];
                acc += p;
                mag += fabs(p);
            }
        }
        double v = use_ab ? da * acc : 0.0;
        double s = use_ab ? fabs(da) * mag : 0.0;
        if (use_c) {
            const double c = db * (double)C0[i * ldc + j];
            v += c;
            s += fabs(c);
        }
        ref[e] = v;
        S[e] = s;
    }
    return 0;
}
