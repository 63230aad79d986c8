/*
 * CPU oracle for row-major single-precision GEMM -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  The product path (the CUDA library) never calls it and
 * shares no code with it.
 *
 * What it computes (the plain definition, nothing more):
 *   C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 * with A (M x K), B (K x N), C (M x N) dense and row-major, leading
 * dimensions K, N and N.  This is the element formula of the problem
 * statement on "LeetGPU problem 2: matrix multiplication" (yekq.top, section
 * "problem statement"), the same product as "Lesson 10: shared-memory tiled
 * GEMM" (hpc.payai.win, section 1, "what it is"), and the dot-product
 * definition on the euler0525 page (section "naive implementation"), whose
 * dimension letters are renamed (there the contraction is called N).
 *
 * Precision choices (the pages fix none):
 *   - every product of two floats is formed in double, where it is exact
 *     (24 + 24 significant bits <= 53);
 *   - products are summed in double in ascending k, starting from +0.0;
 *   - the double sum is rounded once to float (round to nearest even, the C
 *     conversion under the default floating-point environment).
 * In the same pass absAB[i][j] = sum_k |A[i][k]| * |B[k][j]| is formed in
 * double; it scales the tolerance |C - C_oracle| <= tol * absAB.
 *
 * Build with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Full product.  absAB may be NULL.  Loop order i (rows, one OpenMP task per
 * row), then k ascending, then j: the textbook triple loop with the k loop
 * hoisted out of j, which keeps the summation order of every C[i][j] equal
 * to plain ascending k.  Returns 0, or -1 on a bad argument / no memory. */
int oracle_gemm_f64acc(const float* A, const float* B, float* C, double* absAB,
                       int64_t M, int64_t N, int64_t K, int nthreads) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(|| : failed)
#endif
    {
        double* acc = (double*)malloc((size_t)N * sizeof(double));
        double* acc_abs = (double*)malloc((size_t)N * sizeof(double));
        if (!acc || !acc_abs) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t i = 0; i < M; ++i) {
                for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; acc_abs[j] = 0.0; }
                const float* a_row = A + i * K;
                for (int64_t k = 0; k < K; ++k) {
                    const double a = (double)a_row[k];
                    const double a_abs = fabs(a);
                    const float* b_row = B + k * N;
                    for (int64_t j = 0; j < N; ++j) {
                        const double b = (double)b_row[j];
                        acc[j] += a * b;
                        acc_abs[j] += a_abs * fabs(b);
                    }
                }
                float* c_row = C + i * N;
                for (int64_t j = 0; j < N; ++j) c_row[j] = (float)acc[j];
                if (absAB) {
                    double* ab_row = absAB + i * N;
                    for (int64_t j = 0; j < N; ++j) ab_row[j] = acc_abs[j];
                }
            }
        }
        free(acc);
        free(acc_abs);
    }
    return failed ? -1 : 0;
}

/* Selected entries only: out[t] = C[rows[t]][cols[t]] and out_abs[t] =
 * absAB[rows[t]][cols[t]], each an ascending-k double dot product rounded
 * once to float, i.e. bitwise the value the full product above gives.
 * Used to check sampled outputs of problems too large for the full loop. */
int oracle_gemm_entries(const float* A, const float* B, int64_t M, int64_t N, int64_t K,
                        const int64_t* rows, const int64_t* cols, int64_t count,
                        float* out, double* out_abs, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    for (int64_t t = 0; t < count; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * K + k];
            const double b = (double)B[k * N + j];
            acc += a * b;
            acc_abs += fabs(a) * fabs(b);
        }
        out[t] = (float)acc;
        if (out_abs) out_abs[t] = acc_abs;
    }
    return 0;
}

/* General form (row-major storage throughout):
 *   C = alpha * op(A) * op(B) + beta * C
 * where op(A) is M x K and is either A, stored M x K with row stride lda
 * (trans_a == 0), or the transpose of A stored K x M with row stride lda
 * (trans_a == 1); likewise op(B) is K x N, either B stored K x N or the
 * transpose of B stored N x K, with row stride ldb; C is stored M x N with
 * row stride ldc, and only that M x N window is read or written.  This is
 * the scaled, strided, optionally transposed product of the cuBLAS call
 * shown on "LeetGPU problem 2: matrix multiplication" (yekq.top, section
 * "cuBLAS reference"), restated for row-major storage.
 *
 * The sum over k is formed exactly as in oracle_gemm_f64acc (exact products,
 * double, ascending k from +0.0); then alpha * sum + beta * C_old is formed in
 * double and rounded once to float.  When beta == 0, C_old is not read, so
 * whatever C held (NaN included) does not matter (the BLAS convention).
 * absC (dense M x N, may be NULL) receives |alpha| * sum_k |op(A)_ik| |op(B)_kj|
 * + |beta| * |C_old_ij|, which scales the tolerance.  Returns 0 or -1. */
int oracle_gemm_general(int trans_a, int trans_b, int64_t M, int64_t N, int64_t K, float alpha,
                        const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                        float* C, int64_t ldc, double* absC, int nthreads) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if ((trans_a != 0 && trans_a != 1) || (trans_b != 0 && trans_b != 1)) return -1;
    if (lda < (trans_a ? M : K) || ldb < (trans_b ? K : N) || ldc < N) return -1;
    if (M == 0 || N == 0) return 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = (double)(trans_a ? A[k * lda + i] : A[i * lda + k]);
                const double b = (double)(trans_b ? B[j * ldb + k] : B[k * ldb + j]);
                acc += a * b;
                acc_abs += fabs(a) * fabs(b);
            }
            double r = (double)alpha * acc;
            double r_abs = fabs((double)alpha) * acc_abs;
            if (beta != 0.0f) {
                const double c = (double)C[i * ldc + j];
                r += (double)beta * c;
                r_abs += fabs((double)beta) * fabs(c);
            }
            C[i * ldc + j] = (float)r;
            if (absC) absC[i * N + j] = r_abs;
        }
    }
    return 0;
}

/* Number of threads an OpenMP region would use (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
