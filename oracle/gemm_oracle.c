/*
 * gemm_oracle.c -- CPU oracle for the FP32 matrix product C = A x B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, constant or helper with
 * the CUDA sources under tiled_matrix_multiply_gb300/csrc.
 *
 * What it computes is the plain definition of the product, written out:
 *
 *   C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]            0 <= i < M, 0 <= j < N
 *
 * ("Tiling Hierarchy on GPUs", section "Inner Product": each output needs K
 * multiplies and K adds, M*N*K FMAs in all; the same sum, with A transposed,
 * is the C_ij formula of "CMU DLSys Lecture 12: GPU Acceleration", section 4;
 * the naive kernel of "Tiling Strategies", section 2, accumulates it over
 * ascending k.)
 *
 * Precision: every operand is widened to double and the sum is accumulated in
 * double, in ascending k, for every (i, j).  The product of two floats is
 * exact in double (24 + 24 significant bits < 53), so a fused or unfused
 * multiply-add gives the same double here on any host.  The caller rounds the
 * double result to float (round to nearest even) where it wants the FP32
 * value; for integer-valued inputs whose partial sums stay below 2^24 that
 * float is the exact result.
 *
 * Layout: row-major with explicit leading dimensions, element (r, c) of a
 * matrix X with leading dimension ldx is X[r * ldx + c].  No blocking and no
 * reordering of any sum: the only liberty taken is the loop order i-k-j for
 * the full product (each output still receives its K terms in ascending k, one
 * after another), so that B is walked along its rows.  Rows of C are shared
 * out over OpenMP threads; a row is never split, so the arithmetic does not
 * depend on the thread count.
 *
 * Error behaviour: returns 0 on success, -1 on a negative size, a leading
 * dimension shorter than its row, or a null pointer with a nonzero extent.
 */
#include <stdint.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int oracle_args_bad(int64_t M, int64_t N, int64_t K,
                           const float *A, int64_t lda,
                           const float *B, int64_t ldb)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (lda < K || ldb < N) return 1;
    if (M > 0 && K > 0 && A == NULL) return 1;
    if (K > 0 && N > 0 && B == NULL) return 1;
    return 0;
}

/* Full product into a double matrix C (M x N, leading dimension ldc). */
int oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    double *C, int64_t ldc, int threads)
{
    if (oracle_args_bad(M, N, K, A, lda, B, ldb)) return -1;
    if (ldc < N || (M > 0 && N > 0 && C == NULL)) return -1;
    if (threads < 1) threads = 1;

#pragma omp parallel for num_threads(threads) schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        double *c_row = C + i * ldc;
        for (int64_t j = 0; j < N; ++j) c_row[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a_ik = (double)A[i * lda + k];
            const float *b_row = B + k * ldb;
            for (int64_t j = 0; j < N; ++j)
                c_row[j] += a_ik * (double)b_row[j];
        }
    }
    return 0;
}

/*
 * Selected entries only: out[t] = C[ii[t]][jj[t]] by the same definition, one
 * dot product per entry in ascending k.  Used where the full product is too
 * large for the host to form in a test (the entries are sampled by the caller).
 */
int oracle_gemm_entries_f64(int64_t M, int64_t N, int64_t K,
                            const float *A, int64_t lda,
                            const float *B, int64_t ldb,
                            const int64_t *ii, const int64_t *jj, int64_t count,
                            double *out, int threads)
{
    if (oracle_args_bad(M, N, K, A, lda, B, ldb)) return -1;
    if (count < 0 || (count > 0 && (ii == NULL || jj == NULL || out == NULL))) return -1;
    for (int64_t t = 0; t < count; ++t)
        if (ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N) return -1;
    if (threads < 1) threads = 1;

#pragma omp parallel for num_threads(threads) schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = ii[t], j = jj[t];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += (double)A[i * lda + k] * (double)B[k * ldb + j];
        out[t] = acc;
    }
    return 0;
}

/* Threads OpenMP would use by default (1 when built without OpenMP). */
int oracle_default_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
