/*
 * reduce_oracle.c -- CPU oracle for the tiled reduction and the row softmax.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code with the CUDA sources.
 *
 * Both operations come from "Tiling Strategies", section 5 ("Tiling Beyond
 * GEMM"), which lists them beside GEMM as kernels that tile their input:
 *
 *   Reduction -- the input array is cut into chunks whose partial sums are
 *   combined.  What is computed is the plain sum of the array,
 *
 *       s = sum_{i=0}^{n-1} x_i,
 *
 *   here every term widened to double and added in ascending i.  The empty
 *   sum is 0.
 *
 *   Softmax -- two passes over the same data, "max, then normalize".  For each
 *   row r of a rows x cols matrix (row stride ldx floats):
 *
 *       pass 1:  m_r = max_j x_{r,j}
 *       pass 2:  s_r = sum_j exp(x_{r,j} - m_r),   y_{r,j} = exp(x_{r,j} - m_r) / s_r
 *
 *   in double, with libm's exp.  Subtracting the row maximum leaves the result
 *   unchanged mathematically and keeps every exponent <= 0, so no term
 *   overflows; the pages do not spell this step out, the "max" pass exists
 *   for it.
 *
 * Each returns 0, or -1 for a negative size, ldx < cols, ldy < cols or a NULL
 * pointer where the size is positive.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

int oracle_sum_f64(int64_t n, const float *x, double *out)
{
    if (n < 0 || out == NULL || (n > 0 && x == NULL)) return -1;
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += (double)x[i];
    *out = s;
    return 0;
}

int oracle_softmax_rows_f64(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                            double *y, int64_t ldy)
{
    if (rows < 0 || cols < 0 || ldx < cols || ldy < cols) return -1;
    if (rows > 0 && cols > 0 && (x == NULL || y == NULL)) return -1;
    for (int64_t r = 0; r < rows && cols > 0; ++r) {
        const float *xr = x + r * ldx;
        double *yr = y + r * ldy;
        /* pass 1: the row maximum */
        double m = (double)xr[0];
        for (int64_t j = 1; j < cols; ++j)
            if ((double)xr[j] > m) m = (double)xr[j];
        /* pass 2: exponentials, their sum, and the normalisation */
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            yr[j] = exp((double)xr[j] - m);
            s += yr[j];
        }
        for (int64_t j = 0; j < cols; ++j) yr[j] = yr[j] / s;
    }
    return 0;
}
