/*
 * window_oracle.c -- CPU oracle for the sliding-window sum.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code with the CUDA sources.
 *
 * Definition ("CMU DLSys Lecture 12: GPU Acceleration", section 3): for n
 * outputs and an input of n + W - 1 valid elements,
 *
 *     y_i = sum_{d=0}^{W-1} x_{i+d},      0 <= i < n,
 *
 * the valid (unpadded) window sum; the page's example is W = 5, and it writes
 * the general width as W = 2R + 1.
 *
 * window_sum_f64: every term widened to double, summed in ascending d -- the
 * definition.  window_sum_f32_ascending: the page's own fragment accumulates a
 * float `sum` over d = 0, 1, ..., W-1 starting from 0; this is that arithmetic
 * (each addition rounded to float, compiled without contraction), the value an
 * implementation with the same order must match bit for bit.
 *
 * Returns 0, or -1 for n < 0, W < 1 or a NULL pointer with n > 0.
 */
#include <stdint.h>
#include <stddef.h>

int oracle_window_sum_f64(int64_t n, int W, const float *x, double *y)
{
    if (n < 0 || W < 1 || (n > 0 && (x == NULL || y == NULL))) return -1;
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int d = 0; d < W; ++d) s += (double)x[i + d];
        y[i] = s;
    }
    return 0;
}

int oracle_window_sum_f32_ascending(int64_t n, int W, const float *x, float *y)
{
    if (n < 0 || W < 1 || (n > 0 && (x == NULL || y == NULL))) return -1;
    for (int64_t i = 0; i < n; ++i) {
        volatile float s = 0.0f;   /* one rounding per addition, in order */
        for (int d = 0; d < W; ++d) s = s + x[i + d];
        y[i] = s;
    }
    return 0;
}
