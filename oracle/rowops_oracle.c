/*
 * rowops_oracle.c -- plain fp64 CPU oracle for the row softmax and the row
 * sum.  TEST INFRASTRUCTURE ONLY: nothing on the product path calls, links or
 * loads it, and it shares no code with the CUDA library.
 *
 * Definitions ("CS336 lecture 6: kernels and Triton", the Triton softmax and
 * row-sum examples):
 *   softmax row i:  y[i][j] = exp(x[i][j] - max_k x[i][k]) / sum_k exp(x[i][k] - max_k x[i][k])
 *   row sum i:      s[i]    = sum_j x[i][j]
 * Inputs arrive as double arrays (exactly upcast from fp32 / bf16 by the
 * caller); everything is computed in double, in plain loops.
 */
#include <math.h>
#include <stdint.h>

int oracle_softmax_rows(const double *x, double *y, int64_t M, int64_t N)
{
    if (M < 0 || N < 0 || (M > 0 && N > 0 && (!x || !y)))
        return 1;
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;
        double *yi = y + i * N;
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j)
            if (xi[j] > m)
                m = xi[j];
        double z = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            yi[j] = exp(xi[j] - m);
            z += yi[j];
        }
        for (int64_t j = 0; j < N; ++j)
            yi[j] /= z;
    }
    return 0;
}

int oracle_row_sum(const double *x, double *s, int64_t M, int64_t N)
{
    if (M < 0 || N < 0 || (M > 0 && (!x || !s)))
        return 1;
    for (int64_t i = 0; i < M; ++i) {
        const double *xi = x + i * N;
        double acc = 0.0;
        for (int64_t j = 0; j < N; ++j)
            acc += xi[j];
        s[i] = acc;
    }
    return 0;
}
