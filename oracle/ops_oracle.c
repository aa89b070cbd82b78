/*
 * ops_oracle.c -- float64 CPU references for the tutorial's building blocks that the CUDA
 * library also provides as standalone kernels.  TEST INFRASTRUCTURE ONLY (see fa_oracle.c).
 *
 *   matrix product  (guide "Guia Prático de Programação de GPU com Tiles", section 5):
 *       C[m,n] = sum_k A[m,k] * B[k,n], A [M,K] and B [K,N] row-major 16-bit;
 *   bias + tanh-GELU epilogue (same guide, section 3, and the course's lesson 9 on fusing a
 *   bias into a matrix product):
 *       h = C[m,n] + bias[n];  gelu(h) = 0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3)));
 *   row softmax (same guide, section 4): y[r,:] = exp(x[r,:] - max) / sum exp(x[r,:] - max).
 *
 * Inputs are decoded exactly (16-bit patterns or fp32) and every step is float64.
 * FA_ORACLE_PLANT 9..11 plant one deliberate mistake each, for the pin tests.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef FA_ORACLE_PLANT
#define FA_ORACLE_PLANT 0
#endif

double fa_oracle_decode(uint16_t bits, int is_fp16);   /* fa_oracle.c */

/* tanh-GELU with the constants of the GELU paper (sqrt(2/pi) and 0.044715). */
static double gelu_tanh(double h)
{
    const double c = sqrt(2.0 / M_PI);
#if FA_ORACLE_PLANT == 11
    const double z = c * (h + 0.0447 * h * h * h);       /* planted: cubic coefficient */
#else
    const double z = c * (h + 0.044715 * h * h * h);
#endif
    return 0.5 * h * (1.0 + tanh(z));
}

double fa_oracle_gelu_tanh(double h) { return gelu_tanh(h); }

/*
 * Entries (m, n) of epilogue(A B): entries[2e], entries[2e+1] = m, n.
 * epilogue: 0 none, 1 + bias[n], 2 gelu(+ bias[n]).  bias may be NULL for epilogue 0.
 */
int fa_oracle_gemm_entries(const uint16_t *a, const uint16_t *b, int is_fp16, int64_t M, int64_t N,
                           int64_t K, const float *bias, int epilogue, const int64_t *entries,
                           int64_t n_entries, double *out)
{
    if (M < 1 || N < 1 || K < 1 || epilogue < 0 || epilogue > 2 || (epilogue && !bias)) return -1;
    for (int64_t e = 0; e < n_entries; ++e)
        if (entries[2 * e] < 0 || entries[2 * e] >= M || entries[2 * e + 1] < 0 || entries[2 * e + 1] >= N)
            return -2;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (int64_t e = 0; e < n_entries; ++e) {
        const int64_t m = entries[2 * e], n = entries[2 * e + 1];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
#if FA_ORACLE_PLANT == 9
            const int64_t bi = n * K + k < K * N ? n * K + k : 0;   /* planted: B read as [N,K] */
            acc += fa_oracle_decode(a[m * K + k], is_fp16) * fa_oracle_decode(b[bi], is_fp16);
#else
            acc += fa_oracle_decode(a[m * K + k], is_fp16) * fa_oracle_decode(b[k * N + n], is_fp16);
#endif
        }
        if (epilogue >= 1) acc += (double)bias[n];
        if (epilogue == 2) acc = gelu_tanh(acc);
        out[e] = acc;
    }
    return 0;
}

/*
 * Row softmax of the listed rows of x [rows, cols]; x is fp32 (x_f32) or 16-bit bf16 bits
 * (x_bf16), exactly one non-NULL.  out is n_rows x cols.
 */
int fa_oracle_softmax_rows(const float *x_f32, const uint16_t *x_bf16, int64_t rows, int64_t cols,
                           const int64_t *row_ids, int64_t n_rows, double *out)
{
    if (rows < 0 || cols < 1 || (!x_f32 == !x_bf16)) return -1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (row_ids[r] < 0 || row_ids[r] >= rows) return -2;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t base = row_ids[r] * cols;
        double *y = out + r * cols;
        for (int64_t c = 0; c < cols; ++c)
            y[c] = x_f32 ? (double)x_f32[base + c] : fa_oracle_decode(x_bf16[base + c], 0);
        double m = y[0];
        for (int64_t c = 1; c < cols; ++c)
            if (y[c] > m) m = y[c];
#if FA_ORACLE_PLANT == 10
        m = 0.0;                                          /* planted: no max subtraction */
#endif
        double sum = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            y[c] = exp(y[c] - m);
            sum += y[c];
        }
        for (int64_t c = 0; c < cols; ++c) y[c] /= sum;
    }
    return 0;
}
