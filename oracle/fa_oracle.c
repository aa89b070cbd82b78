/*
 * fa_oracle.c -- slow, plain float64 CPU reference for the attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or run this file.  It shares no code, header,
 * table or helper with the CUDA path and includes nothing from it.
 *
 * What it computes (per query row), following the pages:
 *   - "Guia Prático de Programação de GPU com Tiles", section 4 (row softmax): subtract the
 *     row maximum, exponentiate, sum, divide -- the numerically stable two-pass softmax;
 *   - same page, section 6 (flash attention): s = (q . k) * scale for every key, softmax over
 *     the keys, output = softmax-weighted sum of the value rows.  The online recurrence of
 *     that section reaches the same values up to rounding, so the oracle writes out the plain
 *     definition instead of the recurrence;
 *   - "Como Domar o Blackwell Sem Enlouquecer com CUDA" (the FlashAttention-4 paragraph):
 *     grouped-query attention -- query head h reads key/value head h / (Hq / Hkv);
 *   - causal masking (named in the FAQ of the first page, no alignment given): with
 *     causal == 1 key j is allowed for query row i when j <= i (top-left alignment); with
 *     causal == 2 when j <= i + (Sk - Sq) (bottom-right alignment: the last query row sees
 *     every key, as when new queries are appended after a cache of Sk - Sq keys);
 *   - a row with no allowed key (possible only for causal == 2 with Sq > Sk) has an empty
 *     softmax: its output is the empty sum, o = 0, and lse = ln 0 = -inf;
 *   - log-sum-exp of the scaled logits, natural log: lse = m + ln(sum_j exp(s_j - m)).
 *
 * Inputs are the raw 16-bit patterns of bf16 or fp16 tensors in [B, H, S, D] contiguous
 * layout; they are decoded exactly to double here, so the oracle sees the very values the
 * GPU sees.  Every arithmetic step is float64.
 *
 * A compile-time switch FA_ORACLE_PLANT (default 0 = off) plants one deliberate mistake;
 * the test suite builds such copies to show that its pins catch each of them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef FA_ORACLE_PLANT
#define FA_ORACLE_PLANT 0
#endif

/* bf16 is the upper half of an IEEE binary32: widen the bit pattern. */
static double decode_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 mantissa bits. */
static double decode_fp16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double val;
    if (e == 0)
        val = ldexp((double)m, -24);                 /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31)
        val = m ? NAN : INFINITY;
    else
        val = ldexp((double)(m | 0x400), e - 25);    /* (1 + m/1024) * 2^(e-15) */
    return sign ? -val : val;
}

static double decode(const uint16_t *p, int64_t idx, int is_fp16)
{
    return is_fp16 ? decode_fp16(p[idx]) : decode_bf16(p[idx]);
}

/* Exposed so the tests can pin the decoders against numpy's own conversions. */
double fa_oracle_decode(uint16_t bits, int is_fp16)
{
    return is_fp16 ? decode_fp16(bits) : decode_bf16(bits);
}

/*
 * One query row (b, h, i).  s is caller scratch of at least Sk doubles.
 * Writes D doubles to o_row and one double to *lse_row.
 */
static void attend_row(const uint16_t *q, const uint16_t *k, const uint16_t *v, int is_fp16,
                       int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t D,
                       int causal, double scale, int64_t b, int64_t h, int64_t i,
                       double *s, double *o_row, double *lse_row)
{
    const int64_t group = Hq / Hkv;
#if FA_ORACLE_PLANT == 1
    const int64_t kvh = h % Hkv;                 /* planted: wrong GQA head mapping */
#else
    const int64_t kvh = h / group;               /* consecutive query heads share a KV head */
#endif
    const int64_t qbase = ((b * Hq + h) * Sq + i) * D;
    const int64_t kvbase = (b * Hkv + kvh) * Sk * D;

    /* allowed keys: j < Sk, and j <= i (causal 1) or j <= i + Sk - Sq (causal 2) */
    int64_t n_allowed = Sk;
    if (causal) {
        int64_t last = (causal == 2) ? i + (Sk - Sq) : i;   /* last allowed key index */
#if FA_ORACLE_PLANT == 2
        last -= 1;                                        /* planted: causal bound off by one */
#elif FA_ORACLE_PLANT == 8
        if (causal == 2) last = i - (Sk - Sq);            /* planted: bottom-right offset sign */
#endif
        if (last + 1 < n_allowed) n_allowed = last + 1;
        if (n_allowed < 0) n_allowed = 0;
    }
    if (n_allowed == 0) {
        for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
        *lse_row = -INFINITY;
        return;
    }

    /* scores s_j = scale * sum_d q[d] k_j[d] */
    for (int64_t j = 0; j < n_allowed; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) {
#if FA_ORACLE_PLANT == 3
            /* planted: transposed key operand (reads k[d][j] of a D x Sk view) */
            dot += decode(q, qbase + d, is_fp16) * decode(k, kvbase + (d * Sk + j) % (Sk * D), is_fp16);
#else
            dot += decode(q, qbase + d, is_fp16) * decode(k, kvbase + j * D + d, is_fp16);
#endif
        }
#if FA_ORACLE_PLANT == 4
        s[j] = dot;                              /* planted: scale dropped */
#else
        s[j] = scale * dot;
#endif
    }

    /* stable softmax: subtract the row maximum, exponentiate, sum */
    double m = s[0];
    for (int64_t j = 1; j < n_allowed; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < n_allowed; ++j) {
        s[j] = exp(s[j] - m);                    /* s now holds the unnormalised weights */
        l += s[j];
    }

    /* weighted sum of value rows, normalised once at the end */
    for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
    for (int64_t j = 0; j < n_allowed; ++j) {
        const double w = s[j];
        for (int64_t d = 0; d < D; ++d) {
#if FA_ORACLE_PLANT == 5
            o_row[d] += w * decode(v, ((b * Hkv + kvh) * Sk + (n_allowed - 1 - j)) * D + d, is_fp16); /* planted: reversed value rows */
#else
            o_row[d] += w * decode(v, kvbase + j * D + d, is_fp16);
#endif
        }
    }
    for (int64_t d = 0; d < D; ++d) {
#if FA_ORACLE_PLANT == 6
        o_row[d] /= (double)n_allowed;           /* planted: divides by the key count, not the weight sum */
#else
        o_row[d] /= l;
#endif
    }
#if FA_ORACLE_PLANT == 7
    *lse_row = m + log(l) - scale;               /* planted: stray term in the log-sum-exp */
#else
    *lse_row = m + log(l);
#endif
}

/*
 * Evaluate n_rows query rows given as (b, h, i) triples in rows[3*r .. 3*r+2].
 * o_out is n_rows x D, lse_out is n_rows.  nthreads <= 0 means "all available".
 * Returns 0 on success, a negative value for invalid arguments.
 */
int fa_oracle_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int is_fp16,
                   int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t D,
                   int causal, double scale, const int64_t *rows, int64_t n_rows,
                   double *o_out, double *lse_out, int nthreads)
{
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Sq < 0 || Sk < 0 || D < 1 || causal < 0 || causal > 2)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t *t = rows + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= Hq || t[2] < 0 || t[2] >= Sq)
            return -2;
    }
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *s = (double *)malloc((size_t)(Sk > 0 ? Sk : 1) * sizeof(double));
        if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (int64_t r = 0; r < n_rows; ++r) {
                const int64_t *t = rows + 3 * r;
                attend_row(q, k, v, is_fp16, Hq, Hkv, Sq, Sk, D, causal, scale,
                           t[0], t[1], t[2], s, o_out + r * D, lse_out + r);
            }
            free(s);
        }
    }
    (void)nthreads;
    return bad ? -3 : 0;
}

/* Number of threads the oracle would use for nthreads <= 0. */
int fa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
