/*
 * Paged decode attention -- fp64 CPU ORACLE.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test-suite, the smoke check and the bench's CPU-baseline leg may load
 * this file's library.  It shares no code, header or constant with the CUDA
 * library it checks.
 *
 * What it computes (the plain definition, not the blocked algorithm):
 *   "Efficient Memory Management for Large Language Model Serving with
 *   PagedAttention" (azimuth.plus summary), section "The PagedAttention
 *   algorithm", block-wise attention equation: the result is identical to
 *   standard softmax attention over the T keys of the sequence, with
 *   s_i = scale * q . K_i.
 *   CSDN tutorial "PagedAttention实战" §3.2 (PagedAttention.compute): gather the
 *   valid rows of every page of the sequence through the page table
 *   (valid_len = min(page_size, seq_len - start)), then dense softmax attention;
 *   an empty sequence yields zeros.
 *
 * Steps per (sequence s, query head h), in order:
 *   1. kv = h / (Hq / Hkv)                  (contiguous GQA groups)
 *   2. token t (0 <= t < T) is row t % B of physical block table[s][t / B]
 *   3. s_t = scale * sum_k q[k] * K_t[k]    (fp64, stored values decoded exactly)
 *   4. m = max_t s_t ; p_t = exp(s_t - m) ; out = sum_t p_t V_t / sum_t p_t
 *
 * Cache layout: [num_blocks][B][Hkv][d] (the tutorial's Page keys/values of shape
 * [page_size, num_heads, head_dim], stacked over pages).  q and out: [S][Hq][d].
 * dtype codes: 0 = fp32, 1 = fp16 (IEEE binary16), 2 = bf16 (upper half of binary32).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, from the format's definition:
 * sign(1) exponent(5, bias 15) fraction(10); exponent 0 = subnormal, 31 = inf/nan. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double: the 16 bits are the upper half of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem(const void *base, int dtype, size_t i)
{
    if (dtype == 0)
        return (double)((const float *)base)[i];
    if (dtype == 1)
        return oracle_f16_to_f64(((const uint16_t *)base)[i]);
    return oracle_bf16_to_f64(((const uint16_t *)base)[i]);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Returns 0 on success, -1 on bad shapes, -2 if a referenced table entry is
 * outside [0, num_blocks) or a context length exceeds the table's capacity. */
int oracle_decode(double *out, const void *q, const void *k_cache, const void *v_cache,
                  int dtype, const int32_t *block_tables, int max_blocks,
                  const int32_t *context_lens, int S, int Hq, int Hkv, int d, int B,
                  long long num_blocks, double scale)
{
    if (S < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || B <= 0 || Hq % Hkv != 0 || dtype < 0 || dtype > 2)
        return -1;
    for (int s = 0; s < S; ++s) {
        int T = context_lens[s];
        if (T < 0 || (long long)T > (long long)max_blocks * B)
            return -2;
        for (int j = 0; j < (T + B - 1) / B; ++j) {
            int32_t p = block_tables[(size_t)s * max_blocks + j];
            if (p < 0 || p >= num_blocks)
                return -2;
        }
    }
    const int G = Hq / Hkv;
    const long long pairs = (long long)S * Hq;

#pragma omp parallel
    {
        double *score = NULL;
        size_t cap = 0;
#pragma omp for schedule(dynamic, 1)
        for (long long ph = 0; ph < pairs; ++ph) {
            const int s = (int)(ph / Hq);
            const int h = (int)(ph % Hq);
            const int kv = h / G;
            const int T = context_lens[s];
            double *o = out + ((size_t)s * Hq + h) * d;
            for (int k = 0; k < d; ++k)
                o[k] = 0.0;
            if (T == 0)
                continue;
            if ((size_t)T > cap) {
                free(score);
                cap = (size_t)T;
                score = (double *)malloc(cap * sizeof(double));
            }
            const size_t qoff = ((size_t)s * Hq + h) * d;
            /* steps 2-3: scores over the gathered keys */
            double m = -INFINITY;
            for (int t = 0; t < T; ++t) {
                const size_t phys = (size_t)block_tables[(size_t)s * max_blocks + t / B];
                const size_t row = ((phys * B + (size_t)(t % B)) * Hkv + kv) * d;
                double acc = 0.0;
                for (int k = 0; k < d; ++k)
                    acc += elem(q, dtype, qoff + k) * elem(k_cache, dtype, row + k);
                score[t] = scale * acc;
                if (score[t] > m)
                    m = score[t];
            }
            /* step 4: softmax weights and the weighted sum of values */
            double l = 0.0;
            for (int t = 0; t < T; ++t) {
                const size_t phys = (size_t)block_tables[(size_t)s * max_blocks + t / B];
                const size_t row = ((phys * B + (size_t)(t % B)) * Hkv + kv) * d;
                const double p = exp(score[t] - m);
                l += p;
                for (int k = 0; k < d; ++k)
                    o[k] += p * elem(v_cache, dtype, row + k);
            }
            for (int k = 0; k < d; ++k)
                o[k] /= l;
        }
        free(score);
    }
    return 0;
}
