/*
 * CPU oracle for blockwise ring self-attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * this file.  It shares no code with the CUDA library.
 *
 * What it computes is the plain definition of scaled dot-product attention
 * from "Sequence parallelism -- splitting the token dimension across GPUs"
 * (llmdaily, day 58), section "Attention wants keys and values from other
 * tokens": out = softmax(Q K^T / sqrt(d_k)) V, with the softmax of section
 * "But softmax seems to require all attention scores at once",
 * p_i = e^{s_i} / sum_j e^{s_j}.  Under the causal mask of section "Causal
 * attention gives us another optimization" the query at position t sees keys
 * 0..t inclusive (the page's token 30,000 attends to 1..30,000).
 *
 * Everything is accumulated in double precision.  The inputs are the exact
 * values the GPU saw: fp32, bf16 (raw 16-bit patterns, widened by placing
 * them in the top half of an fp32) or fp64.
 *
 * For one query row the steps are, in order:
 *   1. s_j = (sum_x q_x k_{j,x}) / sqrt(d)      for every allowed key j
 *   2. m = max_j s_j,  l = sum_j e^{s_j - m}     (softmax is unchanged by
 *      subtracting the same m from every score; it keeps e^{.} finite)
 *   3. p_j = e^{s_j - m} / l,  o_x = sum_j p_j v_{j,x},  lse = m + ln l
 * A row with no allowed key gets o = 0 and lse = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

static double load_elem(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    if (dtype == ORACLE_F64)
        return ((const double *)base)[idx];
    /* bf16: the 16 stored bits are the top half of an IEEE fp32 */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Attend each listed query row to the keys [kv_lo, kv_hi) of its own head.
 *
 *   q_rows  [n, d]          the query vectors of the listed rows
 *   k, v    [B, H, T, d]    full key and value tensors (row-major)
 *   rows    [n, 3]          (b, h, t) of each query; t is its global position
 *   causal                  if set, key j is allowed only when j <= t
 *   out     [n, d], lse [n] double results
 * Returns 0, or -1 on a bad argument or a failed allocation.
 */
int rsa_oracle_attend(const void *q_rows, const void *k, const void *v, int dtype,
                      int64_t B, int64_t H, int64_t T, int64_t d,
                      const int64_t *rows, int64_t n, int64_t kv_lo, int64_t kv_hi,
                      int causal, double *out, double *lse, int nthreads)
{
    if (B < 1 || H < 1 || T < 1 || d < 1 || n < 0 || kv_lo < 0 || kv_hi > T)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64)
        return -1;
    int bad = 0;
    const double scale = 1.0 / sqrt((double)d);
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
#endif
    {
        int64_t span = kv_hi > kv_lo ? kv_hi - kv_lo : 1;
        double *s = (double *)malloc((size_t)span * sizeof(double));
        double *q = (double *)malloc((size_t)d * sizeof(double));
        if (!s || !q)
            bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < n; ++r) {
            if (!s || !q)
                continue;
            const int64_t b = rows[3 * r], h = rows[3 * r + 1], t = rows[3 * r + 2];
            double *o = out + r * d;
            for (int64_t x = 0; x < d; ++x)
                o[x] = 0.0;
            if (b < 0 || b >= B || h < 0 || h >= H || t < 0 || t >= T) {
                bad = 1;
                lse[r] = NAN;
                continue;
            }
            int64_t hi = kv_hi;
            if (causal && t + 1 < hi)
                hi = t + 1;
            if (hi <= kv_lo) {
                lse[r] = -INFINITY;
                continue;
            }
            const int64_t head = (b * H + h) * T; /* first row of this head */
            for (int64_t x = 0; x < d; ++x)
                q[x] = load_elem(q_rows, dtype, r * d + x);

            /* step 1: scores, and their maximum */
            double m = -INFINITY;
            for (int64_t j = kv_lo; j < hi; ++j) {
                double dot = 0.0;
                for (int64_t x = 0; x < d; ++x)
                    dot += q[x] * load_elem(k, dtype, (head + j) * d + x);
                s[j - kv_lo] = dot * scale;
                if (s[j - kv_lo] > m)
                    m = s[j - kv_lo];
            }
            /* step 2: normaliser */
            double l = 0.0;
            for (int64_t j = kv_lo; j < hi; ++j)
                l += exp(s[j - kv_lo] - m);
            /* step 3: probabilities times values */
            for (int64_t j = kv_lo; j < hi; ++j) {
                const double p = exp(s[j - kv_lo] - m) / l;
                for (int64_t x = 0; x < d; ++x)
                    o[x] += p * load_elem(v, dtype, (head + j) * d + x);
            }
            lse[r] = m + log(l);
        }
        free(s);
        free(q);
    }
    return bad ? -1 : 0;
}

/* Number of threads OpenMP would use by default (1 without OpenMP). */
int rsa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
