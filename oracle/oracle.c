/*
 * fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it. It shares no code with the CUDA library.
 *
 * What it computes (plain definitions, written out with no tiling, fusion
 * or reordering):
 *
 *  oracle_attn -- "Why FlashAttention is fast", section 2, item 4 (the
 *    standard attention that materialises the score matrix): for every
 *    batch b, head h and query row i,
 *        s_j   = scale * sum_t q[b,i,h,t] * k[b,j,h,t]      (j in the key range)
 *        m     = max_j s_j
 *        l     = sum_j exp(s_j - m)
 *        P_j   = exp(s_j - m) / l                           (stable softmax)
 *        O     = sum_j P_j * v[b,j,h,:]
 *        LSE   = m + ln(l)                                  (natural log)
 *    The per-row log-sum-exp is the quantity each split emits in the
 *    flash-decoding issue ("where is flash decoding second stage (reduce)
 *    code?"). An empty key range gives LSE = -inf and O = 0, the identity
 *    of the combine below.
 *    Causal masking is not on the pages. With `causal` set, the reading
 *    used is the bottom-right-aligned mask: query row i (of sq) sees key j
 *    (of sk) only if j <= i + sk - sq, so the last query row sees every key
 *    and, with sq == sk, row i sees keys 0..i. That only shortens row i's
 *    key range; a row left with no key is an empty range (O = 0,
 *    LSE = -inf).
 *
 *  oracle_combine -- the second (reduce) stage of split-KV decoding, from
 *    the same flash-decoding issue: with the max of the split LSEs taken out
 *    first,
 *        M         = max_i LSE_i
 *        LSE_final = M + ln(sum_i exp(LSE_i - M))
 *        O_final   = sum_i exp(LSE_i - LSE_final) * O_i
 *
 * Inputs may be fp64, fp32, IEEE binary16 or bfloat16; 16-bit inputs are
 * decoded to fp64 element by element, so no fp64 copy of a large cache is
 * ever built. Outputs are always fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F64 0
#define ORACLE_F32 1
#define ORACLE_F16 2
#define ORACLE_BF16 3

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int f = bits & 0x3ff;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        mag = f ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE 754 binary32. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double load(const void *p, int dtype, int64_t i) {
    switch (dtype) {
    case ORACLE_F64: return ((const double *)p)[i];
    case ORACLE_F32: return (double)((const float *)p)[i];
    case ORACLE_F16: return oracle_f16_to_f64(((const uint16_t *)p)[i]);
    default: return oracle_bf16_to_f64(((const uint16_t *)p)[i]);
    }
}

/*
 * q: [b, sq, h, d]; k, v: [b, sk, h, d] (contiguous, d innermost).
 * rows: the query rows to evaluate (nrows of them), or NULL for 0..sq-1.
 * Keys j0 <= j < j1 take part; with causal != 0, row i also only keys
 * j <= i + sk - sq.
 * o: [b, nrows, h, d] fp64; lse: [b, h, nrows] fp64.
 * Returns 0, or -1 on a bad argument or allocation failure.
 */
int oracle_attn(const void *q, const void *k, const void *v, int dtype,
                int b, int sq, int sk, int h, int d, double scale,
                int j0, int j1, int causal, const int32_t *rows, int nrows,
                double *o, double *lse) {
    if (b < 0 || sq < 0 || sk < 0 || h < 0 || d <= 0 || j0 < 0 || j1 > sk || j0 > j1)
        return -1;
    if (rows == NULL) nrows = sq;
    if (nrows < 0) return -1;
    const int64_t total = (int64_t)b * h * nrows;
    int failed = 0;

#pragma omp parallel reduction(| : failed)
    {
        const int n_all = j1 - j0;
        double *s = (double *)malloc(sizeof(double) * (n_all > 0 ? n_all : 1));
        double *acc = (double *)malloc(sizeof(double) * d);
        {
#pragma omp for schedule(dynamic, 16)
            for (int64_t u = 0; u < total; ++u) {
                if (!s || !acc) {
                    failed = 1;
                    continue;
                }
                const int r = (int)(u % nrows);
                const int hh = (int)((u / nrows) % h);
                const int bb = (int)(u / ((int64_t)nrows * h));
                const int i = rows ? rows[r] : r;
                double *orow = o + (((int64_t)bb * nrows + r) * h + hh) * d;
                double *lrow = lse + ((int64_t)bb * h + hh) * nrows + r;
                if (i < 0 || i >= sq) {
                    failed = 1;
                    continue;
                }
                int n = n_all;
                if (causal) {
                    /* keys j0 .. min(j1, i + sk - sq + 1) - 1 */
                    const int64_t end = (int64_t)i + sk - sq + 1;
                    n = end <= j0 ? 0 : (end < j1 ? (int)(end - j0) : n_all);
                }
                if (n == 0) {
                    for (int t = 0; t < d; ++t) orow[t] = 0.0;
                    *lrow = -INFINITY;
                    continue;
                }
                const int64_t qoff = (((int64_t)bb * sq + i) * h + hh) * d;
                /* the score row s_j = scale * q_i . k_j */
                for (int j = 0; j < n; ++j) {
                    const int64_t koff = (((int64_t)bb * sk + (j0 + j)) * h + hh) * d;
                    double dot = 0.0;
                    for (int t = 0; t < d; ++t)
                        dot += load(q, dtype, qoff + t) * load(k, dtype, koff + t);
                    s[j] = scale * dot;
                }
                /* stable softmax of the row */
                double m = s[0];
                for (int j = 1; j < n; ++j)
                    if (s[j] > m) m = s[j];
                double l = 0.0;
                for (int j = 0; j < n; ++j) {
                    s[j] = exp(s[j] - m);
                    l += s[j];
                }
                for (int j = 0; j < n; ++j) s[j] /= l;
                /* O = P V */
                for (int t = 0; t < d; ++t) acc[t] = 0.0;
                for (int j = 0; j < n; ++j) {
                    const int64_t voff = (((int64_t)bb * sk + (j0 + j)) * h + hh) * d;
                    for (int t = 0; t < d; ++t) acc[t] += s[j] * load(v, dtype, voff + t);
                }
                for (int t = 0; t < d; ++t) orow[t] = acc[t];
                *lrow = m + log(l);
            }
        }
        free(s);
        free(acc);
    }
    return failed ? -1 : 0;
}

/*
 * Split-KV reduce. o_parts: [nsplit, nrows, d]; lse_parts: [nsplit, nrows].
 * o: [nrows, d]; lse: [nrows]. A row whose splits are all empty (every
 * LSE_i = -inf) gets LSE = -inf and O = 0.
 */
int oracle_combine(const double *o_parts, const double *lse_parts, int nsplit,
                   int64_t nrows, int d, double *o, double *lse) {
    if (nsplit <= 0 || nrows < 0 || d <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        double M = -INFINITY;
        for (int i = 0; i < nsplit; ++i) {
            double x = lse_parts[(int64_t)i * nrows + r];
            if (x > M) M = x;
        }
        double *orow = o + r * d;
        for (int t = 0; t < d; ++t) orow[t] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int i = 0; i < nsplit; ++i) sum += exp(lse_parts[(int64_t)i * nrows + r] - M);
        const double L = M + log(sum);
        for (int i = 0; i < nsplit; ++i) {
            const double w = exp(lse_parts[(int64_t)i * nrows + r] - L);
            const double *op = o_parts + ((int64_t)i * nrows + r) * d;
            for (int t = 0; t < d; ++t) orow[t] += w * op[t];
        }
        lse[r] = L;
    }
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
