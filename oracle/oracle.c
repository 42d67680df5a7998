/*
 * oracle.c -- plain CPU fp64 oracle for PowerInfer-style activation-sparse FFN decode.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg may build, load or call this file. It shares no code, header,
 * table or constant with the CUDA library; neither side includes the other.
 *
 * What it computes, step by step, in the order the pages give them:
 *   predictor ("PowerInfer" walk-through page, section "activation predictor", eq.
 *   a = sigmoid(x Wp + b_p), neuron active if a_i > tau), read as the two-layer
 *   low-rank MLP  z = ReLU(u P1) P2 + b_p  (the same page's diagram calls the
 *   predictor a small MLP), active iff z > 0 (sigmoid(z) > 0.5 <=> z > 0), strict;
 *   the active set of a batch is the union over its rows;
 *   sparse FFN (same page, section "technical details", eq. FFN(x) =
 *   sigma(x W1) (.) (x W2) W3, with sigma = ReLU for the ReLU models the project
 *   targets) evaluated only on the active neurons:
 *     gated      h_i = max(0, u.Wg_i + bg_i) * (u.Wu_i)
 *     non-gated  h_i = max(0, u.W1_i + b1_i)
 *     y = sum_i h_i * WdT_i              (WdT = W_down transposed, [f x d])
 *   offline hot-first order (same page, offline profiling code block): neurons
 *   sorted by activation count, descending, ties by ascending index (Python's
 *   sorted() is stable).
 *
 * Weights are read at their exact stored values: f32, bf16 and f16 widened to
 * double exactly, int4 group-128 as q * fp16 scale (exact in double).
 * Every sum is taken in a fixed sequential order in double precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* stored element types (this file's own numbering) */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2, ORC_INT4G128 = 3 };
enum { ORC_GATED = 0, ORC_RELU = 1 };

/* ---------------------------------------------------------------- widening ---------- */

static double orc_from_bf16(uint16_t bits)
{
    /* bfloat16 is the top half of an IEEE binary32 */
    uint32_t w = (uint32_t)bits << 16;
    float v;
    memcpy(&v, &w, sizeof v);
    return (double)v;
}

static double orc_from_f16(uint16_t bits)
{
    /* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits */
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                 /* zero / subnormal: frac * 2^-14 * 2^-10 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(frac | 0x400), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    return sign ? -mag : mag;
}

static int orc_int4_at(const uint8_t *packed_row, int64_t t)
{
    /* two's-complement nibbles, element 2k in the low nibble of byte k */
    uint8_t byte = packed_row[t >> 1];
    int nib = (t & 1) ? (byte >> 4) : (byte & 0x0f);
    return nib >= 8 ? nib - 16 : nib;
}

/* Widen columns [c0, c1) of row `row` of a [rows x d] matrix to double: out[0 .. c1-c0). */
static void orc_row_span(const void *mat, const void *scales, int dt, int64_t d, int64_t row,
                         int64_t c0, int64_t c1, double *out)
{
    int64_t t;
    switch (dt) {
    case ORC_F32: {
        const float *m = (const float *)mat + row * d;
        for (t = c0; t < c1; ++t) out[t - c0] = (double)m[t];
        break;
    }
    case ORC_BF16: {
        const uint16_t *m = (const uint16_t *)mat + row * d;
        for (t = c0; t < c1; ++t) out[t - c0] = orc_from_bf16(m[t]);
        break;
    }
    case ORC_F16: {
        const uint16_t *m = (const uint16_t *)mat + row * d;
        for (t = c0; t < c1; ++t) out[t - c0] = orc_from_f16(m[t]);
        break;
    }
    case ORC_INT4G128: {
        const uint8_t *m = (const uint8_t *)mat + row * (d / 2);
        const uint16_t *s = (const uint16_t *)scales + row * (d / 128);
        for (t = c0; t < c1; ++t) out[t - c0] = (double)orc_int4_at(m, t) * orc_from_f16(s[t / 128]);
        break;
    }
    default:
        for (t = c0; t < c1; ++t) out[t - c0] = NAN;
    }
}

/* Widen all of row `row` (length d). */
static void orc_row(const void *mat, const void *scales, int dt, int64_t d, int64_t row, double *out)
{
    orc_row_span(mat, scales, dt, d, row, 0, d, out);
}

static double orc_dot(const double *a, const double *b, int64_t n)
{
    double acc = 0.0;
    for (int64_t t = 0; t < n; ++t) acc += a[t] * b[t];
    return acc;
}

/* Exposed for the pins: widen `n` elements (a [1 x n] row) of type dt. */
void orc_widen(const void *src, const void *scales, int dt, int64_t n, double *out)
{
    orc_row(src, scales, dt, n, 0, out);
}

int orc_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- predictor --------- */

/*
 * hp[b,k] = max(0, sum_t u[b,t] * P1T[k,t])                       (predictor hidden layer)
 * z[b,i]  = sum_k hp[b,k] * P2T[i,k] + b_pred[i]                   (predictor logits)
 * mask[i] = 1 iff z[b,i] > tau for some row b                      (union over the batch)
 * idx     = the i with mask[i] = 1, ascending; returns their number.
 * hp, z may be NULL. b_pred may be NULL (zero).
 */
int64_t orc_predict(const double *u, int B, int64_t d, int64_t r, int64_t f, int pdt,
                    const void *p1t, const void *p2t, const float *b_pred, double tau,
                    double *hp_out, double *z_out, uint8_t *mask, int32_t *idx)
{
    double *hp = (double *)malloc(sizeof(double) * (size_t)B * (size_t)r);
    double *z = (double *)malloc(sizeof(double) * (size_t)B * (size_t)f);
    int64_t k, i, n = 0;

#pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)(d > r ? d : r));
#pragma omp for schedule(static)
        for (k = 0; k < r; ++k) {
            orc_row(p1t, NULL, pdt, d, k, row);
            for (int b = 0; b < B; ++b) {
                double a = orc_dot(u + (size_t)b * d, row, d);
                hp[(size_t)b * r + k] = a > 0.0 ? a : 0.0;
            }
        }
#pragma omp for schedule(static)
        for (i = 0; i < f; ++i) {
            orc_row(p2t, NULL, pdt, r, i, row);
            for (int b = 0; b < B; ++b)
                z[(size_t)b * f + i] = orc_dot(hp + (size_t)b * r, row, r) + (b_pred ? (double)b_pred[i] : 0.0);
        }
        free(row);
    }

    for (i = 0; i < f; ++i) {
        int on = 0;
        for (int b = 0; b < B; ++b) on |= z[(size_t)b * f + i] > tau;
        mask[i] = (uint8_t)on;
        if (on) idx[n++] = (int32_t)i;
    }
    if (hp_out) memcpy(hp_out, hp, sizeof(double) * (size_t)B * (size_t)r);
    if (z_out) memcpy(z_out, z, sizeof(double) * (size_t)B * (size_t)f);
    free(hp);
    free(z);
    return n;
}

/* ---------------------------------------------------------------- sparse FFN -------- */

/*
 * For each listed neuron j (i = idx[j], j < n) and batch row b:
 *   gated:     h[b,j] = max(0, u_b.Wg_i + bg_i) * (u_b.Wu_i)
 *   non-gated: h[b,j] = max(0, u_b.W1_i + b1_i)          (W1 passed as wg)
 * then y[b,:] = sum_j h[b,j] * WdT[i,:], j ascending.
 * bg may be NULL (zero). h may be NULL. Returns 0, or -1 if an index is out of range.
 */
int orc_sparse_ffn(const double *u, int B, int64_t d, int64_t f, int kind, int wdt,
                   const void *wg, const void *wu, const void *wdn,
                   const void *sg, const void *su, const void *sd,
                   const float *bg, const int32_t *idx, int64_t n, double *h_out, double *y)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)B * (size_t)(n > 0 ? n : 1));
    int64_t j, c;
    for (j = 0; j < n; ++j)
        if (idx[j] < 0 || idx[j] >= f) {
            free(h);
            return -1;
        }

#pragma omp parallel
    {
        double *rg = (double *)malloc(sizeof(double) * (size_t)d);
        double *ru = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static)
        for (j = 0; j < n; ++j) {
            int64_t i = idx[j];
            orc_row(wg, sg, wdt, d, i, rg);
            if (kind == ORC_GATED) orc_row(wu, su, wdt, d, i, ru);
            for (int b = 0; b < B; ++b) {
                const double *ub = u + (size_t)b * d;
                double g = orc_dot(ub, rg, d) + (bg ? (double)bg[i] : 0.0);
                double a = g > 0.0 ? g : 0.0;
                h[(size_t)b * n + j] = kind == ORC_GATED ? a * orc_dot(ub, ru, d) : a;
            }
        }
        free(rg);
        free(ru);
    }

    /* y = sum_j h_j * WdT[idx_j]: threads own column blocks, j runs in order inside each. */
    memset(y, 0, sizeof(double) * (size_t)B * (size_t)d);
#pragma omp parallel
    {
        double *rd = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static)
        for (c = 0; c < d; c += 512) {
            int64_t c1 = c + 512 < d ? c + 512 : d;
            for (int64_t jj = 0; jj < n; ++jj) {
                orc_row_span(wdn, sd, wdt, d, idx[jj], c, c1, rd);
                for (int b = 0; b < B; ++b) {
                    double hb = h[(size_t)b * n + jj];
                    double *yb = y + (size_t)b * d;
                    for (int64_t t = c; t < c1; ++t) yb[t] += hb * rd[t - c];
                }
            }
        }
        free(rd);
    }
    if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)B * (size_t)(n > 0 ? n : 0));
    free(h);
    return 0;
}

/*
 * The dense FFN of the definition, every neuron included:
 *   y_b = sum_{i<f} ReLU(u_b.W1_i + b_i) * (u_b.W2_i) * W3_i   (gated; the factor (u.W2_i) absent if non-gated)
 * Written on its own (no call into the sparse routine).
 */
void orc_dense_ffn(const double *u, int B, int64_t d, int64_t f, int kind, int wdt,
                   const void *wg, const void *wu, const void *wdn,
                   const void *sg, const void *su, const void *sd, const float *bg, double *y)
{
    double *rg = (double *)malloc(sizeof(double) * (size_t)d);
    double *ru = (double *)malloc(sizeof(double) * (size_t)d);
    double *rd = (double *)malloc(sizeof(double) * (size_t)d);
    memset(y, 0, sizeof(double) * (size_t)B * (size_t)d);
    for (int64_t i = 0; i < f; ++i) {
        orc_row(wg, sg, wdt, d, i, rg);
        if (kind == ORC_GATED) orc_row(wu, su, wdt, d, i, ru);
        orc_row(wdn, sd, wdt, d, i, rd);
        for (int b = 0; b < B; ++b) {
            const double *ub = u + (size_t)b * d;
            double pre = orc_dot(ub, rg, d) + (bg ? (double)bg[i] : 0.0);
            double act = pre > 0.0 ? pre : 0.0;
            double hval = kind == ORC_GATED ? act * orc_dot(ub, ru, d) : act;
            for (int64_t t = 0; t < d; ++t) y[(size_t)b * d + t] += hval * rd[t];
        }
    }
    free(rg);
    free(ru);
    free(rd);
}

/* ---------------------------------------------------------------- stack glue -------- */

/* u_b = x_b / sqrt(mean_t x_b[t]^2 + eps): parameter-free RMS pre-norm between layers. */
void orc_rms_norm(const double *x, int B, int64_t d, double eps, double *u)
{
    for (int b = 0; b < B; ++b) {
        const double *xb = x + (size_t)b * d;
        double ss = 0.0;
        for (int64_t t = 0; t < d; ++t) ss += xb[t] * xb[t];
        double inv = 1.0 / sqrt(ss / (double)d + eps);
        for (int64_t t = 0; t < d; ++t) u[(size_t)b * d + t] = xb[t] * inv;
    }
}

/* ---------------------------------------------------------------- offline order ----- */

static const uint32_t *orc_sort_counts;

static int orc_cmp_hot_first(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    uint32_t ca = orc_sort_counts[a], cb = orc_sort_counts[b];
    if (ca != cb) return ca > cb ? -1 : 1; /* larger count first */
    return a < b ? -1 : (a > b);            /* equal counts: original order */
}

/* perm[k] = the neuron that goes to position k (hot-first). */
void orc_hot_first_order(const uint32_t *counts, int64_t f, int32_t *perm)
{
    for (int64_t i = 0; i < f; ++i) perm[i] = (int32_t)i;
    orc_sort_counts = counts;
    qsort(perm, (size_t)f, sizeof(int32_t), orc_cmp_hot_first);
    orc_sort_counts = NULL;
}
