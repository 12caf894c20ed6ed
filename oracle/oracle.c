/*
 * oracle.c -- plain, slow fp64 CPU oracle of the neuron-aware sparse FFN
 * decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library: every value here is computed
 * from the definitions below, in double precision, with plain loops.
 *
 * Sources (the pages describing PowerInfer):
 *  - PowerInfer summary (CSDN), section "Background" (MLP block): FC1 and FC2
 *    are matrix-vector products whose outputs are dot products of the input
 *    with neurons (rows/columns of the weight matrices); ReLU keeps only the
 *    positive FC1 outputs, and only those neurons influence FC2.
 *  - same page, section "Neuron-aware operator": an operator first decides
 *    whether a neuron is active and, if so, processes that neuron's row or
 *    column of the weight matrix; inactive neurons are skipped.
 *  - same page, section "Adaptive sparse predictor": the activation predictor
 *    is an MLP with an input, a hidden and an output layer whose input and
 *    output sizes are fixed by the transformer layer.
 *  - same page, section "Neuron placement and management": neuron tables map
 *    each stored neuron to its original position in the matrix.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - the predictor is linear and low rank: u = P1 x, s = P2 u + b, and a
 *    neuron is predicted active iff s > tau (strict);
 *  - the predicted-active decision is taken in fp32 (the precision of the
 *    CUDA kernels): fl32(s) > tau; a guard band says where fp32 rounding could
 *    flip it;
 *  - weights are IEEE binary16 (or INT4 group-32 codes with binary16 scales),
 *    inputs x are binary16, everything else is exact fp64 arithmetic;
 *  - INT4: code q in [-8, 7] (two's complement nibble), the even element in
 *    the low nibble, value q * scale, one scale per 32 consecutive elements;
 *  - gated layer: h = ReLU(Wg x + bg) * (Wu x);
 *  - inter-layer normalisation: x' = fp16(y / sqrt(mean(y^2) + eps)), round
 *    to nearest even;
 *  - attention heads as the self-attention block's neurons (see
 *    oracle_attn_heads): the head mask comes from the same low-rank predictor
 *    form (oracle_predict with F = heads); a head not predicted active adds
 *    nothing to this token's output, but the token's key and value are
 *    projected for every KV head and stored as binary16, so the cache stays
 *    complete for later tokens.
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int kind;               /* 0: binary16 rows [rows, d]; 1: INT4 group-32 */
    const uint16_t *f16;    /* kind 0: binary16 bit patterns, row-major     */
    const uint8_t *q;       /* kind 1: packed codes [rows, d/2]             */
    const uint16_t *scales; /* kind 1: binary16 scales [rows, d/32]         */
} oracle_mat;

/* ---------------------------------------------------------------- numbers */

/* IEEE 754 binary16 -> double, from the format's definition. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* subnormal: m * 2^-24   */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);  /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* double -> binary16, round to nearest, ties to even (the default rounding
 * mode of rint), with overflow to infinity and gradual underflow. */
uint16_t oracle_double_to_half(double v)
{
    if (isnan(v))
        return 0x7e00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a < ldexp(1.0, -14)) {                  /* subnormal range */
        double q = rint(ldexp(a, 24));          /* units of 2^-24  */
        return sign | (uint16_t)q;              /* q == 1024 is the smallest normal */
    }
    int ex;
    frexp(a, &ex);                              /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;                             /* a in [2^E, 2^(E+1))         */
    double m = rint(ldexp(a, 10 - E));          /* in [1024, 2048]             */
    if (m == 2048.0) {
        m = 1024.0;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)m - 1024));
}

/* Element (row, col) of a weight matrix with rows of d elements. */
static double mat_at(const oracle_mat *m, int d, long row, int col)
{
    if (m->kind == 0)
        return oracle_half_to_double(m->f16[row * (long)d + col]);
    uint8_t byte = m->q[row * (long)(d / 2) + col / 2];
    int code = (col % 2 == 0) ? (byte & 0xf) : (byte >> 4);
    if (code >= 8)
        code -= 16;
    double scale = oracle_half_to_double(m->scales[row * (long)(d / 32) + col / 32]);
    return (double)code * scale;
}

/* Decode one full row (exported so tests can look at the weight decoding). */
int oracle_decode_row(const oracle_mat *m, int d, long row, double *out)
{
    if (!m || !out || d <= 0 || (m->kind == 1 && d % 32 != 0))
        return -1;
    for (int c = 0; c < d; ++c)
        out[c] = mat_at(m, d, row, c);
    return 0;
}

static double dot_row(const oracle_mat *m, int d, long row, const uint16_t *x)
{
    double acc = 0.0;
    for (int c = 0; c < d; ++c)
        acc += mat_at(m, d, row, c) * oracle_half_to_double(x[c]);
    return acc;
}

static int mask_bit(const uint32_t *mask, long k)
{
    return (mask[k / 32] >> (k % 32)) & 1u;
}

static double gamma_n(double n, double unit_roundoff)
{
    return n * unit_roundoff / (1.0 - n * unit_roundoff);
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------- predictor */

/*
 * u_i = sum_j P1[i,j] x_j                       (i < r)
 * s_k = sum_i P2[k,i] u_i + b_k                  (k < F)
 * mask bit k (word k/32, bit k%32) = fl32(s_k) > tau
 *
 * band_k bounds, with a factor-2 margin, how far an fp32 evaluation of s_k in
 * any summation order (unit roundoff `unit_roundoff`) can be from s_k:
 *   a_i  = sum_j |P1[i,j] x_j|,   e_i = gamma(d) a_i   (error of u_i)
 *   E_k  = gamma(r+1) (sum_i |P2[k,i]| (|u_i| + e_i) + |b_k|) + sum_i |P2[k,i]| e_i
 *   band = 2 E_k + 2 unit_roundoff |s_k|
 * Outside [s_k - band_k, s_k + band_k] an fp32 evaluation cannot change side.
 * u, s, band may be NULL.
 */
int oracle_predict(int d, int F, int r, const uint16_t *x, const uint16_t *p1,
                   const uint16_t *p2, const uint16_t *bpred, float tau,
                   double unit_roundoff, double *u_out, double *s_out,
                   double *band_out, uint32_t *mask)
{
    if (d <= 0 || F <= 0 || r <= 0 || !x || !p1 || !p2 || !bpred || !mask)
        return -1;
    double *u = (double *)malloc(sizeof(double) * r);
    double *a = (double *)malloc(sizeof(double) * r);
    if (!u || !a) {
        free(u);
        free(a);
        return -2;
    }
#pragma omp parallel for schedule(static)
    for (int i = 0; i < r; ++i) {
        double acc = 0.0, absacc = 0.0;
        for (int j = 0; j < d; ++j) {
            double t = oracle_half_to_double(p1[(long)i * d + j]) * oracle_half_to_double(x[j]);
            acc += t;
            absacc += fabs(t);
        }
        u[i] = acc;
        a[i] = absacc;
    }
    double gd = gamma_n((double)d, unit_roundoff);
    double gr = gamma_n((double)r + 1.0, unit_roundoff);
    memset(mask, 0, sizeof(uint32_t) * (size_t)((F + 31) / 32));
    int words = (F + 31) / 32;
#pragma omp parallel for schedule(static)
    for (int w = 0; w < words; ++w) {
        uint32_t bits = 0;
        for (int k = w * 32; k < F && k < w * 32 + 32; ++k) {
            double b = oracle_half_to_double(bpred[k]);
            double s = b, mag = fabs(b), prop = 0.0;
            for (int i = 0; i < r; ++i) {
                double p = oracle_half_to_double(p2[(long)k * r + i]);
                s += p * u[i];
                mag += fabs(p) * (fabs(u[i]) + gd * a[i]);
                prop += fabs(p) * gd * a[i];
            }
            if ((float)s > tau)
                bits |= 1u << (k % 32);
            if (s_out)
                s_out[k] = s;
            if (band_out)
                band_out[k] = 2.0 * (gr * mag + prop) + 2.0 * unit_roundoff * fabs(s);
        }
        mask[w] = bits;
    }
    if (u_out)
        memcpy(u_out, u, sizeof(double) * r);
    free(u);
    free(a);
    return 0;
}

/* ------------------------------------------------------------ compaction */

/*
 * idx  = storage positions k with mask bit k set, ascending;
 * orig = table[idx] (original neuron ids; skipped when table or orig is NULL);
 * *count = number of positions.
 */
int oracle_compact(int F, const uint32_t *mask, const int32_t *table, int32_t *idx,
                   int32_t *orig, int32_t *count)
{
    if (F < 0 || !mask || !idx || !count)
        return -1;
    int n = 0;
    for (long k = 0; k < F; ++k) {
        if (mask_bit(mask, k)) {
            idx[n] = (int32_t)k;
            if (table && orig)
                orig[n] = table[k];
            ++n;
        }
    }
    *count = n;
    return 0;
}

/* out = bitwise OR of B masks of F bits each (the batch's union). */
int oracle_mask_union(int B, int F, const uint32_t *masks, uint32_t *out)
{
    if (B <= 0 || F < 0 || !masks || !out)
        return -1;
    int words = (F + 31) / 32;
    for (int w = 0; w < words; ++w) {
        uint32_t acc = 0;
        for (int b = 0; b < B; ++b)
            acc |= masks[(long)b * words + w];
        out[w] = acc;
    }
    return 0;
}

/* ------------------------------------------------------------------- FFN */

/* One neuron's FC1 output: ReLU(W1[k] x + b1[k]), or for a gated layer
 * ReLU(Wg[k] x + bg[k]) * (Wu[k] x). */
static double neuron_h(int d, int gated, const uint16_t *x, const oracle_mat *w1,
                       const uint16_t *b1, const oracle_mat *wu, long k)
{
    double z = dot_row(w1, d, k, x) + oracle_half_to_double(b1[k]);
    double h = z > 0.0 ? z : 0.0;
    if (gated)
        h *= dot_row(wu, d, k, x);
    return h;
}

/* h_j = FC1 output of storage row idx_j, j < n. */
int oracle_fc1(int d, int gated, const uint16_t *x, const oracle_mat *w1,
               const uint16_t *b1, const oracle_mat *wu, const int32_t *idx, int n,
               double *h)
{
    if (d <= 0 || n < 0 || !x || !w1 || !b1 || (gated && !wu) || (n > 0 && (!idx || !h)))
        return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int j = 0; j < n; ++j)
        h[j] = neuron_h(d, gated, x, w1, b1, wu, idx[j]);
    return 0;
}

/* y_c = b2_c + sum_{j<n} h_j W2t[idx_j, c]  (j ascending). */
int oracle_fc2(int d, const oracle_mat *w2t, const uint16_t *b2, const double *h,
               const int32_t *idx, int n, double *y)
{
    if (d <= 0 || n < 0 || !w2t || !b2 || !y || (n > 0 && (!h || !idx)))
        return -1;
#pragma omp parallel for schedule(static)
    for (int c = 0; c < d; ++c) {
        double acc = oracle_half_to_double(b2[c]);
        for (int j = 0; j < n; ++j)
            acc += h[j] * mat_at(w2t, d, idx[j], c);
        y[c] = acc;
    }
    return 0;
}

/*
 * Masked FFN, the neuron-aware definition: only neurons whose mask bit is set
 * are computed; y = b2 + sum over those neurons of h_k * W2t[k, :].  The sum
 * runs over neurons in ORIGINAL id order (through the neuron table), so the
 * result does not depend on the storage order at all.
 */
int oracle_ffn_masked(int d, int F, int gated, const uint16_t *x, const oracle_mat *w1,
                      const uint16_t *b1, const oracle_mat *wu, const oracle_mat *w2t,
                      const uint16_t *b2, const int32_t *table, const uint32_t *mask,
                      double *y)
{
    if (d <= 0 || F <= 0 || !x || !w1 || !b1 || (gated && !wu) || !w2t || !b2 || !table ||
        !mask || !y)
        return -1;
    int32_t *row_of = (int32_t *)malloc(sizeof(int32_t) * F);   /* original id -> storage row */
    double *h = (double *)malloc(sizeof(double) * F);
    if (!row_of || !h) {
        free(row_of);
        free(h);
        return -2;
    }
    for (int k = 0; k < F; ++k)
        row_of[k] = -1;
    for (int k = 0; k < F; ++k) {
        if (table[k] < 0 || table[k] >= F || row_of[table[k]] != -1) {
            free(row_of);
            free(h);
            return -3;                                        /* not a permutation */
        }
        row_of[table[k]] = k;
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int k = 0; k < F; ++k)
        h[k] = mask_bit(mask, k) ? neuron_h(d, gated, x, w1, b1, wu, k) : 0.0;
#pragma omp parallel for schedule(static)
    for (int c = 0; c < d; ++c) {
        double acc = oracle_half_to_double(b2[c]);
        for (int o = 0; o < F; ++o) {
            int k = row_of[o];
            if (mask_bit(mask, k))
                acc += h[k] * mat_at(w2t, d, k, c);
        }
        y[c] = acc;
    }
    free(row_of);
    free(h);
    return 0;
}

/* Dense FFN: every neuron, storage order, no table:
 * y = b2 + sum_k h_k W2t[k, :]. */
int oracle_ffn_dense(int d, int F, int gated, const uint16_t *x, const oracle_mat *w1,
                     const uint16_t *b1, const oracle_mat *wu, const oracle_mat *w2t,
                     const uint16_t *b2, double *y)
{
    if (d <= 0 || F <= 0 || !x || !w1 || !b1 || (gated && !wu) || !w2t || !b2 || !y)
        return -1;
    double *h = (double *)malloc(sizeof(double) * F);
    if (!h)
        return -2;
#pragma omp parallel for schedule(dynamic, 16)
    for (int k = 0; k < F; ++k)
        h[k] = neuron_h(d, gated, x, w1, b1, wu, k);
#pragma omp parallel for schedule(static)
    for (int c = 0; c < d; ++c) {
        double acc = oracle_half_to_double(b2[c]);
        for (int k = 0; k < F; ++k)
            acc += h[k] * mat_at(w2t, d, k, c);
        y[c] = acc;
    }
    free(h);
    return 0;
}

/* ------------------------------------------------------- normalisation */

/*
 * x'_c = fp16( y_c / sqrt(mean(y^2) + eps) ), round to nearest even.
 * pre_c is the value before rounding; band_c bounds, with a factor-2 margin,
 * how far an fp32 evaluation (sum of squares in any order, a reciprocal
 * square root within 2 ulp, one product) can be from pre_c.  pre and band may
 * be NULL.
 */
int oracle_rmsnorm_half(int d, const double *y, double eps, double unit_roundoff,
                        uint16_t *x_out, double *pre, double *band)
{
    if (d <= 0 || !y || !x_out)
        return -1;
    double ss = 0.0;
    for (int c = 0; c < d; ++c)
        ss += y[c] * y[c];
    double scale = 1.0 / sqrt(ss / d + eps);
    double rel = gamma_n((double)d + 1.0, unit_roundoff) + 6.0 * unit_roundoff;
    for (int c = 0; c < d; ++c) {
        double v = y[c] * scale;
        x_out[c] = oracle_double_to_half(v);
        if (pre)
            pre[c] = v;
        if (band)
            band[c] = 2.0 * rel * fabs(v);
    }
    return 0;
}

/* ------------------------------------------------------- attention heads */

/*
 * One decode token through a self-attention block whose neurons are its
 * heads.  Sources: PowerInfer summary (CSDN), section "Background", paragraph
 * on activation sparsity (in the self-attention block about half of the heads
 * contribute little, so that block is sparse too) and section "Adaptive
 * sparse predictor"; the unite.ai page, section on adaptive sparsity
 * predictors (one predictor for the MLP block and one for the self-attention
 * block of each layer, and only the neurons predicted active are computed).
 *
 * For the token x (binary16, length d) with cache positions 0 .. pos-1 filled:
 *   k_g = Wk_g x + bk_g,  v_g = Wv_g x + bv_g   for every KV head g, stored as
 *                          binary16 (nearest even) at cache position pos;
 *   for every head h whose bit is set in head_mask (KV head g = h / (H/KVH)):
 *     q   = Wq_h x + bq_h
 *     a_t = exp(e_t - max_t e_t) / sum_t exp(e_t - max_t e_t),
 *           e_t = (q . K_g[t]) / sqrt(dh),   t = 0 .. pos (the new token included)
 *     o_h = sum_t a_t V_g[t]
 *   y = bo + sum over those h of  sum_i o_h[i] * Wot[h*dh + i, :]
 * Heads whose bit is clear: no query, no attention, no output-projection rows.
 *
 * Layouts (binary16 bit patterns): wqkv [(H + 2 KVH) dh, d] with the query
 * rows of head h at h*dh, the key rows of KV head g at (H + g) dh and its value
 * rows at (H + KVH + g) dh; bqkv [(H + 2 KVH) dh]; wot = Wo transposed,
 * [H dh, d], row j = column j of Wo; bo [d]; kcache, vcache [KVH, smax, dh]
 * (position pos is written); head_mask ceil(H/32) words.  y [d] out;
 * o_out (nullable) [H dh]: every o_h, zero for heads left out.
 * kv_pre, kv_band (nullable) [2 KVH dh]: the keys then the values before
 * rounding, and a bound (factor-2 margin) on how far an fp32 evaluation of
 * each, in any summation order with unit roundoff `unit_roundoff`, can be
 * from it: 2 gamma(d + 1) (sum_c |w_c x_c| + |b|).
 */
int oracle_attn_heads(int d, int H, int KVH, int dh, int smax, int pos, const uint16_t *x,
                      const uint16_t *wqkv, const uint16_t *bqkv, const uint16_t *wot,
                      const uint16_t *bo, const uint32_t *head_mask, uint16_t *kcache,
                      uint16_t *vcache, double *o_out, double *y, double unit_roundoff,
                      double *kv_pre, double *kv_band)
{
    if (d <= 0 || H <= 0 || KVH <= 0 || H % KVH != 0 || dh <= 0 || smax <= 0 || pos < 0 ||
        pos >= smax || !x || !wqkv || !bqkv || !wot || !bo || !head_mask || !kcache || !vcache || !y)
        return -1;
    const int G = H / KVH;
    const long nkv = 2L * KVH * dh;
    double *kv = (double *)malloc(sizeof(double) * (size_t)nkv);
    double *q = (double *)malloc(sizeof(double) * (size_t)dh);
    double *e = (double *)malloc(sizeof(double) * (size_t)(pos + 1));
    double *o = (double *)malloc(sizeof(double) * (size_t)dh);
    if (!kv || !q || !e || !o) {
        free(kv);
        free(q);
        free(e);
        free(o);
        return -2;
    }
    /* keys and values of the new token, every KV head */
#pragma omp parallel for schedule(static)
    for (long j = 0; j < nkv; ++j) {
        long row = (long)H * dh + j;
        double acc = oracle_half_to_double(bqkv[row]);
        double mag = fabs(acc);
        for (int c = 0; c < d; ++c) {
            double t = oracle_half_to_double(wqkv[row * d + c]) * oracle_half_to_double(x[c]);
            acc += t;
            mag += fabs(t);
        }
        kv[j] = acc;
        if (kv_pre)
            kv_pre[j] = acc;
        if (kv_band)
            kv_band[j] = 2.0 * gamma_n((double)d + 1.0, unit_roundoff) * mag;
    }
    for (int g = 0; g < KVH; ++g)
        for (int i = 0; i < dh; ++i) {
            long at = ((long)g * smax + pos) * dh + i;
            kcache[at] = oracle_double_to_half(kv[(long)g * dh + i]);
            vcache[at] = oracle_double_to_half(kv[(long)KVH * dh + (long)g * dh + i]);
        }
    for (int c = 0; c < d; ++c)
        y[c] = oracle_half_to_double(bo[c]);
    if (o_out)
        memset(o_out, 0, sizeof(double) * (size_t)H * dh);
    const double inv_sqrt = 1.0 / sqrt((double)dh);
    for (int h = 0; h < H; ++h) {
        if (!mask_bit(head_mask, h))
            continue;
        const int g = h / G;
        for (int i = 0; i < dh; ++i) {
            long row = (long)h * dh + i;
            double acc = oracle_half_to_double(bqkv[row]);
            for (int c = 0; c < d; ++c)
                acc += oracle_half_to_double(wqkv[row * d + c]) * oracle_half_to_double(x[c]);
            q[i] = acc;
        }
        double emax = -INFINITY;
        for (int t = 0; t <= pos; ++t) {
            double acc = 0.0;
            for (int i = 0; i < dh; ++i)
                acc += q[i] * oracle_half_to_double(kcache[((long)g * smax + t) * dh + i]);
            e[t] = acc * inv_sqrt;
            if (e[t] > emax)
                emax = e[t];
        }
        double den = 0.0;
        for (int t = 0; t <= pos; ++t)
            den += exp(e[t] - emax);
        for (int i = 0; i < dh; ++i)
            o[i] = 0.0;
        for (int t = 0; t <= pos; ++t) {
            double a = exp(e[t] - emax) / den;
            for (int i = 0; i < dh; ++i)
                o[i] += a * oracle_half_to_double(vcache[((long)g * smax + t) * dh + i]);
        }
        if (o_out)
            memcpy(o_out + (long)h * dh, o, sizeof(double) * (size_t)dh);
#pragma omp parallel for schedule(static)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int i = 0; i < dh; ++i)
                acc += o[i] * oracle_half_to_double(wot[((long)h * dh + i) * d + c]);
            y[c] += acc;
        }
    }
    free(kv);
    free(q);
    free(e);
    free(o);
    return 0;
}
