/*
 * cbq_oracle.c -- plain, slow CPU oracle for the codebook-4bit matvec.
 *
 * TEST INFRASTRUCTURE ONLY (see cbq_oracle.h): loaded by the tests, the
 * smoke check and the benchmark's CPU-baseline leg, never by the product.
 *
 * Compiled with -ffp-contract=off and without fast-math so that every fp32
 * and fp64 operation below is one correctly rounded IEEE operation, on x86-64
 * and on aarch64 alike.  Loops follow the definitions in the header, one
 * element at a time; nothing is blocked, fused or reordered.
 */
#include "cbq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* The 16 int8 levels of the 4-bit codebook, in index order. */
const int8_t oracle_codebook[16] = {
    -127, -104, -83, -65, -49, -35, -22, -10,
       1,   13,  25,  38,  53,  69,  89, 113,
};

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0 -> subnormal: fraction * 2^-24; exponent 31 -> inf/NaN;
 * otherwise (1024 + fraction) * 2^(exponent - 25). */
float oracle_half_to_float(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25);
    }
    return (float)(sign ? -mag : mag);
}

static uint16_t block_scale_bits(const uint8_t *blk)
{
    return (uint16_t)(blk[0] | (blk[1] << 8));
}

int oracle_block_index(const uint8_t *blk, int i)
{
    const uint8_t *qs = blk + 2;
    if (i < 16) return qs[i] & 0x0f;
    return qs[i - 16] >> 4;
}

void oracle_dequantize_block(const uint8_t *blk, double out[32])
{
    const double dw = (double)oracle_half_to_float(block_scale_bits(blk));
    for (int i = 0; i < ORACLE_QK; ++i)
        out[i] = dw * (double)oracle_codebook[oracle_block_index(blk, i)];
}

void oracle_quantize_act(const float *x, int64_t K, int n, int8_t *qx, float *dx)
{
    const int64_t nb = K / ORACLE_QK;
    for (int c = 0; c < n; ++c) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + (int64_t)c * K + b * ORACLE_QK;
            int8_t *qb = qx + (int64_t)c * K + b * ORACLE_QK;
            float amax = 0.0f;
            for (int i = 0; i < ORACLE_QK; ++i) {
                const float ax = fabsf(xb[i]);
                if (ax > amax) amax = ax;
            }
            const float d = amax / 127.0f;
            dx[(int64_t)c * nb + b] = d;
            for (int i = 0; i < ORACLE_QK; ++i) {
                if (d == 0.0f) {
                    qb[i] = 0;
                    continue;
                }
                float q = rintf(xb[i] / d);
                if (q > 127.0f) q = 127.0f;
                if (q < -127.0f) q = -127.0f;
                qb[i] = (int8_t)q;
            }
        }
    }
}

static int32_t block_dot(const uint8_t *blk, const int8_t *qxb)
{
    int32_t s = 0;
    for (int i = 0; i < ORACLE_QK; ++i)
        s += (int32_t)oracle_codebook[oracle_block_index(blk, i)] * (int32_t)qxb[i];
    return s;
}

void oracle_block_dots(const uint8_t *W, int64_t M, int64_t K,
                       const int8_t *qx, int n, int32_t *s)
{
    const int64_t nb = K / ORACLE_QK;
    for (int c = 0; c < n; ++c)
        for (int64_t r = 0; r < M; ++r)
            for (int64_t b = 0; b < nb; ++b)
                s[((int64_t)c * M + r) * nb + b] =
                    block_dot(W + (r * nb + b) * ORACLE_BLOCK_BYTES,
                              qx + (int64_t)c * K + b * ORACLE_QK);
}

/* One output: sum over blocks of dw * dx * s, fp64. */
static double row_dot(const uint8_t *Wrow, int64_t nb, const int8_t *qxc, const float *dxc)
{
    double acc = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = Wrow + b * ORACLE_BLOCK_BYTES;
        const double dw = (double)oracle_half_to_float(block_scale_bits(blk));
        const double s = (double)block_dot(blk, qxc + b * ORACLE_QK);
        acc += dw * (double)dxc[b] * s;
    }
    return acc;
}

/* One tolerance base: sum_i |w_i * xhat_i|. */
static double row_bound(const uint8_t *Wrow, int64_t nb, const int8_t *qxc, const float *dxc)
{
    double acc = 0.0;
    double w[ORACLE_QK];
    for (int64_t b = 0; b < nb; ++b) {
        oracle_dequantize_block(Wrow + b * ORACLE_BLOCK_BYTES, w);
        for (int i = 0; i < ORACLE_QK; ++i)
            acc += fabs(w[i] * ((double)qxc[b * ORACLE_QK + i] * (double)dxc[b]));
    }
    return acc;
}

void oracle_matvec_q(const uint8_t *W, int64_t M, int64_t K,
                     const int8_t *qx, const float *dx, int n, double *y)
{
    const int64_t nb = K / ORACLE_QK;
    for (int c = 0; c < n; ++c)
        for (int64_t r = 0; r < M; ++r)
            y[(int64_t)c * M + r] = row_dot(W + r * nb * ORACLE_BLOCK_BYTES, nb,
                                            qx + (int64_t)c * K, dx + (int64_t)c * nb);
}

void oracle_matvec_q_rows(const uint8_t *W, int64_t M, int64_t K,
                          const int8_t *qx, const float *dx, int n,
                          const int64_t *rows, int64_t nrows, double *y)
{
    const int64_t nb = K / ORACLE_QK;
    (void)M;
    for (int c = 0; c < n; ++c)
        for (int64_t i = 0; i < nrows; ++i)
            y[(int64_t)c * nrows + i] = row_dot(W + rows[i] * nb * ORACLE_BLOCK_BYTES, nb,
                                                qx + (int64_t)c * K, dx + (int64_t)c * nb);
}

void oracle_matvec(const uint8_t *W, int64_t M, int64_t K,
                   const float *x, int n, double *y)
{
    const int64_t nb = K / ORACLE_QK;
    int8_t *qx = (int8_t *)malloc((size_t)(n * K));
    float *dx = (float *)malloc((size_t)(n * nb) * sizeof(float));
    oracle_quantize_act(x, K, n, qx, dx);
    oracle_matvec_q(W, M, K, qx, dx, n, y);
    free(qx);
    free(dx);
}

void oracle_matvec_bound(const uint8_t *W, int64_t M, int64_t K,
                         const int8_t *qx, const float *dx, int n, double *bound)
{
    const int64_t nb = K / ORACLE_QK;
    for (int c = 0; c < n; ++c)
        for (int64_t r = 0; r < M; ++r)
            bound[(int64_t)c * M + r] = row_bound(W + r * nb * ORACLE_BLOCK_BYTES, nb,
                                                  qx + (int64_t)c * K, dx + (int64_t)c * nb);
}

void oracle_matvec_bound_rows(const uint8_t *W, int64_t M, int64_t K,
                              const int8_t *qx, const float *dx, int n,
                              const int64_t *rows, int64_t nrows, double *bound)
{
    const int64_t nb = K / ORACLE_QK;
    (void)M;
    for (int c = 0; c < n; ++c)
        for (int64_t i = 0; i < nrows; ++i)
            bound[(int64_t)c * nrows + i] = row_bound(W + rows[i] * nb * ORACLE_BLOCK_BYTES, nb,
                                                      qx + (int64_t)c * K, dx + (int64_t)c * nb);
}

double oracle_silu(double z)
{
    return z / (1.0 + exp(-z));
}

int oracle_moe(const uint8_t *gate_up, const uint8_t *down, int E, int64_t H, int64_t F,
               const float *h, int n_tok, const int32_t *ids, const float *wts, int k,
               int swiglu, double *y, float *a_out, int8_t *qa_out, float *da_out)
{
    const int64_t nbH = H / ORACLE_QK;
    const int64_t nbF = F / ORACLE_QK;
    const size_t gu_bytes = (size_t)(2 * F * nbH * ORACLE_BLOCK_BYTES);
    const size_t dn_bytes = (size_t)(H * nbF * ORACLE_BLOCK_BYTES);
    int8_t *qh = (int8_t *)malloc((size_t)H);
    float *dh = (float *)malloc((size_t)nbH * sizeof(float));
    float *a = (float *)malloc((size_t)F * sizeof(float));
    int8_t *qa = (int8_t *)malloc((size_t)F);
    float *da = (float *)malloc((size_t)nbF * sizeof(float));
    int bad = 0;

    for (int t = 0; t < n_tok; ++t) {
        double *yt = y + (int64_t)t * H;
        for (int64_t r = 0; r < H; ++r) yt[r] = 0.0;
        oracle_quantize_act(h + (int64_t)t * H, H, 1, qh, dh);
        for (int j = 0; j < k; ++j) {
            const int p = t * k + j;
            const int32_t e = ids[p];
            if (e < 0 || e >= E) {
                ++bad;
                if (a_out) memset(a_out + (int64_t)p * F, 0, (size_t)F * sizeof(float));
                if (qa_out) memset(qa_out + (int64_t)p * F, 0, (size_t)F);
                if (da_out) memset(da_out + (int64_t)p * nbF, 0, (size_t)nbF * sizeof(float));
                continue;
            }
            const uint8_t *gu = gate_up + (size_t)e * gu_bytes;
            const uint8_t *dn = down + (size_t)e * dn_bytes;
            for (int64_t r = 0; r < F; ++r) {
                const double g = row_dot(gu + r * nbH * ORACLE_BLOCK_BYTES, nbH, qh, dh);
                const double u = row_dot(gu + (F + r) * nbH * ORACLE_BLOCK_BYTES, nbH, qh, dh);
                a[r] = (float)(swiglu ? oracle_silu(g) * u : g * u);
            }
            oracle_quantize_act(a, F, 1, qa, da);
            if (a_out) memcpy(a_out + (int64_t)p * F, a, (size_t)F * sizeof(float));
            if (qa_out) memcpy(qa_out + (int64_t)p * F, qa, (size_t)F);
            if (da_out) memcpy(da_out + (int64_t)p * nbF, da, (size_t)nbF * sizeof(float));
            const double wj = (double)wts[p];
            for (int64_t r = 0; r < H; ++r)
                yt[r] += wj * row_dot(dn + r * nbF * ORACLE_BLOCK_BYTES, nbF, qa, da);
        }
    }
    free(qh);
    free(dh);
    free(a);
    free(qa);
    free(da);
    return bad;
}

int oracle_moe_shared(const uint8_t *gate_up, const uint8_t *down, int E, int64_t H, int64_t F,
                      const uint8_t *sh_gate_up, const uint8_t *sh_down,
                      const float *h, int n_tok, const int32_t *ids, const float *wts, int k,
                      int swiglu, double *y)
{
    const int bad = oracle_moe(gate_up, down, E, H, F, h, n_tok, ids, wts, k, swiglu, y, NULL, NULL, NULL);
    /* the shared expert as a one-expert table: every token routed to its
     * expert 0 with weight 1 */
    double *ys = (double *)malloc((size_t)n_tok * (size_t)H * sizeof(double));
    int32_t *sh_ids = (int32_t *)calloc((size_t)n_tok, sizeof(int32_t));
    float *sh_wts = (float *)malloc((size_t)n_tok * sizeof(float));
    for (int t = 0; t < n_tok; ++t) sh_wts[t] = 1.0f;
    oracle_moe(sh_gate_up, sh_down, 1, H, F, h, n_tok, sh_ids, sh_wts, 1, swiglu, ys, NULL, NULL, NULL);
    for (int64_t i = 0; i < (int64_t)n_tok * H; ++i) y[i] += ys[i];
    free(ys);
    free(sh_ids);
    free(sh_wts);
    return bad;
}

int oracle_moe_down_combine(const uint8_t *down, int E, int64_t H, int64_t F,
                            int n_tok, const int32_t *ids, const float *wts, int k,
                            const int8_t *qa, const float *da,
                            double *y, double *ybound)
{
    const int64_t nbF = F / ORACLE_QK;
    const size_t dn_bytes = (size_t)(H * nbF * ORACLE_BLOCK_BYTES);
    int bad = 0;
    for (int t = 0; t < n_tok; ++t) {
        double *yt = y + (int64_t)t * H;
        double *bt = ybound + (int64_t)t * H;
        for (int64_t r = 0; r < H; ++r) {
            yt[r] = 0.0;
            bt[r] = 0.0;
        }
        for (int j = 0; j < k; ++j) {
            const int p = t * k + j;
            const int32_t e = ids[p];
            if (e < 0 || e >= E) {
                ++bad;
                continue;
            }
            const uint8_t *dn = down + (size_t)e * dn_bytes;
            const int8_t *qap = qa + (int64_t)p * F;
            const float *dap = da + (int64_t)p * nbF;
            const double wj = (double)wts[p];
            for (int64_t r = 0; r < H; ++r) {
                const uint8_t *row = dn + r * nbF * ORACLE_BLOCK_BYTES;
                yt[r] += wj * row_dot(row, nbF, qap, dap);
                bt[r] += fabs(wj) * row_bound(row, nbF, qap, dap);
            }
        }
    }
    return bad;
}

/* Top-k by repeated selection of the largest remaining logit (the lowest
 * index among equal ones), then the softmax of the selected logits. */
void oracle_router_topk(const float *logits, int n_tok, int E, int k, int32_t *ids, double *wts) {
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    for (int t = 0; t < n_tok; ++t) {
        const float *l = logits + (int64_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            ids[t * k + j] = best;
        }
        const double lmax = (double)l[ids[t * k]];
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            const double w = exp((double)l[ids[t * k + j]] - lmax);
            wts[t * k + j] = w;
            sum += w;
        }
        for (int j = 0; j < k; ++j) wts[t * k + j] /= sum;
    }
    free(taken);
}

/* binary16 has 11 significant bits: a value in [2^(e-1), 2^e) is a multiple
 * of 2^(e-11); below 2^-14 (subnormals) every value is a multiple of 2^-24.
 * Scaling by a power of two is exact in fp64, so nearbyint() (the default
 * rounding mode: nearest, ties to even) is the one rounding. */
uint16_t oracle_float_to_half(float f)
{
    const uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    const double a = fabs((double)f);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        const double q = nearbyint(ldexp(a, 24));  /* 1024 is the smallest normal */
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e;
    frexp(a, &e);                                  /* a in [2^(e-1), 2^e) */
    double q = nearbyint(ldexp(a, 11 - e));        /* in [1024, 2048] */
    int expo = e + 14;                             /* biased exponent of 2^(e-1) */
    if (q == 2048.0) {
        q = 1024.0;
        expo += 1;
    }
    return (uint16_t)(sign | (uint16_t)(expo << 10) | (uint16_t)((int)q - 1024));
}

void oracle_quantize_weights_block(const float *w, uint8_t *blk)
{
    memset(blk, 0, ORACLE_BLOCK_BYTES);
    int imax = 0;
    for (int i = 1; i < ORACLE_QK; ++i)
        if (fabsf(w[i]) > fabsf(w[imax])) imax = i;
    const float m = w[imax];
    if (m == 0.0f) return;
    const uint16_t hb = oracle_float_to_half(m / -127.0f);
    const double dw = (double)oracle_half_to_float(hb);
    blk[0] = (uint8_t)(hb & 0xff);
    blk[1] = (uint8_t)(hb >> 8);
    for (int i = 0; i < ORACLE_QK; ++i) {
        int best = 0;
        double best_d = fabs((double)w[i] - dw * (double)oracle_codebook[0]);
        for (int j = 1; j < 16; ++j) {
            const double d = fabs((double)w[i] - dw * (double)oracle_codebook[j]);
            if (d < best_d) {
                best = j;
                best_d = d;
            }
        }
        if (i < 16) blk[2 + i] |= (uint8_t)best;
        else blk[2 + i - 16] |= (uint8_t)(best << 4);
    }
}

void oracle_quantize_weights(const float *w, int64_t M, int64_t K, uint8_t *blocks)
{
    const int64_t nb = K / ORACLE_QK;
    for (int64_t r = 0; r < M; ++r)
        for (int64_t b = 0; b < nb; ++b)
            oracle_quantize_weights_block(w + r * K + b * ORACLE_QK, blocks + (r * nb + b) * ORACLE_BLOCK_BYTES);
}

/* One matrix at a time: P = exp(c - max c), then `iters` rounds of row
 * normalisation followed by column normalisation. */
void oracle_hc_sinkhorn(const float *logits, int64_t n, int nhc, int iters, double *out) {
    const int nn = nhc * nhc;
    for (int64_t m = 0; m < n; ++m) {
        const float *c = logits + m * nn;
        double *P = out + m * nn;
        double cmax = (double)c[0];
        for (int i = 1; i < nn; ++i)
            if ((double)c[i] > cmax) cmax = (double)c[i];
        for (int i = 0; i < nn; ++i) P[i] = exp((double)c[i] - cmax);
        for (int t = 0; t < iters; ++t) {
            for (int r = 0; r < nhc; ++r) {
                double sum = 0.0;
                for (int j = 0; j < nhc; ++j) sum += P[r * nhc + j];
                for (int j = 0; j < nhc; ++j) P[r * nhc + j] /= sum;
            }
            for (int j = 0; j < nhc; ++j) {
                double sum = 0.0;
                for (int r = 0; r < nhc; ++r) sum += P[r * nhc + j];
                for (int r = 0; r < nhc; ++r) P[r * nhc + j] /= sum;
            }
        }
    }
}
