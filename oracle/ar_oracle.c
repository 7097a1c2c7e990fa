/*
 * Plain CPU oracle for the depth-routing read (test infrastructure only).
 *
 * This file is the checker, not the product: only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg call it. It shares no
 * code, header or constant with the CUDA path.
 *
 * Everything is written as the definitions read, one token at a time (tokens
 * are independent: the attention runs over depth, not over tokens), in one
 * arithmetic type `real`: float64 for the parity reference (the default
 * build), float32 for the timed CPU baseline (built with -DORC_FLOAT; the
 * same source, so the two builds differ only in precision). OpenMP, when
 * available, only splits the token loop.
 *
 * Notation (per token; N sources s_0..s_{N-1} in R^d; H heads):
 *   key coordinates   : the last r of the d coordinates (r = d is the plain
 *                       full-width key of "Multi-Head Attention Residuals",
 *                       Eq. 3; r < d is the sliced key of "Low-Rank Attention
 *                       Residuals", Eq. 11);
 *   value slice of h  : coordinates [h*d/H, (h+1)*d/H)            (MHAR Eq. 3)
 *   key slice of h    : coordinates d-r + [h*r/H, (h+1)*r/H)
 *   inv_n             : (mean over the RMS coordinates of s_n^2 + eps)^(-1/2);
 *                       the RMS coordinates are the key coordinates
 *                       ("slice" norm, LR-AttnRes Eq. 13 first line) or all d
 *                       ("full" norm: MHAR Appendix E, and the full-width-RMS
 *                       control of LR-AttnRes Eq. 13 second line)
 *   z_{n,h}           : inv_n * sum_{c in key slice h} q_c g_c s_{n,c}
 *   alpha_{n,h}       : softmax over n of z_{.,h}                    (Eq. 2/3)
 *   out_c             : sum_n alpha_{n,h(c)} s_{n,c}                   (Eq. 3)
 *   lse_h             : max_n z + log sum_n exp(z - max)
 */
#include <stdint.h>
#include <tgmath.h> /* exp, log, sqrt follow the type of their argument */
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifdef ORC_FLOAT
typedef float real;
#else
typedef double real;
#endif

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_NO_MEMORY 2

/* Bytes of the arithmetic type this file was compiled with (8: float64, 4: float32). */
int orc_real_bytes(void) { return (int)sizeof(real); }

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int check_shape(int N, int64_t T, int d, int r, int H)
{
    if (N < 1 || T < 0 || d < 1 || r < 1 || r > d || H < 1) return ORC_BAD_ARG;
    if (d % H != 0 || r % H != 0) return ORC_BAD_ARG;
    return ORC_OK;
}

/* Inverse RMS of one token's vector over the RMS coordinates.
 * "Multi-Head Attention Residuals", Appendix E: r = (||s||^2/d + eps)^(-1/2);
 * "Low-Rank Attention Residuals", Eq. 13 (slice: over the last r coordinates). */
static real inv_rms_one(const real *x, int d, int r, int full_width, real eps)
{
    int c0 = full_width ? 0 : d - r;
    int w = d - c0;
    real ss = (real)0;
    for (int c = c0; c < d; ++c) ss += x[c] * x[c];
    return (real)1 / sqrt(ss / (real)w + eps);
}

/* inv[t] for every token of one [T,d] source. */
int orc_inv_rms(const real *x, int64_t T, int d, int r, int full_width, double eps, real *inv)
{
    if (check_shape(1, T, d, r, 1)) return ORC_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) inv[t] = inv_rms_one(x + t * d, d, r, full_width, (real)eps);
    return ORC_OK;
}

/*
 * Forward of one routing site ("Multi-Head Attention Residuals", Eq. 3 and
 * Figure 3; "Low-Rank Attention Residuals", Eq. 8-11 for r < d).
 *   src[n]  : [T,d] source n            q, g : [r]
 *   out     : [T,d]   lse : [T,H]       alpha: [T,N,H] or NULL
 * Softmax is the explicit two-pass form: max, then normalised exponentials.
 */
int orc_route_fwd(const real *const *src, int N, int64_t T, int d, int r, int H,
                  int full_width, double eps, const real *q, const real *g,
                  real *out, real *lse, real *alpha)
{
    if (check_shape(N, T, d, r, H)) return ORC_BAD_ARG;
    const int K = d / H, Kr = r / H, c_key = d - r;
    int bad = 0;
#pragma omp parallel
    {
        real *z = (real *)malloc(sizeof(real) * (size_t)N * H);
        real *a = (real *)malloc(sizeof(real) * (size_t)N * H);
        if (!z || !a) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            if (!z || !a) continue;
            /* scores z_{n,h} = q_h . RMSNorm(s_n)_[h] (g folded into the key) */
            for (int n = 0; n < N; ++n) {
                const real *s = src[n] + t * d;
                real inv = inv_rms_one(s, d, r, full_width, (real)eps);
                for (int h = 0; h < H; ++h) {
                    real dot = (real)0;
                    for (int k = 0; k < Kr; ++k) {
                        int j = h * Kr + k; /* index into q, g */
                        dot += q[j] * (g ? g[j] : (real)1) * s[c_key + j];
                    }
                    z[n * H + h] = inv * dot;
                }
            }
            /* softmax over sources, per head */
            for (int h = 0; h < H; ++h) {
                real m = z[h];
                for (int n = 1; n < N; ++n)
                    if (z[n * H + h] > m) m = z[n * H + h];
                real sum = (real)0;
                for (int n = 0; n < N; ++n) sum += exp(z[n * H + h] - m);
                for (int n = 0; n < N; ++n) a[n * H + h] = exp(z[n * H + h] - m) / sum;
                lse[t * H + h] = m + log(sum);
            }
            /* mix: each head mixes only its own value slice */
            for (int c = 0; c < d; ++c) {
                int h = c / K;
                real acc = (real)0;
                for (int n = 0; n < N; ++n) acc += a[n * H + h] * src[n][t * d + c];
                out[t * d + c] = acc;
            }
            if (alpha) memcpy(alpha + t * (int64_t)N * H, a, sizeof(real) * (size_t)N * H);
        }
        free(z);
        free(a);
    }
    return bad ? ORC_NO_MEMORY : ORC_OK;
}

/*
 * Backward of one routing site, written from the value/routing decomposition
 * of "Low-Rank Attention Residuals", Eq. 15 and Lemma 2 (Eq. 20), applied to
 * each head's own softmax:
 *   dL/ds_n = sum_h [ alpha_{n,h} G_[h]  +  alpha_{n,h} <G_[h], s_{n,[h]} - out_[h]> grad z_{n,h} ]
 * with G = dL/dout, and the score gradient of Eq. 21 (slice norm) or Eq. 22
 * (full-width norm), extended by the head's key slice and the norm weight g:
 *   grad z_{n,h} = inv_n (q g) on key slice h  -  inv_n^3 zraw_{n,h} s_n / w  on the RMS coordinates,
 *   zraw_{n,h}   = sum_{c in key slice h} q_c g_c s_{n,c},  w = width of the RMS coordinates.
 * Query and norm-weight gradients follow from z = inv * sum q g s
 * ("Multi-Head Attention Residuals", Appendix E, dq and dg):
 *   dq_c = sum_{t,n} fb_{n,h(c)} inv_n g_c s_{n,c},   dg_c = sum_{t,n} fb_{n,h(c)} inv_n q_c s_{n,c},
 * where fb_{n,h} = alpha_{n,h} <G_[h], s_{n,[h]} - out_[h]> is the routing feedback.
 *   fwd_out : [T,d] or NULL. NULL: out in the feedback is the read itself,
 *             recomputed here (the definition). Otherwise out_[h] in the
 *             feedback is taken from this array: the forward output a
 *             one-pass backward is given (as stored, e.g. rounded to bf16),
 *             where "Multi-Head Attention Residuals", Appendix E (Figure 10)
 *             accumulates the coupling sum_n alpha <G_[h], s_{n,[h]}> over the
 *             sources in a first pass.
 *   dsrc[n] : [T,d], ADDED to (the caller zeroes it; a row read by several
 *             sites sums their contributions)
 *   dq, dg  : [r], overwritten; dg may be NULL. g may be NULL (= ones).
 */
int orc_route_bwd(const real *const *src, int N, int64_t T, int d, int r, int H,
                  int full_width, double eps, const real *q, const real *g,
                  const real *dout, const real *fwd_out, real *const *dsrc, real *dq, real *dg)
{
    if (check_shape(N, T, d, r, H)) return ORC_BAD_ARG;
    const int K = d / H, Kr = r / H, c_key = d - r;
    const int c_rms = full_width ? 0 : d - r, w_rms = d - c_rms;
    for (int j = 0; j < r; ++j) {
        dq[j] = (real)0;
        if (dg) dg[j] = (real)0;
    }
    int bad = 0;
#pragma omp parallel
    {
        size_t nh = (size_t)N * H;
        real *inv = (real *)malloc(sizeof(real) * N);
        real *zraw = (real *)malloc(sizeof(real) * nh);
        real *a = (real *)malloc(sizeof(real) * nh);
        real *fb = (real *)malloc(sizeof(real) * nh);
        real *o = (real *)malloc(sizeof(real) * d);
        real *dq_p = (real *)calloc((size_t)r, sizeof(real));
        real *dg_p = (real *)calloc((size_t)r, sizeof(real));
        int ok = inv && zraw && a && fb && o && dq_p && dg_p;
        if (!ok) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            if (!ok) continue;
            const real *G = dout + t * d;
            /* recompute the forward of this token: inv, raw scores, alpha, out */
            for (int n = 0; n < N; ++n) {
                const real *s = src[n] + t * d;
                inv[n] = inv_rms_one(s, d, r, full_width, (real)eps);
                for (int h = 0; h < H; ++h) {
                    real dot = (real)0;
                    for (int k = 0; k < Kr; ++k) {
                        int j = h * Kr + k;
                        dot += q[j] * (g ? g[j] : (real)1) * s[c_key + j];
                    }
                    zraw[n * H + h] = dot;
                }
            }
            for (int h = 0; h < H; ++h) {
                real m = inv[0] * zraw[h];
                for (int n = 1; n < N; ++n) {
                    real zz = inv[n] * zraw[n * H + h];
                    if (zz > m) m = zz;
                }
                real sum = (real)0;
                for (int n = 0; n < N; ++n) sum += exp(inv[n] * zraw[n * H + h] - m);
                for (int n = 0; n < N; ++n) a[n * H + h] = exp(inv[n] * zraw[n * H + h] - m) / sum;
            }
            for (int c = 0; c < d; ++c) {
                int h = c / K;
                real acc = (real)0;
                for (int n = 0; n < N; ++n) acc += a[n * H + h] * src[n][t * d + c];
                o[c] = fwd_out ? fwd_out[t * d + c] : acc;
            }
            /* routing feedback fb_{n,h} = alpha <G_[h], s_[h] - out_[h]>  (Eq. 15, 20) */
            for (int n = 0; n < N; ++n) {
                const real *s = src[n] + t * d;
                for (int h = 0; h < H; ++h) {
                    real dot = (real)0;
                    for (int c = h * K; c < (h + 1) * K; ++c) dot += G[c] * (s[c] - o[c]);
                    fb[n * H + h] = a[n * H + h] * dot;
                }
            }
            for (int n = 0; n < N; ++n) {
                const real *s = src[n] + t * d;
                real *ds = dsrc[n] + t * d;
                /* direct value gradient alpha_{n,h(c)} G_c */
                for (int c = 0; c < d; ++c) ds[c] += a[n * H + c / K] * G[c];
                /* routing feedback times the score gradient (Eq. 21 / 22) */
                real iv = inv[n], iv3 = iv * iv * iv;
                for (int h = 0; h < H; ++h) {
                    real f = fb[n * H + h];
                    for (int k = 0; k < Kr; ++k) {
                        int j = h * Kr + k, c = c_key + j;
                        ds[c] += f * iv * q[j] * (g ? g[j] : (real)1);
                        dq_p[j] += f * iv * (g ? g[j] : (real)1) * s[c];
                        dg_p[j] += f * iv * q[j] * s[c];
                    }
                    real coef = f * iv3 * zraw[n * H + h] / (real)w_rms;
                    for (int c = c_rms; c < d; ++c) ds[c] -= coef * s[c];
                }
            }
        }
        if (ok) {
#pragma omp critical
            {
                for (int j = 0; j < r; ++j) {
                    dq[j] += dq_p[j];
                    if (dg) dg[j] += dg_p[j];
                }
            }
        }
        free(inv);
        free(zraw);
        free(a);
        free(fb);
        free(o);
        free(dq_p);
        free(dg_p);
    }
    return bad ? ORC_NO_MEMORY : ORC_OK;
}
