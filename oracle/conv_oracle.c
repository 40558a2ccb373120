/*
 * conv_oracle.c -- FP64 CPU oracle for the forward 2D convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA path is checked against.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load it.  It shares no code, header or
 * constant with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (the plain definition, no blocking, no reordering):
 *
 *   y[n][co][ho][wo] = bias[co]
 *       + sum_{ci'=0}^{C_in/G-1} sum_{kh} sum_{kw}
 *             x[n][g*C_in/G + ci'][ho*S + kh*D - P][wo*S + kw*D - P]
 *           * w[co][ci'][kh][kw]
 *   with g = co / (C_out/G); taps whose input coordinate falls outside
 *   [0,H) x [0,W) contribute nothing; then ReLU if requested.
 *
 *   With a per-channel scale (folded batch normalisation) the sum is first
 *   multiplied by scale[co], then bias[co] is added, then the activation:
 *   y = act(scale[co] * sum + bias[co]).
 *
 * Sources:
 *   - the dot-product definition and the index map h_i = h_o*S_h + k_h - P_h:
 *     "GPU lesson 9: how a GPU executes neural-network convolution"
 *     (lincklin.cn), section 2 and its equations;
 *   - dilation k*D in the index and the effective kernel K + (K-1)(D-1):
 *     "Convolution variants and their matrix operations" (lpnh.cn/news/2674933),
 *     sections 2.3 and 4.2 (the formula is printed garbled there; the reading
 *     used is K + (K-1)(D-1));
 *   - zero padding as an address predicate (no padded copy): lesson 9, section 26;
 *   - output size floor((H + 2P - D(K-1) - 1)/S) + 1: variants page, section 6.2
 *     (printed garbled; this is the reading used);
 *   - groups as G independent convolutions on contiguous channel blocks:
 *     variants page, sections 2.2 and 4.3; depthwise is G = C_in (lesson 9,
 *     section 23);
 *   - bias added after the sum, then the activation: lesson 9, section 31;
 *     the same section's per-channel scale and shift (a folded batch norm)
 *     multiply the sum before the shift is added.
 *
 * Loop order follows the seven-loop nest of lesson 9, section 34
 * (n, co, ho, wo outer; ci, kh, kw inner), parallelised over (n, co) with
 * OpenMP.  Tensors are addressed through element strides so that the same
 * oracle reads NCHW or NHWC buffers; the layout is stride arithmetic only.
 */
#include <stdint.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int N, C_in, H, W, C_out, Kh, Kw, S, P, D, G;
    int relu;
    /* element strides */
    int64_t xs_n, xs_c, xs_h, xs_w;      /* x[n][c][h][w]          */
    int64_t ws_o, ws_i, ws_h, ws_w;      /* w[co][ci'][kh][kw]     */
    int64_t ys_n, ys_c, ys_h, ys_w;      /* y[n][co][ho][wo]       */
} oracle_conv_desc;

/* Output extent along one spatial axis; 0 when the window never fits. */
int oracle_out_size(int in, int k, int s, int p, int d)
{
    if (in <= 0 || k <= 0 || s <= 0 || p < 0 || d <= 0) return 0;
    long num = (long)in + 2L * p - (long)d * (k - 1) - 1;
    if (num < 0) return 0;
    return (int)(num / s + 1);
}

/* One output element, summed in the definition's order.  When macs is
 * non-NULL it receives the number of multiply terms actually taken. */
static double one_output(const oracle_conv_desc *c, const double *x,
                         const double *w, const double *scale, const double *bias,
                         int n, int co, int ho, int wo, long *macs)
{
    const int cin_g = c->C_in / c->G;
    const int cout_g = c->C_out / c->G;
    const int g = co / cout_g;
    double acc = 0.0;
    long count = 0;
    for (int ci = 0; ci < cin_g; ++ci) {
        const int cin = g * cin_g + ci;
        for (int kh = 0; kh < c->Kh; ++kh) {
            const int hi = ho * c->S + kh * c->D - c->P;
            if (hi < 0 || hi >= c->H) continue;          /* zero padding */
            for (int kw = 0; kw < c->Kw; ++kw) {
                const int wi = wo * c->S + kw * c->D - c->P;
                if (wi < 0 || wi >= c->W) continue;      /* zero padding */
                const double xv = x[n * c->xs_n + cin * c->xs_c + hi * c->xs_h + wi * c->xs_w];
                const double wv = w[co * c->ws_o + ci * c->ws_i + kh * c->ws_h + kw * c->ws_w];
                acc += xv * wv;
                ++count;
            }
        }
    }
    if (scale) acc *= scale[co];
    if (bias) acc += bias[co];
    if (c->relu && acc < 0.0) acc = 0.0;
    if (macs) *macs = count;
    return acc;
}

static int check_desc(const oracle_conv_desc *c)
{
    if (c->N <= 0 || c->C_in <= 0 || c->H <= 0 || c->W <= 0 || c->C_out <= 0) return -1;
    if (c->Kh <= 0 || c->Kw <= 0 || c->S <= 0 || c->P < 0 || c->D <= 0 || c->G <= 0) return -1;
    if (c->C_in % c->G || c->C_out % c->G) return -1;
    return 0;
}

/* Full output; scale may be NULL (no scaling).  Returns 0, or -1 on a bad descriptor. */
int oracle_conv2d_f64(const oracle_conv_desc *c, const double *x, const double *w,
                      const double *scale, const double *bias, double *y, int nthreads)
{
    if (check_desc(c)) return -1;
    const int Ho = oracle_out_size(c->H, c->Kh, c->S, c->P, c->D);
    const int Wo = oracle_out_size(c->W, c->Kw, c->S, c->P, c->D);
    if (Ho <= 0 || Wo <= 0) return -1;
    const long total = (long)c->N * c->C_out;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long nc = 0; nc < total; ++nc) {
        const int n = (int)(nc / c->C_out);
        const int co = (int)(nc % c->C_out);
        for (int ho = 0; ho < Ho; ++ho)
            for (int wo = 0; wo < Wo; ++wo)
                y[n * c->ys_n + co * c->ys_c + ho * c->ys_h + wo * c->ys_w] =
                    one_output(c, x, w, scale, bias, n, co, ho, wo, 0);
    }
    return 0;
}

/* Selected outputs: pts holds npts quadruples (n, co, ho, wo); out[i] gets
 * the value at pts[i].  Returns 0, or -1 on a bad descriptor or point. */
int oracle_conv2d_points_f64(const oracle_conv_desc *c, const double *x, const double *w,
                             const double *scale, const double *bias, const int64_t *pts,
                             int64_t npts, double *out, int nthreads)
{
    if (check_desc(c)) return -1;
    const int Ho = oracle_out_size(c->H, c->Kh, c->S, c->P, c->D);
    const int Wo = oracle_out_size(c->W, c->Kw, c->S, c->P, c->D);
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t *q = pts + 4 * i;
        if (q[0] < 0 || q[0] >= c->N || q[1] < 0 || q[1] >= c->C_out ||
            q[2] < 0 || q[2] >= Ho || q[3] < 0 || q[3] >= Wo) return -1;
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t *q = pts + 4 * i;
        out[i] = one_output(c, x, w, scale, bias, (int)q[0], (int)q[1], (int)q[2], (int)q[3], 0);
    }
    return 0;
}

/* Number of multiply terms the oracle takes for output (n, co, ho, wo). */
long oracle_conv2d_macs_at(const oracle_conv_desc *c, const double *x, const double *w,
                           int n, int co, int ho, int wo)
{
    if (check_desc(c)) return -1;
    long macs = 0;
    (void)one_output(c, x, w, 0, 0, n, co, ho, wo, &macs);
    return macs;
}

/* Threads the OpenMP runtime would use (1 when built without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
