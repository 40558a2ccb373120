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

/* ------------------------------------------------------------------------
 * Transposed convolution: the adjoint (matrix transpose) of the convolution
 * with the same S, P, D, G.  "Convolution variants and their matrix
 * operations" (lpnh.cn/news/2674933), sections 2.3 and 4.2: it upsamples, it
 * is still a convolution, and in matrix form the weight matrix enters
 * transposed (Y_col = W^T X); equivalently s-1 zeros are inserted between
 * neighbouring input pixels before a stride-1 convolution.  Each input pixel
 * (i, j) of channel ci = g*C_in/G + ci' adds x * w[ci][co'][kh][kw] to output
 * (i*S + kh*D - P, j*S + kw*D - P) of channel co = g*C_out/G + co'; positions
 * outside the output are dropped.  The weight is indexed [C_in][C_out/G][Kh][Kw]
 * here: the desc's ws_o strides ci, ws_i strides co'.  Output extent
 * (H - 1)*S - 2P + D*(Kh - 1) + 1 (section 6.2 says only that it differs from
 * the convolution's; this is the adjoint's size, with no output padding).
 * ------------------------------------------------------------------------ */
int oracle_out_size_transposed(int in, int k, int s, int p, int d)
{
    if (in <= 0 || k <= 0 || s <= 0 || p < 0 || d <= 0) return 0;
    long v = (long)(in - 1) * s - 2L * p + (long)d * (k - 1) + 1;
    return v > 0 ? (int)v : 0;
}

/* Full output, scatter order (each input pixel stamps its weighted kernel). */
int oracle_conv_transpose2d_f64(const oracle_conv_desc *c, const double *x, const double *w,
                                const double *scale, const double *bias, double *y, int nthreads)
{
    if (check_desc(c)) return -1;
    const int Ho = oracle_out_size_transposed(c->H, c->Kh, c->S, c->P, c->D);
    const int Wo = oracle_out_size_transposed(c->W, c->Kw, c->S, c->P, c->D);
    if (Ho <= 0 || Wo <= 0) return -1;
    const int cin_g = c->C_in / c->G, cout_g = c->C_out / c->G;
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
        const int g = co / cout_g, cop = co % cout_g;
        double *yp = y + n * c->ys_n + co * c->ys_c;
        for (int h = 0; h < Ho; ++h)
            for (int v = 0; v < Wo; ++v) yp[h * c->ys_h + v * c->ys_w] = 0.0;
        for (int cp = 0; cp < cin_g; ++cp) {
            const int ci = g * cin_g + cp;
            for (int i = 0; i < c->H; ++i)
                for (int j = 0; j < c->W; ++j) {
                    const double xv = x[n * c->xs_n + ci * c->xs_c + i * c->xs_h + j * c->xs_w];
                    for (int kh = 0; kh < c->Kh; ++kh) {
                        const int h = i * c->S + kh * c->D - c->P;
                        if (h < 0 || h >= Ho) continue;
                        for (int kw = 0; kw < c->Kw; ++kw) {
                            const int v = j * c->S + kw * c->D - c->P;
                            if (v < 0 || v >= Wo) continue;
                            yp[h * c->ys_h + v * c->ys_w] +=
                                xv * w[ci * c->ws_o + cop * c->ws_i + kh * c->ws_h + kw * c->ws_w];
                        }
                    }
                }
        }
        for (int h = 0; h < Ho; ++h)
            for (int v = 0; v < Wo; ++v) {
                double a = yp[h * c->ys_h + v * c->ys_w];
                if (scale) a *= scale[co];
                if (bias) a += bias[co];
                if (c->relu && a < 0.0) a = 0.0;
                yp[h * c->ys_h + v * c->ys_w] = a;
            }
    }
    return 0;
}

/* Selected outputs, gather order: output (h, v) takes input row i = (h + P - kh*D)/S
 * for every kh where that division is exact and i is inside the input (same for
 * columns).  pts holds (n, co, h, v) quadruples. */
int oracle_conv_transpose2d_points_f64(const oracle_conv_desc *c, const double *x, const double *w,
                                       const double *scale, const double *bias, const int64_t *pts,
                                       int64_t npts, double *out, int nthreads)
{
    if (check_desc(c)) return -1;
    const int Ho = oracle_out_size_transposed(c->H, c->Kh, c->S, c->P, c->D);
    const int Wo = oracle_out_size_transposed(c->W, c->Kw, c->S, c->P, c->D);
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t *q = pts + 4 * i;
        if (q[0] < 0 || q[0] >= c->N || q[1] < 0 || q[1] >= c->C_out ||
            q[2] < 0 || q[2] >= Ho || q[3] < 0 || q[3] >= Wo) return -1;
    }
    const int cin_g = c->C_in / c->G, cout_g = c->C_out / c->G;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < npts; ++t) {
        const int64_t *q = pts + 4 * t;
        const int n = (int)q[0], co = (int)q[1], h = (int)q[2], v = (int)q[3];
        const int g = co / cout_g, cop = co % cout_g;
        double acc = 0.0;
        for (int cp = 0; cp < cin_g; ++cp) {
            const int ci = g * cin_g + cp;
            for (int kh = 0; kh < c->Kh; ++kh) {
                const int nh = h + c->P - kh * c->D;
                if (nh < 0 || nh % c->S) continue;
                const int i = nh / c->S;
                if (i >= c->H) continue;
                for (int kw = 0; kw < c->Kw; ++kw) {
                    const int nv = v + c->P - kw * c->D;
                    if (nv < 0 || nv % c->S) continue;
                    const int j = nv / c->S;
                    if (j >= c->W) continue;
                    acc += x[n * c->xs_n + ci * c->xs_c + i * c->xs_h + j * c->xs_w] *
                           w[ci * c->ws_o + cop * c->ws_i + kh * c->ws_h + kw * c->ws_w];
                }
            }
        }
        if (scale) acc *= scale[co];
        if (bias) acc += bias[co];
        if (c->relu && acc < 0.0) acc = 0.0;
        out[t] = acc;
    }
    return 0;
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
