/*
 * ddpm_oracle.c -- plain, slow CPU FP64 restatement of the DDPM core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes (source: "lartpang/DynamicConvolutionOperator" README --
 * the Dynamic Dilated Pyramid Module of HDFNet, ECCV 2020):
 *
 *   - "问题与目标" (problem and goal): the math reference is three Unfolds of x
 *     plus a 1x1 generator whose output holds the dynamic kernels,
 *     N * 3 * C * K^2 * H * W values.
 *   - "CUDA 动态过滤" (dynamic filtering): one pass covers dilations (1,3,5),
 *     accumulates and writes [x, d1, d3, d5] directly; its backward forms dX
 *     and dK (the taps' gradient) without a patch matrix.
 *   - "CUDA 融合生成器推理" (fused generator inference):
 *     y tile -> dot(weight, y) -> dynamic taps -> consume with shifted x.
 *   - "CUDA Flash 式融合训练" (flash-style fused training): dX gathers each
 *     dilation's contribution with recomputed taps; dY contracts
 *     dK = shifted(x) * grad with the generator weight; dWeight / dbias are
 *     spatial reductions of dK.  BF16 taps are quantised before use.
 *
 * Notation (all tensors NCHW, contiguous, FP64 here):
 *   x, y    [B, C, H, W]         filtered input and guide features
 *   Wg      [O, C], O = 3*C*K*K  generator weight; bias [O] (may be NULL)
 *   T       [B, O, H, W]         taps, channel o = (di*C + c)*K*K + ky*K + kx
 *   out     [B, 4C, H, W]        [x, d1, d3, d5]
 *   r = K/2; tap (ky,kx) of dilation d reads x at (h+(ky-r)*d, w+(kx-r)*d),
 *   zero outside the image (Unfold with padding d*r, i.e. correlation).
 *
 * BF16 mode (bf16 != 0): inputs are already bf16-valued (exact in FP64);
 * each tap is rounded to bf16 (round to nearest, ties to even) right after
 * the generator, before it is used; everything else stays FP64.  The
 * rounding is straight-through for gradients (a dtype cast has identity
 * derivative), so backward uses the rounded taps wherever taps multiply.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "ddpm_oracle.h"

/* ---------------------------------------------------------------- bf16 -- */

/* Round a double to the nearest bfloat16 value (8 significant bits, 8
 * exponent bits, IEEE-style subnormals, ties to even), returned as a double.
 * Written from the format's definition, not from any library routine. */
double ddpmo_round_bf16(double v)
{
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    int e;
    (void)frexp(v, &e);                 /* v = m * 2^e with 0.5 <= |m| < 1 */
    /* the quantum (one unit in the last place) for 8 significant bits */
    int q = e - 8;
    if (q < -133) q = -133;             /* bf16 subnormal quantum is 2^-133 */
    double scaled = ldexp(v, -q);       /* exact: a power-of-two scale */
    double ip = nearbyint(scaled);      /* default mode: to nearest, ties even */
    double r = ldexp(ip, q);
    /* largest finite bf16 is (2 - 2^-7) * 2^127 = 255 * 2^120 */
    const double bf16_max = ldexp(255.0, 120);
    if (fabs(r) > bf16_max) return v > 0 ? INFINITY : -INFINITY;
    return r;
}

/* ------------------------------------------------------------- helpers -- */

static int shape_ok(const ddpmo_shape* s)
{
    if (!s) return 0;
    if (s->B < 1 || s->C < 1 || s->H < 1 || s->W < 1) return 0;
    if (s->K < 1 || (s->K % 2) == 0) return 0;
    for (int i = 0; i < 3; ++i)
        if (s->dil[i] < 1) return 0;
    return 1;
}

static inline int64_t n_taps(const ddpmo_shape* s) { return (int64_t)3 * s->C * s->K * s->K; }

/* x with zero padding: Unfold's padded input */
static inline double xpad(const ddpmo_shape* s, const double* x, int b, int c, int h, int w)
{
    if (h < 0 || h >= s->H || w < 0 || w >= s->W) return 0.0;
    return x[(((int64_t)b * s->C + c) * s->H + h) * s->W + w];
}

/* One generator output: T[b,o,h,w] = bias[o] + sum_j Wg[o,j] * y[b,j,h,w],
 * rounded to bf16 in BF16 mode (the 1x1 generator of "CUDA 融合生成器推理"). */
double ddpmo_tap(const ddpmo_shape* s, const double* y, const double* Wg, const double* bias,
                 int b, int o, int h, int w)
{
    const int64_t HW = (int64_t)s->H * s->W;
    double t = bias ? bias[o] : 0.0;
    const double* yp = y + (int64_t)b * s->C * HW + (int64_t)h * s->W + w;
    const double* wr = Wg + (int64_t)o * s->C;
    for (int j = 0; j < s->C; ++j) t += wr[j] * yp[j * HW];
    if (s->bf16) t = ddpmo_round_bf16(t);
    return t;
}

/* y transposed to pixel-major order yt[b][h][w][j]: the same values, laid out so
 * that the generator's dot product over j reads consecutive memory. */
static double* pixel_major(const ddpmo_shape* s, const double* y)
{
    const int64_t HW = (int64_t)s->H * s->W;
    double* yt = (double*)malloc(sizeof(double) * (size_t)s->B * (size_t)HW * (size_t)s->C);
    if (!yt) return NULL;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < s->B; ++b)
        for (int64_t p = 0; p < HW; ++p)
            for (int j = 0; j < s->C; ++j)
                yt[((int64_t)b * HW + p) * s->C + j] = y[((int64_t)b * s->C + j) * HW + p];
    return yt;
}

/* ddpmo_tap with y given pixel-major (identical arithmetic, same order of terms) */
static double tap_pm(const ddpmo_shape* s, const double* yt, const double* Wg, const double* bias,
                     int b, int o, int h, int w)
{
    double t = bias ? bias[o] : 0.0;
    const double* yp = yt + (((int64_t)b * s->H + h) * s->W + w) * s->C;
    const double* wr = Wg + (int64_t)o * s->C;
    for (int j = 0; j < s->C; ++j) t += wr[j] * yp[j];
    if (s->bf16) t = ddpmo_round_bf16(t);
    return t;
}

/* Decompose a tap channel o into (di, c, ky, kx): o = (di*C + c)*K*K + ky*K + kx */
static inline void split_tap(const ddpmo_shape* s, int o, int* di, int* c, int* ky, int* kx)
{
    const int K2 = s->K * s->K;
    const int k = o % K2;
    const int dc = o / K2;
    *di = dc / s->C;
    *c = dc % s->C;
    *ky = k / s->K;
    *kx = k % s->K;
}

static void unflatten4(int64_t idx, int d1, int d2, int d3, int* a, int* b, int* c, int* d)
{
    *d = (int)(idx % d3); idx /= d3;
    *c = (int)(idx % d2); idx /= d2;
    *b = (int)(idx % d1); idx /= d1;
    *a = (int)idx;
}

/* ----------------------------------------------------------- forward -- */

/* Generator: the materialised taps T[B,O,H,W] (the reference's second large
 * intermediate in "问题与目标"). */
int ddpmo_generate_taps(const ddpmo_shape* s, const double* y, const double* Wg, const double* bias,
                        double* T)
{
    if (!shape_ok(s)) return 1;
    const int64_t O = n_taps(s);
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < s->B; ++b)
        for (int64_t o = 0; o < O; ++o)
            for (int h = 0; h < s->H; ++h)
                for (int w = 0; w < s->W; ++w)
                    T[(((int64_t)b * O + o) * s->H + h) * s->W + w] =
                        ddpmo_tap(s, y, Wg, bias, b, (int)o, h, w);
    return 0;
}

/* One output element of the dynamic filter with taps supplied by `tapfn`.
 *   out[b, c]               = x[b, c]
 *   out[b, (1+di)*C + c]    = sum_{ky,kx} T[b, (di*C+c)*K^2 + ky*K + kx] * xpad(shifted)
 */
typedef double (*tap_fn)(const ddpmo_shape*, const void*, int b, int o, int h, int w);

static double filter_point(const ddpmo_shape* s, const double* x, tap_fn tapfn, const void* ctx,
                           int b, int ch, int h, int w)
{
    if (ch < s->C) return x[(((int64_t)b * s->C + ch) * s->H + h) * s->W + w];
    const int di = ch / s->C - 1, c = ch % s->C, K = s->K, r = K / 2, d = s->dil[di];
    double acc = 0.0;
    for (int ky = 0; ky < K; ++ky)
        for (int kx = 0; kx < K; ++kx) {
            const int o = (di * s->C + c) * K * K + ky * K + kx;
            const double xv = xpad(s, x, b, c, h + (ky - r) * d, w + (kx - r) * d);
            acc += tapfn(s, ctx, b, o, h, w) * xv;
        }
    return acc;
}

typedef struct { const double* yt; const double* Wg; const double* bias; } gen_ctx;
typedef struct { const double* T; } mat_ctx;

/* ctx.yt holds the pixel-major copy of y (see pixel_major) */
static double tap_from_generator(const ddpmo_shape* s, const void* ctx, int b, int o, int h, int w)
{
    const gen_ctx* g = (const gen_ctx*)ctx;
    return tap_pm(s, g->yt, g->Wg, g->bias, b, o, h, w);
}

static double tap_from_tensor(const ddpmo_shape* s, const void* ctx, int b, int o, int h, int w)
{
    const mat_ctx* m = (const mat_ctx*)ctx;
    return m->T[(((int64_t)b * n_taps(s) + o) * s->H + h) * s->W + w];
}

static void filter_all(const ddpmo_shape* s, const double* x, tap_fn fn, const void* ctx, double* out)
{
    const int C4 = 4 * s->C;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < s->B; ++b)
        for (int ch = 0; ch < C4; ++ch)
            for (int h = 0; h < s->H; ++h)
                for (int w = 0; w < s->W; ++w)
                    out[(((int64_t)b * C4 + ch) * s->H + h) * s->W + w] =
                        filter_point(s, x, fn, ctx, b, ch, h, w);
}

/* Fused forward: generator then filter, out [B,4C,H,W]. */
int ddpmo_forward(const ddpmo_shape* s, const double* x, const double* y, const double* Wg,
                  const double* bias, double* out)
{
    if (!shape_ok(s)) return 1;
    double* yt = pixel_major(s, y);
    if (!yt) return 2;
    gen_ctx g = {yt, Wg, bias};
    filter_all(s, x, tap_from_generator, &g, out);
    free(yt);
    return 0;
}

/* Filter with pregenerated taps T [B,O,H,W] (the taps are used as given). */
int ddpmo_filter(const ddpmo_shape* s, const double* x, const double* T, double* out)
{
    if (!shape_ok(s)) return 1;
    mat_ctx m = {T};
    filter_all(s, x, tap_from_tensor, &m, out);
    return 0;
}

/* Sampled outputs: idx[i] is a flat index into out [B,4C,H,W]. */
int ddpmo_forward_points(const ddpmo_shape* s, const double* x, const double* y, const double* Wg,
                         const double* bias, int64_t n, const int64_t* idx, double* vals)
{
    if (!shape_ok(s)) return 1;
    double* yt = pixel_major(s, y);
    if (!yt) return 2;
    gen_ctx g = {yt, Wg, bias};
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < n; ++i) {
        int b, ch, h, w;
        unflatten4(idx[i], 4 * s->C, s->H, s->W, &b, &ch, &h, &w);
        vals[i] = filter_point(s, x, tap_from_generator, &g, b, ch, h, w);
    }
    free(yt);
    return 0;
}

int ddpmo_filter_points(const ddpmo_shape* s, const double* x, const double* T, int64_t n,
                        const int64_t* idx, double* vals)
{
    if (!shape_ok(s)) return 1;
    mat_ctx m = {T};
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < n; ++i) {
        int b, ch, h, w;
        unflatten4(idx[i], 4 * s->C, s->H, s->W, &b, &ch, &h, &w);
        vals[i] = filter_point(s, x, tap_from_tensor, &m, b, ch, h, w);
    }
    return 0;
}

/* ---------------------------------------------------------- backward -- */
/*
 * Upstream gradient g [B,4C,H,W].  With the loss L = <g, out>:
 *   dK[b,o,h,w]  = g[b,(1+di)C+c,h,w] * xpad(b,c,h+(ky-r)d, w+(kx-r)d)
 *                                         ("dK = shifted(x) * grad")
 *   dbias[o]     = sum_{b,h,w} dK[b,o,h,w]
 *   dW[o,j]      = sum_{b,h,w} dK[b,o,h,w] * y[b,j,h,w]
 *   dy[b,j,h,w]  = sum_o Wg[o,j] * dK[b,o,h,w]
 *   dx[b,c,h,w]  = g[b,c,h,w]
 *                + sum_{di,ky,kx} T[b,o,h',w'] * g[b,(1+di)C+c,h',w'],
 *                  (h',w') = (h-(ky-r)d, w-(kx-r)d) inside the image
 *                  (the gather of each dilation's contribution).
 */

static inline double dK_at(const ddpmo_shape* s, const double* g, const double* x, int b, int o, int h, int w)
{
    int di, c, ky, kx;
    split_tap(s, o, &di, &c, &ky, &kx);
    const int r = s->K / 2, d = s->dil[di];
    const double gv = g[(((int64_t)b * 4 * s->C + (1 + di) * s->C + c) * s->H + h) * s->W + w];
    return gv * xpad(s, x, b, c, h + (ky - r) * d, w + (kx - r) * d);
}

/* yt: pixel-major copy of y */
static double dx_point(const ddpmo_shape* s, const double* g, const double* yt, const double* Wg,
                       const double* bias, int b, int c, int h, int w)
{
    const int K = s->K, r = K / 2, C = s->C;
    double acc = g[(((int64_t)b * 4 * C + c) * s->H + h) * s->W + w];
    for (int di = 0; di < 3; ++di) {
        const int d = s->dil[di];
        for (int ky = 0; ky < K; ++ky)
            for (int kx = 0; kx < K; ++kx) {
                const int hs = h - (ky - r) * d, ws = w - (kx - r) * d;
                if (hs < 0 || hs >= s->H || ws < 0 || ws >= s->W) continue;
                const int o = (di * C + c) * K * K + ky * K + kx;
                const double gv = g[(((int64_t)b * 4 * C + (1 + di) * C + c) * s->H + hs) * s->W + ws];
                acc += tap_pm(s, yt, Wg, bias, b, o, hs, ws) * gv;
            }
    }
    return acc;
}

/* dy at one pixel for every j: form the dK vector of the pixel once, then
 * dy[j] = sum_o Wg[o,j] * dK[o].  dk is scratch of length O. */
static void dy_pixel(const ddpmo_shape* s, const double* g, const double* x, const double* Wg,
                     int b, int h, int w, double* dk, double* dyv)
{
    const int64_t O = n_taps(s);
    for (int64_t o = 0; o < O; ++o) dk[o] = dK_at(s, g, x, b, (int)o, h, w);
    for (int j = 0; j < s->C; ++j) {
        double acc = 0.0;
        for (int64_t o = 0; o < O; ++o) acc += Wg[o * s->C + j] * dk[o];
        dyv[j] = acc;
    }
}

/* The dK plane of one tap channel o over all (b,h,w): plane[(b*H + h)*W + w]. */
static void dK_plane(const ddpmo_shape* s, const double* g, const double* x, int o, double* plane)
{
    for (int b = 0; b < s->B; ++b)
        for (int h = 0; h < s->H; ++h)
            for (int w = 0; w < s->W; ++w)
                plane[((int64_t)b * s->H + h) * s->W + w] = dK_at(s, g, x, b, o, h, w);
}

/* dW[o,j] = sum_{b,h,w} dK[b,o,h,w] * y[b,j,h,w] for one (o,j), plane = dK_plane(o) */
static double dW_from_plane(const ddpmo_shape* s, const double* plane, const double* y, int j)
{
    const int64_t HW = (int64_t)s->H * s->W;
    double acc = 0.0;
    for (int b = 0; b < s->B; ++b)
        for (int64_t p = 0; p < HW; ++p)
            acc += plane[(int64_t)b * HW + p] * y[((int64_t)b * s->C + j) * HW + p];
    return acc;
}

/* dbias[o] = sum_{b,h,w} dK[b,o,h,w] */
static double db_from_plane(const ddpmo_shape* s, const double* plane)
{
    const int64_t n = (int64_t)s->B * s->H * s->W;
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) acc += plane[i];
    return acc;
}

/* Full backward.  dbias may be NULL.  dx, dy and dW are always written. */
int ddpmo_backward(const ddpmo_shape* s, const double* g, const double* x, const double* y,
                   const double* Wg, const double* bias, double* dx, double* dy, double* dW,
                   double* dbias)
{
    if (!shape_ok(s)) return 1;
    const int B = s->B, C = s->C, H = s->H, W = s->W;
    const int64_t O = n_taps(s), HW = (int64_t)H * W, NP = (int64_t)B * HW;
    double* yt = pixel_major(s, y);
    if (!yt) return 2;
    int err = 0;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c)
            for (int h = 0; h < H; ++h)
                for (int w = 0; w < W; ++w)
                    dx[((int64_t)b * C + c) * HW + (int64_t)h * W + w] = dx_point(s, g, yt, Wg, bias, b, c, h, w);

#pragma omp parallel
    {
        double* dk = (double*)malloc(sizeof(double) * (size_t)O);
        double* dyv = (double*)malloc(sizeof(double) * (size_t)C);
        if (!dk || !dyv) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h) {
                if (!dk || !dyv) continue;
                for (int w = 0; w < W; ++w) {
                    dy_pixel(s, g, x, Wg, b, h, w, dk, dyv);
                    for (int j = 0; j < C; ++j) dy[((int64_t)b * C + j) * HW + (int64_t)h * W + w] = dyv[j];
                }
            }
        free(dk);
        free(dyv);
    }

#pragma omp parallel
    {
        double* plane = (double*)malloc(sizeof(double) * (size_t)NP);
        if (!plane) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t o = 0; o < O; ++o) {
            if (!plane) continue;
            dK_plane(s, g, x, (int)o, plane);
            for (int j = 0; j < C; ++j) dW[o * C + j] = dW_from_plane(s, plane, y, j);
            if (dbias) dbias[o] = db_from_plane(s, plane);
        }
        free(plane);
    }
    free(yt);
    return err;
}

/* ------------------------------------------------- filter-only backward -- */

/* Backward of the filter with given taps (README section "CUDA 动态过滤":
 * with the dynamic kernels already generated, the backward forms dX and dK
 * directly, without a patch matrix).  For L = <g, out>, out = filter(x, T):
 *   dT[b,o,h,w] = g[b,(1+di)C+c,h,w] * x~[b,c,h+(ky-r)d, w+(kx-r)d]      (dK)
 *   dx[b,c,h,w] = g[b,c,h,w]
 *                + sum_{di,ky,kx} T[b,o,h',w'] * g[b,(1+di)C+c,h',w'],
 *                  (h',w') = (h-(ky-r)d, w-(kx-r)d) inside the image.
 * The taps are used as given (no rounding in either mode). */
static double dx_point_given(const ddpmo_shape* s, const double* g, const double* T, int b, int c, int h, int w)
{
    const int K = s->K, r = K / 2, C = s->C;
    const int64_t HW = (int64_t)s->H * s->W;
    double acc = g[((int64_t)b * 4 * C + c) * HW + (int64_t)h * s->W + w];
    for (int di = 0; di < 3; ++di) {
        const int d = s->dil[di];
        for (int ky = 0; ky < K; ++ky)
            for (int kx = 0; kx < K; ++kx) {
                const int hs = h - (ky - r) * d, ws = w - (kx - r) * d;
                if (hs < 0 || hs >= s->H || ws < 0 || ws >= s->W) continue;
                const int64_t o = (int64_t)(di * C + c) * K * K + ky * K + kx;
                const double gv = g[((int64_t)b * 4 * C + (1 + di) * C + c) * HW + (int64_t)hs * s->W + ws];
                acc += T[((int64_t)b * n_taps(s) + o) * HW + (int64_t)hs * s->W + ws] * gv;
            }
    }
    return acc;
}

int ddpmo_filter_backward(const ddpmo_shape* s, const double* g, const double* x, const double* T, double* dx,
                          double* dT)
{
    if (!shape_ok(s)) return 1;
    const int B = s->B, C = s->C, H = s->H, W = s->W;
    const int64_t O = n_taps(s), HW = (int64_t)H * W;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c)
            for (int h = 0; h < H; ++h)
                for (int w = 0; w < W; ++w)
                    dx[((int64_t)b * C + c) * HW + (int64_t)h * W + w] = dx_point_given(s, g, T, b, c, h, w);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int64_t o = 0; o < O; ++o)
            for (int h = 0; h < H; ++h)
                for (int w = 0; w < W; ++w)
                    dT[((int64_t)b * O + o) * HW + (int64_t)h * W + w] = dK_at(s, g, x, b, (int)o, h, w);
    return 0;
}

/* Sampled gradients.  which: 0 = dx [B,C,H,W], 1 = dy [B,C,H,W],
 * 2 = dW [O,C], 3 = dbias [O]; idx are flat indices into that tensor. */
int ddpmo_backward_points(const ddpmo_shape* s, const double* g, const double* x, const double* y,
                          const double* Wg, const double* bias, int which, int64_t n,
                          const int64_t* idx, double* vals)
{
    if (!shape_ok(s) || which < 0 || which > 3) return 1;
    const int64_t O = n_taps(s), NP = (int64_t)s->B * s->H * s->W;
    double* yt = which == 0 ? pixel_major(s, y) : NULL;
    if (which == 0 && !yt) return 2;
    int err = 0;
#pragma omp parallel
    {
        double* buf = (double*)malloc(sizeof(double) * (size_t)(which == 1 ? O + s->C : NP));
        if (!buf) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n; ++i) {
            int b, c, h, w;
            if (!buf) continue;
            if (which == 0) {
                unflatten4(idx[i], s->C, s->H, s->W, &b, &c, &h, &w);
                vals[i] = dx_point(s, g, yt, Wg, bias, b, c, h, w);
            } else if (which == 1) {
                unflatten4(idx[i], s->C, s->H, s->W, &b, &c, &h, &w);
                dy_pixel(s, g, x, Wg, b, h, w, buf, buf + O);
                vals[i] = buf[O + c];
            } else if (which == 2) {
                dK_plane(s, g, x, (int)(idx[i] / s->C), buf);
                vals[i] = dW_from_plane(s, buf, y, (int)(idx[i] % s->C));
            } else {
                dK_plane(s, g, x, (int)idx[i], buf);
                vals[i] = db_from_plane(s, buf);
            }
        }
        free(buf);
    }
    free(yt);
    return err;
}

#ifdef _OPENMP
#include <omp.h>
#endif

int ddpmo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
