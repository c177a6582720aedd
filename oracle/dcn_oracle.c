/*
 * Oracle for the forward pass of modulated deformable convolution and its
 * gradients (the backward pass, at the end of this file).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never links, calls or includes it, and it shares no code
 * with the CUDA sources.
 *
 * What it computes (page "litert-community/Idol ... deform_conv.py", module
 * docstring and the four-corner loop of deform_conv2d_gather; page "deformops
 * 3.0.1", section "Deformable convolution": torchvision deform_conv2d with a
 * (C_out, C_in / groups, kH, kW) weight, v2 with a mask, v1 without).  For
 * image b, output channel o and output pixel (h, w):
 *
 *   out[b,o,h,w] = bias[o] + sum_{i<kh} sum_{j<kw} sum_{c in group(o)}
 *                  weight[o,c - c0(o),i,j] * m * S(b, c, py, px)
 *
 *   k  = i*kw + j                           (row-major taps)
 *   g  = o / (O/groups), channels of group g: c0 = g*(C/groups) .. +C/groups
 *   q  = c / (C/offset_groups)              (the channel's offset group)
 *   dy = offset[b, 2*kh*kw*q + 2k,   h, w]  (vertical shift first)
 *   dx = offset[b, 2*kh*kw*q + 2k+1, h, w]
 *   m  = mask[b, kh*kw*q + k, h, w]         (1 when no mask is given)
 *   py = (h*stride_h - pad_h + i*dil_h) + dy
 *   px = (w*stride_w - pad_w + j*dil_w) + dx
 *   S  = sum over the four corners (y0+a, x0+e), a,e in {0,1}, with
 *        y0 = floor(py), x0 = floor(px), ly = py - y0, lx = px - x0,
 *        of wy_a * wx_e * x[b, c, y0+a, x0+e], where wy_0 = 1-ly, wy_1 = ly,
 *        wx_0 = 1-lx, wx_1 = lx, and a corner outside [0,H-1]x[0,W-1]
 *        contributes nothing.
 *   Ho = (H + 2*pad_h - dil_h*(kh-1) - 1) / stride_h + 1, likewise Wo.
 *
 * The pages fix stride 1, dilation 1, one padding, one weight group and one
 * offset group for the page-1 routine; the general form is the plain
 * convolution reading of those parameters (the torchvision operator the
 * deformops page names), with each offset group laid out like the
 * single-group offsets, one block after another.
 *
 * Precision: the sampling coordinate py/px is formed in fp32, the dtype in
 * which the page builds its sampling grid (the offsets are fp32), so that
 * the integer floor(py) is decided in the same precision as on the GPU.
 * Everything after that (corner weights, products, all sums) is fp64, in
 * the fixed order o -> (i, j) -> c -> corner (0,0), (0,1), (1,0), (1,1).
 * The geometry of a tap is computed once per offset group.
 * Non-finite or huge coordinates make every corner invalid (the comparisons
 * are done in double), so they contribute 0 and never index memory.
 *
 * Layouts (all dense, row-major, host memory; G = offset_groups):
 *   x      [B, C, H, W]          fp32 (bf16 inputs are passed as their exact
 *                                fp32 values)
 *   offset [B, 2*G*kh*kw, Ho, Wo] fp32
 *   mask   [B, G*kh*kw, Ho, Wo]  fp32, or NULL
 *   weight [O, C/groups, kh, kw] fp32
 *   bias   [O]                   fp32, or NULL
 *   out    [B, O, Ho, Wo]        fp64
 *
 * Parity of every part of this definition is pinned by the CPU tests:
 * zero offsets against a library direct convolution (with stride,
 * padding, dilation and groups), integer offsets against a shifted
 * convolution, fractional offsets against hand-derived bilinear values and
 * against a library bilinear resampler (per offset group), out-of-image
 * samples against the bias, and the mask against linearity.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    const float *x, *offset, *mask, *weight, *bias;
    int B, C, H, W, O, kh, kw;
    int sh, sw, ph, pw, dh, dw, groups, ogroups;
    int Ho, Wo;
} oracle_problem;

/* All O output channels of output pixel (b, h, w). */
static void oracle_pixel(const oracle_problem *p, int b, int h, int w,
                         double *out, ptrdiff_t out_stride)
{
    const int k_total = p->kh * p->kw;
    const size_t plane_out = (size_t)p->Ho * p->Wo;
    const size_t pix = (size_t)h * p->Wo + w;
    const int Cg = p->C / p->groups;       /* input channels per weight group */
    const int Og = p->O / p->groups;       /* output channels per weight group */
    const int Cq = p->C / p->ogroups;      /* channels per offset group */

    for (int o = 0; o < p->O; ++o) {
        const int g = o / Og;
        const int c_end = (g + 1) * Cg;
        double acc = 0.0;
        for (int i = 0; i < p->kh; ++i) {
            for (int j = 0; j < p->kw; ++j) {
                const int k = i * p->kw + j;
                int c = g * Cg;
                while (c < c_end) {
                    /* the channels of this weight group in offset group q */
                    const int q = c / Cq;
                    const int q_end = (q + 1) * Cq < c_end ? (q + 1) * Cq : c_end;
                    const size_t oq = (size_t)b * p->ogroups + q;
                    const float dy = p->offset[(oq * 2 * k_total + 2 * k) * plane_out + pix];
                    const float dx = p->offset[(oq * 2 * k_total + 2 * k + 1) * plane_out + pix];
                    const double m = p->mask
                        ? (double)p->mask[(oq * k_total + k) * plane_out + pix]
                        : 1.0;
                    /* fp32 sampling coordinate, as in the page's grid */
                    const float py = (float)(h * p->sh - p->ph + i * p->dh) + dy;
                    const float px = (float)(w * p->sw - p->pw + j * p->dw) + dx;
                    const float fy0 = floorf(py);
                    const float fx0 = floorf(px);
                    const double ly = (double)py - (double)fy0;
                    const double lx = (double)px - (double)fx0;
                    const double wy[2] = {1.0 - ly, ly};
                    const double wx[2] = {1.0 - lx, lx};

                    for (; c < q_end; ++c) {
                        const float *xc = p->x + ((size_t)b * p->C + c) * p->H * p->W;
                        double s = 0.0;
                        for (int a = 0; a < 2; ++a) {
                            for (int e = 0; e < 2; ++e) {
                                const double yy = (double)fy0 + a;
                                const double xx = (double)fx0 + e;
                                if (yy >= 0.0 && yy <= p->H - 1 && xx >= 0.0 && xx <= p->W - 1) {
                                    s += wy[a] * wx[e] * (double)xc[(size_t)yy * p->W + (size_t)xx];
                                }
                            }
                        }
                        const double wt = p->weight[(((size_t)o * Cg + (c - g * Cg)) * p->kh + i) * p->kw + j];
                        acc += wt * m * s;
                    }
                }
            }
        }
        out[o * out_stride] = acc + (p->bias ? (double)p->bias[o] : 0.0);
    }
}

static int oracle_check(const oracle_problem *p)
{
    if (!p->x || !p->offset || !p->weight) return -1;
    if (p->B <= 0 || p->C <= 0 || p->H <= 0 || p->W <= 0 || p->O <= 0) return -1;
    if (p->kh <= 0 || p->kw <= 0 || p->ph < 0 || p->pw < 0) return -1;
    if (p->sh <= 0 || p->sw <= 0 || p->dh <= 0 || p->dw <= 0) return -1;
    if (p->groups <= 0 || p->C % p->groups || p->O % p->groups) return -1;
    if (p->ogroups <= 0 || p->C % p->ogroups) return -1;
    if (p->Ho <= 0 || p->Wo <= 0) return -1;
    return 0;
}

/* desc = {B, C, H, W, O, kh, kw, stride_h, stride_w, pad_h, pad_w,
 *         dil_h, dil_w, groups, offset_groups} */
static oracle_problem oracle_make(const float *x, const float *offset, const float *mask,
                                  const float *weight, const float *bias, const int *d)
{
    oracle_problem p = {x, offset, mask, weight, bias,
                        d[0], d[1], d[2], d[3], d[4], d[5], d[6],
                        d[7], d[8], d[9], d[10], d[11], d[12], d[13], d[14], 0, 0};
    if (p.sh > 0 && p.sw > 0) {
        p.Ho = (p.H + 2 * p.ph - p.dh * (p.kh - 1) - 1) / p.sh + 1;
        p.Wo = (p.W + 2 * p.pw - p.dw * (p.kw - 1) - 1) / p.sw + 1;
        if (p.H + 2 * p.ph - p.dh * (p.kh - 1) - 1 < 0) p.Ho = 0;
        if (p.W + 2 * p.pw - p.dw * (p.kw - 1) - 1 < 0) p.Wo = 0;
    }
    return p;
}

#ifdef _OPENMP
#define ORACLE_SET_THREADS(n) do { if ((n) > 0) omp_set_num_threads(n); } while (0)
#else
#define ORACLE_SET_THREADS(n) do { (void)(n); } while (0)
#endif

/* Whole output, NCHW fp64, of the general problem `desc` (see
 * oracle_make).  nthreads <= 0 keeps the OpenMP default.  Returns 0, or -1
 * on a bad argument.  Threads split the (b, h) rows; every pixel runs the
 * same body, so the result does not depend on the thread count. */
int oracle_dcn_forward_ex(const float *x, const float *offset, const float *mask,
                          const float *weight, const float *bias, double *out,
                          const int *desc, int nthreads)
{
    if (!desc) return -1;
    const oracle_problem p = oracle_make(x, offset, mask, weight, bias, desc);
    if (oracle_check(&p) || !out) return -1;
    const size_t plane_out = (size_t)p.Ho * p.Wo;
    ORACLE_SET_THREADS(nthreads);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < p.B * p.Ho; ++bh) {
        const int b = bh / p.Ho, h = bh % p.Ho;
        for (int w = 0; w < p.Wo; ++w) {
            oracle_pixel(&p, b, h, w,
                         out + (size_t)b * p.O * plane_out + (size_t)h * p.Wo + w,
                         (ptrdiff_t)plane_out);
        }
    }
    return 0;
}

/* Selected output pixels only: pts holds n triples (b, h, w); out receives
 * n rows of O channels (fp64, [n, O]).  Same body as the full version. */
int oracle_dcn_forward_points_ex(const float *x, const float *offset, const float *mask,
                                 const float *weight, const float *bias,
                                 const int *pts, int n, double *out,
                                 const int *desc, int nthreads)
{
    if (!desc) return -1;
    const oracle_problem p = oracle_make(x, offset, mask, weight, bias, desc);
    if (oracle_check(&p) || !out || (n > 0 && !pts) || n < 0) return -1;
    for (int t = 0; t < n; ++t) {
        const int b = pts[3 * t], h = pts[3 * t + 1], w = pts[3 * t + 2];
        if (b < 0 || b >= p.B || h < 0 || h >= p.Ho || w < 0 || w >= p.Wo) return -1;
    }
    ORACLE_SET_THREADS(nthreads);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int t = 0; t < n; ++t) {
        oracle_pixel(&p, pts[3 * t], pts[3 * t + 1], pts[3 * t + 2],
                     out + (size_t)t * p.O, 1);
    }
    return 0;
}

/* The page-1 problem: stride 1, dilation 1, one padding, one weight group
 * and one offset group. */
int oracle_dcn_forward(const float *x, const float *offset, const float *mask,
                       const float *weight, const float *bias, double *out,
                       int B, int C, int H, int W, int O, int kh, int kw, int pad,
                       int nthreads)
{
    const int d[15] = {B, C, H, W, O, kh, kw, 1, 1, pad, pad, 1, 1, 1, 1};
    return oracle_dcn_forward_ex(x, offset, mask, weight, bias, out, d, nthreads);
}

int oracle_dcn_forward_points(const float *x, const float *offset, const float *mask,
                              const float *weight, const float *bias,
                              const int *pts, int n, double *out,
                              int B, int C, int H, int W, int O, int kh, int kw, int pad,
                              int nthreads)
{
    const int d[15] = {B, C, H, W, O, kh, kw, 1, 1, pad, pad, 1, 1, 1, 1};
    return oracle_dcn_forward_points_ex(x, offset, mask, weight, bias, pts, n, out, d, nthreads);
}

/* Number of threads an OpenMP region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ backward
 *
 * The gradients of the forward above with respect to each of its inputs,
 * given the cotangent grad_out [B, O, Ho, Wo] of its output: the chain rule
 * applied to the forward's definition, term by term.  (The deformops page,
 * section "Deformable convolution", has the backward keep fp32 accumulation
 * and no TF32 so that rounding does not reach the offset gradients; the
 * definition itself follows from the forward.)  For image b, output pixel
 * (h, w), tap k = (i, j), offset group q and channel c of q, with m, py, px,
 * y0, x0, ly, lx, wy, wx and S as in the forward, and
 *
 *   gA = sum over the outputs o of c's weight group of
 *        grad_out[b,o,h,w] * weight[o, c - c0, i, j]     (column gradient)
 *
 * the contributions are
 *
 *   grad_bias[o]                 += grad_out[b,o,h,w]
 *   grad_weight[o, c-c0, i, j]   += grad_out[b,o,h,w] * m * S
 *   grad_mask[b, q*kk + k, h, w] += gA * S
 *   grad_x[b, c, y0+a, x0+e]     += gA * m * wy_a * wx_e     (inside corners)
 *   grad_offset[b, 2(q*kk+k), h, w]   += gA * m * dS/dpy
 *   grad_offset[b, 2(q*kk+k)+1, h, w] += gA * m * dS/dpx
 *
 * with kk = kh*kw, dS/dpy = sum over inside corners of (2a-1) * wx_e * x,
 * dS/dpx = sum over inside corners of (2e-1) * wy_a * x (d wy_1/d py = 1,
 * d wy_0/d py = -1, likewise for x).  The corner weights are piecewise
 * linear in the coordinate; at an integer coordinate the derivative is that
 * of the cell [y0, y0+1) which floor selects (the right-hand derivative).
 * A sample whose corners are all outside gives 0 to every gradient.
 *
 * All sums are fp64 in the fixed order b -> h -> w -> (i, j) -> q -> c ->
 * o / corner.  Images are independent except for grad_weight and
 * grad_bias, which are summed per image and then over images in order, so
 * the result does not depend on the thread count.
 *
 * Layouts (host memory): x, offset, mask, weight as in the forward;
 * grad_out [B, O, Ho, Wo] fp32; results fp64: grad_x [B, C, H, W],
 * grad_offset like offset, grad_mask like mask (NULL: not computed),
 * grad_weight like weight, grad_bias [O] (NULL: not computed).
 */
/* One output pixel (b, h, w) of the backward pass.  gw and gb receive its
 * weight and bias contributions (added), gx_b its scatter into image b's
 * grad_x (added); each may be NULL (not wanted).  goff and gmask point at
 * this pixel's first offset / mask gradient; consecutive channels of those
 * arrays are `stride` apart; gmask may be NULL. */
static void oracle_bwd_pixel(const oracle_problem *p, const float *grad_out, int b, int h, int w,
                             double *gw, double *gb, double *gx_b,
                             double *goff, double *gmask, ptrdiff_t stride)
{
    const int k_total = p->kh * p->kw;
    const int Cg = p->C / p->groups, Og = p->O / p->groups, Cq = p->C / p->ogroups;
    const size_t plane_in = (size_t)p->H * p->W;
    const size_t plane_out = (size_t)p->Ho * p->Wo;
    const size_t pix = (size_t)h * p->Wo + w;
    const float *go = grad_out + (size_t)b * p->O * plane_out + pix;
    if (gb)
        for (int o = 0; o < p->O; ++o) gb[o] += (double)go[o * plane_out];
    for (int i = 0; i < p->kh; ++i) {
        for (int j = 0; j < p->kw; ++j) {
            const int k = i * p->kw + j;
            for (int q = 0; q < p->ogroups; ++q) {
                const size_t oq = (size_t)b * p->ogroups + q;
                const float dy = p->offset[(oq * 2 * k_total + 2 * k) * plane_out + pix];
                const float dx = p->offset[(oq * 2 * k_total + 2 * k + 1) * plane_out + pix];
                const double m = p->mask
                    ? (double)p->mask[(oq * k_total + k) * plane_out + pix]
                    : 1.0;
                const float py = (float)(h * p->sh - p->ph + i * p->dh) + dy;
                const float px = (float)(w * p->sw - p->pw + j * p->dw) + dx;
                const float fy0 = floorf(py);
                const float fx0 = floorf(px);
                const double ly = (double)py - (double)fy0;
                const double lx = (double)px - (double)fx0;
                const double wy[2] = {1.0 - ly, ly};
                const double wx[2] = {1.0 - lx, lx};
                double g_dy = 0.0, g_dx = 0.0, g_m = 0.0;
                for (int c = q * Cq; c < (q + 1) * Cq; ++c) {
                    const int g = c / Cg;
                    const int cl = c - g * Cg;
                    const float *xc = p->x + ((size_t)b * p->C + c) * plane_in;
                    double s = 0.0, s_y = 0.0, s_x = 0.0;
                    for (int a = 0; a < 2; ++a) {
                        for (int e = 0; e < 2; ++e) {
                            const double yy = (double)fy0 + a;
                            const double xx = (double)fx0 + e;
                            if (yy >= 0.0 && yy <= p->H - 1 && xx >= 0.0 && xx <= p->W - 1) {
                                const double v = (double)xc[(size_t)yy * p->W + (size_t)xx];
                                s += wy[a] * wx[e] * v;
                                s_y += (a ? 1.0 : -1.0) * wx[e] * v;
                                s_x += (e ? 1.0 : -1.0) * wy[a] * v;
                            }
                        }
                    }
                    double ga = 0.0;
                    for (int o = g * Og; o < (g + 1) * Og; ++o) {
                        const double gov = (double)go[o * plane_out];
                        const size_t wi = (((size_t)o * Cg + cl) * p->kh + i) * p->kw + j;
                        ga += gov * (double)p->weight[wi];
                        if (gw) gw[wi] += gov * m * s;
                    }
                    g_m += ga * s;
                    g_dy += ga * m * s_y;
                    g_dx += ga * m * s_x;
                    if (gx_b) {
                        double *gxc = gx_b + (size_t)c * plane_in;
                        for (int a = 0; a < 2; ++a) {
                            for (int e = 0; e < 2; ++e) {
                                const double yy = (double)fy0 + a;
                                const double xx = (double)fx0 + e;
                                if (yy >= 0.0 && yy <= p->H - 1 && xx >= 0.0 && xx <= p->W - 1)
                                    gxc[(size_t)yy * p->W + (size_t)xx] += ga * m * wy[a] * wx[e];
                            }
                        }
                    }
                }
                goff[(ptrdiff_t)(q * 2 * k_total + 2 * k) * stride] = g_dy;
                goff[(ptrdiff_t)(q * 2 * k_total + 2 * k + 1) * stride] = g_dx;
                if (gmask) gmask[(ptrdiff_t)(q * k_total + k) * stride] = g_m;
            }
        }
    }
}

int oracle_dcn_backward_ex(const float *x, const float *offset, const float *mask,
                           const float *weight, const float *grad_out,
                           double *grad_x, double *grad_offset, double *grad_mask,
                           double *grad_weight, double *grad_bias,
                           const int *desc, int nthreads)
{
    if (!desc || !grad_out || !grad_x || !grad_offset || !grad_weight) return -1;
    const oracle_problem p = oracle_make(x, offset, mask, weight, NULL, desc);
    if (oracle_check(&p)) return -1;
    const int k_total = p.kh * p.kw;
    const int Cg = p.C / p.groups;
    const size_t plane_in = (size_t)p.H * p.W;
    const size_t plane_out = (size_t)p.Ho * p.Wo;
    const size_t n_w = (size_t)p.O * Cg * k_total;
    const size_t per_image = n_w + (size_t)p.O;
    double *part = (double *)calloc((size_t)p.B * per_image, sizeof(double));
    if (!part) return -2;
    memset(grad_x, 0, sizeof(double) * (size_t)p.B * p.C * plane_in);
    ORACLE_SET_THREADS(nthreads);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < p.B; ++b) {
        double *gw = part + (size_t)b * per_image;   /* this image's grad_weight */
        double *gb = gw + n_w;                        /* and grad_bias */
        double *gx_b = grad_x + (size_t)b * p.C * plane_in;
        double *goff_b = grad_offset + (size_t)b * 2 * p.ogroups * k_total * plane_out;
        double *gm_b = grad_mask ? grad_mask + (size_t)b * p.ogroups * k_total * plane_out : NULL;
        for (int h = 0; h < p.Ho; ++h) {
            for (int w = 0; w < p.Wo; ++w) {
                const size_t pix = (size_t)h * p.Wo + w;
                oracle_bwd_pixel(&p, grad_out, b, h, w, gw, gb, gx_b, goff_b + pix,
                                 gm_b ? gm_b + pix : NULL, (ptrdiff_t)plane_out);
            }
        }
    }
    for (size_t t = 0; t < n_w; ++t) {
        double acc = 0.0;
        for (int b = 0; b < p.B; ++b) acc += part[(size_t)b * per_image + t];
        grad_weight[t] = acc;
    }
    if (grad_bias) {
        for (int o = 0; o < p.O; ++o) {
            double acc = 0.0;
            for (int b = 0; b < p.B; ++b) acc += part[(size_t)b * per_image + n_w + o];
            grad_bias[o] = acc;
        }
    }
    free(part);
    return 0;
}

/* The offset and mask gradients of selected output pixels only (they
 * depend on that pixel alone): pts holds n triples (b, h, w); goff receives
 * n rows of 2*G*kh*kw values, gmask (may be NULL) n rows of G*kh*kw.  Same
 * body as the full version. */
int oracle_dcn_backward_points_ex(const float *x, const float *offset, const float *mask,
                                  const float *weight, const float *grad_out,
                                  const int *pts, int n, double *goff, double *gmask,
                                  const int *desc, int nthreads)
{
    if (!desc || !grad_out || !goff || n < 0 || (n > 0 && !pts)) return -1;
    const oracle_problem p = oracle_make(x, offset, mask, weight, NULL, desc);
    if (oracle_check(&p)) return -1;
    for (int t = 0; t < n; ++t) {
        const int b = pts[3 * t], h = pts[3 * t + 1], w = pts[3 * t + 2];
        if (b < 0 || b >= p.B || h < 0 || h >= p.Ho || w < 0 || w >= p.Wo) return -1;
    }
    const int k_total = p.kh * p.kw;
    ORACLE_SET_THREADS(nthreads);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int t = 0; t < n; ++t) {
        oracle_bwd_pixel(&p, grad_out, pts[3 * t], pts[3 * t + 1], pts[3 * t + 2], NULL, NULL, NULL,
                         goff + (size_t)t * 2 * p.ogroups * k_total,
                         gmask ? gmask + (size_t)t * p.ogroups * k_total : NULL, 1);
    }
    return 0;
}
