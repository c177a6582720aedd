/*
 * Oracle for the forward pass of modulated deformable convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never links, calls or includes it, and it shares no code
 * with the CUDA sources.
 *
 * What it computes (page "litert-community/Idol ... deform_conv.py", module
 * docstring and the four-corner loop of deform_conv2d_gather; page "deformops
 * 3.0.1", section "Deformable convolution"): torchvision deform_conv2d with
 * stride 1, dilation 1, one offset group and one weight group.  For image b,
 * output channel o and output pixel (h, w):
 *
 *   out[b,o,h,w] = bias[o] + sum_{i<kh} sum_{j<kw} sum_{c<C}
 *                  weight[o,c,i,j] * m * S(b, c, py, px)
 *
 *   k  = i*kw + j                           (row-major taps)
 *   dy = offset[b, 2k,   h, w]              (vertical shift first)
 *   dx = offset[b, 2k+1, h, w]
 *   m  = mask[b, k, h, w]                   (1 when no mask is given)
 *   py = (h - pad + i) + dy,  px = (w - pad + j) + dx
 *   S  = sum over the four corners (y0+a, x0+e), a,e in {0,1}, with
 *        y0 = floor(py), x0 = floor(px), ly = py - y0, lx = px - x0,
 *        of wy_a * wx_e * x[b, c, y0+a, x0+e], where wy_0 = 1-ly, wy_1 = ly,
 *        wx_0 = 1-lx, wx_1 = lx, and a corner outside [0,H-1]x[0,W-1]
 *        contributes nothing.
 *
 * Precision: the sampling coordinate py/px is formed in fp32, the dtype in
 * which the page builds its sampling grid (the offsets are fp32), so that
 * the integer floor(py) is decided in the same precision as on the GPU.
 * Everything after that (corner weights, products, all sums) is fp64, in
 * the fixed order o -> (i, j) -> c -> corner (0,0), (0,1), (1,0), (1,1).
 * Non-finite or huge coordinates make every corner invalid (the comparisons
 * are done in double), so they contribute 0 and never index memory.
 *
 * Layouts (all dense, row-major, host memory):
 *   x      [B, C, H, W]        fp32 (bf16 inputs are passed as their exact
 *                              fp32 values)
 *   offset [B, 2*kh*kw, Ho, Wo] fp32
 *   mask   [B, kh*kw, Ho, Wo]  fp32, or NULL
 *   weight [O, C, kh, kw]      fp32
 *   bias   [O]                 fp32, or NULL
 *   out    [B, O, Ho, Wo]      fp64
 *   Ho = H + 2*pad - kh + 1,  Wo = W + 2*pad - kw + 1
 *
 * Parity of every part of this definition is pinned by the CPU tests:
 * zero offsets against a library direct convolution, integer offsets
 * against a shifted convolution, fractional offsets against hand-derived
 * bilinear values and against a library bilinear resampler, out-of-image
 * samples against the bias, and the mask against linearity.
 */
#include <math.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    const float *x, *offset, *mask, *weight, *bias;
    int B, C, H, W, O, kh, kw, pad, Ho, Wo;
} oracle_problem;

/* All O output channels of output pixel (b, h, w). */
static void oracle_pixel(const oracle_problem *p, int b, int h, int w,
                         double *out, ptrdiff_t out_stride)
{
    const int k_total = p->kh * p->kw;
    const size_t plane_out = (size_t)p->Ho * p->Wo;
    const size_t pix = (size_t)h * p->Wo + w;

    for (int o = 0; o < p->O; ++o) {
        double acc = 0.0;
        for (int i = 0; i < p->kh; ++i) {
            for (int j = 0; j < p->kw; ++j) {
                const int k = i * p->kw + j;
                const float dy = p->offset[((size_t)b * 2 * k_total + 2 * k) * plane_out + pix];
                const float dx = p->offset[((size_t)b * 2 * k_total + 2 * k + 1) * plane_out + pix];
                const double m = p->mask
                    ? (double)p->mask[((size_t)b * k_total + k) * plane_out + pix]
                    : 1.0;
                /* fp32 sampling coordinate, as in the page's grid */
                const float py = (float)(h - p->pad + i) + dy;
                const float px = (float)(w - p->pad + j) + dx;
                const float fy0 = floorf(py);
                const float fx0 = floorf(px);
                const double ly = (double)py - (double)fy0;
                const double lx = (double)px - (double)fx0;
                const double wy[2] = {1.0 - ly, ly};
                const double wx[2] = {1.0 - lx, lx};

                for (int c = 0; c < p->C; ++c) {
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
                    const double wt = p->weight[(((size_t)o * p->C + c) * p->kh + i) * p->kw + j];
                    acc += wt * m * s;
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
    if (p->kh <= 0 || p->kw <= 0 || p->pad < 0) return -1;
    if (p->Ho <= 0 || p->Wo <= 0) return -1;
    return 0;
}

#ifdef _OPENMP
#define ORACLE_SET_THREADS(n) do { if ((n) > 0) omp_set_num_threads(n); } while (0)
#else
#define ORACLE_SET_THREADS(n) do { (void)(n); } while (0)
#endif

/* Whole output, NCHW fp64.  nthreads <= 0 keeps the OpenMP default.
 * Returns 0, or -1 on a bad argument.  Threads split the (b, h) rows;
 * every pixel runs the same body, so the result does not depend on the
 * thread count. */
int oracle_dcn_forward(const float *x, const float *offset, const float *mask,
                       const float *weight, const float *bias, double *out,
                       int B, int C, int H, int W, int O, int kh, int kw, int pad,
                       int nthreads)
{
    oracle_problem p = {x, offset, mask, weight, bias, B, C, H, W, O, kh, kw, pad,
                        H + 2 * pad - kh + 1, W + 2 * pad - kw + 1};
    if (oracle_check(&p) || !out) return -1;
    const size_t plane_out = (size_t)p.Ho * p.Wo;
    ORACLE_SET_THREADS(nthreads);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * p.Ho; ++bh) {
        const int b = bh / p.Ho, h = bh % p.Ho;
        for (int w = 0; w < p.Wo; ++w) {
            oracle_pixel(&p, b, h, w,
                         out + (size_t)b * O * plane_out + (size_t)h * p.Wo + w,
                         (ptrdiff_t)plane_out);
        }
    }
    return 0;
}

/* Selected output pixels only: pts holds n triples (b, h, w); out receives
 * n rows of O channels (fp64, [n, O]).  Same body as the full version. */
int oracle_dcn_forward_points(const float *x, const float *offset, const float *mask,
                              const float *weight, const float *bias,
                              const int *pts, int n, double *out,
                              int B, int C, int H, int W, int O, int kh, int kw, int pad,
                              int nthreads)
{
    oracle_problem p = {x, offset, mask, weight, bias, B, C, H, W, O, kh, kw, pad,
                        H + 2 * pad - kh + 1, W + 2 * pad - kw + 1};
    if (oracle_check(&p) || !out || (n > 0 && !pts) || n < 0) return -1;
    for (int t = 0; t < n; ++t) {
        const int b = pts[3 * t], h = pts[3 * t + 1], w = pts[3 * t + 2];
        if (b < 0 || b >= B || h < 0 || h >= p.Ho || w < 0 || w >= p.Wo) return -1;
    }
    ORACLE_SET_THREADS(nthreads);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int t = 0; t < n; ++t) {
        oracle_pixel(&p, pts[3 * t], pts[3 * t + 1], pts[3 * t + 2],
                     out + (size_t)t * O, 1);
    }
    return 0;
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
