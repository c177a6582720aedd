/*
 * Oracle for single-scale deformable sampling (the DCNv3 operator).
 *
 * TEST INFRASTRUCTURE ONLY, like dcn_oracle.c: the plain, slow CPU
 * definition the CUDA kernel is checked against; the product library never
 * links or calls it, and it shares no code with the CUDA sources.
 *
 * What it computes (page "deformops 3.0.1", section "Single-scale
 * deformable sampling": the operator of the layers DeformAttn2d and
 * DeformSample2d, functional form attn, which samples and aggregates
 * without the spatial weight of deformable convolution; the references
 * section names it the DCNv3 operator of InternImage).  With B batch, G
 * groups of D channels (C = G*D), a kh x kw tap grid (K = kh*kw taps),
 * stride (sh, sw), padding (ph, pw), dilation (dh, dw):
 *
 *   value    [B, H, W, G, D]          channels-last
 *   offsets  [B, Ho, Wo, G, K, 2]     (dy, dx) in pixels, tap k = i*kw + j
 *   weights  [B, Ho, Wo, G, K]        used as given, or (softmax) normalized
 *                                     over the K taps of (b, ho, wo, g)
 *   out      [B, Ho, Wo, G, D]
 *
 *   out[b,ho,wo,g,d] = sum_k a[b,ho,wo,g,k] * S(value[b,:,:,g,d], py, px)
 *   py = ho*sh - ph + i*dh + dy,   px = wo*sw - pw + j*dw + dx
 *
 * S the bilinear sample from corners (y0 + a, x0 + e), y0 = floor(py),
 * x0 = floor(px), weights (1-ly)(1-lx), (1-ly)lx, ly(1-lx), ly lx, every
 * corner outside [0, H-1] x [0, W-1] contributing 0, and
 * Ho = (H + 2ph - dh(kh-1) - 1)/sh + 1 (likewise Wo).
 *
 * Readings (the page fixes none of these): the sampling positions are the
 * deformable convolution's own (its tap grid, stride, padding, dilation
 * and (dy, dx) pixel offsets, as torchvision's deform_conv2d defines them),
 * one offset pair and one aggregation weight per (group, tap), every
 * tensor channels-last.  So the operator equals a depthwise deformable
 * convolution with unit weights, G offset groups and the aggregation
 * weights as its mask.
 *
 * Precision: py and px are formed in fp32 (as in the forward of the
 * convolution: the integer base converted, then the offset added), so that
 * floor() is decided in the kernel's precision; the softmax, corner weights
 * and sums are fp64, in the order k -> corner.
 */
#include <math.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ATTN_MAX_TAPS 1024

/* Returns 0, or -1 on a bad argument. */
int oracle_attn_forward(const float *value, const float *offsets, const float *weights,
                        int softmax, double *out, int B, int H, int W, int G, int D, int kh,
                        int kw, int sh, int sw, int ph, int pw, int dh, int dw, int nthreads)
{
    if (!value || !offsets || !weights || !out) return -1;
    if (B <= 0 || H <= 0 || W <= 0 || G <= 0 || D <= 0 || kh <= 0 || kw <= 0) return -1;
    if (sh <= 0 || sw <= 0 || ph < 0 || pw < 0 || dh <= 0 || dw <= 0) return -1;
    const int K = kh * kw;
    if (K > ATTN_MAX_TAPS) return -1;
    const int span_h = H + 2 * ph - dh * (kh - 1) - 1;
    const int span_w = W + 2 * pw - dw * (kw - 1) - 1;
    if (span_h < 0 || span_w < 0) return -1;
    const int Ho = span_h / sh + 1, Wo = span_w / sw + 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    #pragma omp parallel for schedule(dynamic, 4)
    for (int bhw = 0; bhw < B * Ho * Wo; ++bhw) {
        const int b = bhw / (Ho * Wo);
        const int ho = (bhw / Wo) % Ho;
        const int wo = bhw % Wo;
        for (int g = 0; g < G; ++g) {
            const size_t row = (size_t)bhw * G + g;            /* (b, ho, wo, g) */
            const float *wrow = weights + row * K;
            const float *orow = offsets + row * K * 2;
            double a[ATTN_MAX_TAPS];
            double wmax = -INFINITY, wsum = 0.0;
            for (int k = 0; k < K; ++k) {
                a[k] = (double)wrow[k];
                if (a[k] > wmax) wmax = a[k];
            }
            if (softmax) {
                for (int k = 0; k < K; ++k) { a[k] = exp(a[k] - wmax); wsum += a[k]; }
                for (int k = 0; k < K; ++k) a[k] /= wsum;
            }
            double *o = out + row * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int k = 0; k < K; ++k) {
                const int i = k / kw, j = k % kw;
                const float py = (float)(ho * sh - ph + i * dh) + orow[2 * k];
                const float px = (float)(wo * sw - pw + j * dw) + orow[2 * k + 1];
                const float fy0 = floorf(py), fx0 = floorf(px);
                const double ly = (double)py - (double)fy0;
                const double lx = (double)px - (double)fx0;
                const double wy[2] = {1.0 - ly, ly};
                const double wx[2] = {1.0 - lx, lx};
                for (int e2 = 0; e2 < 4; ++e2) {
                    const int ay = e2 >> 1, ex = e2 & 1;
                    const double yy = (double)fy0 + ay, xx = (double)fx0 + ex;
                    if (!(yy >= 0.0 && yy <= H - 1 && xx >= 0.0 && xx <= W - 1)) continue;
                    const float *v = value + ((((size_t)b * H + (size_t)yy) * W + (size_t)xx) * G + g) * D;
                    const double cw = a[k] * wy[ay] * wx[ex];
                    for (int d = 0; d < D; ++d) o[d] += cw * (double)v[d];
                }
            }
        }
    }
    return 0;
}

/*
 * Backward of oracle_attn_forward: the chain rule applied to the definition
 * above, term by term, every gradient in fp64 (the float32-accumulator
 * reading of the page's section "Backend selection", which gives
 * single-scale sampling the same gradient rule as multi-scale attention).
 * With go = grad_out[b,ho,wo,g,:], per tap k and inside corner c of its
 * sample, bilinear weights wy, wx:
 *
 *   grad_a[k]        = sum_c wy wx <go, v_c>
 *   grad_value[c]   += a[k] wy wx go
 *   grad_offsets[k]  = a[k] (sum_c sy wx <go, v_c>,  sum_c wy sx <go, v_c>)   (dy, dx)
 *   grad_weights[k]  = grad_a[k], or with softmax a[k] (grad_a[k] - sum_s a[s] grad_a[s])
 *
 * sx, sy = -1 for the left/top corner and +1 for the right/bottom one: at
 * an integer coordinate the derivative of the cell floor() picks; a tap
 * whose corners are all outside has zero gradients.  grad_value
 * [B,H,W,G,D], grad_offsets [B,Ho,Wo,G,K,2], grad_weights [B,Ho,Wo,G,K] are
 * overwritten.  Parallel over (b, g) pairs: the value gradient of one
 * (b, g) receives only that pair's output pixels.
 */
int oracle_attn_backward(const float *value, const float *offsets, const float *weights,
                         int softmax, const float *grad_out, double *grad_value,
                         double *grad_offsets, double *grad_weights, int B, int H, int W, int G,
                         int D, int kh, int kw, int sh, int sw, int ph, int pw, int dh, int dw,
                         int nthreads)
{
    if (!value || !offsets || !weights || !grad_out) return -1;
    if (!grad_value || !grad_offsets || !grad_weights) return -1;
    if (B <= 0 || H <= 0 || W <= 0 || G <= 0 || D <= 0 || kh <= 0 || kw <= 0) return -1;
    if (sh <= 0 || sw <= 0 || ph < 0 || pw < 0 || dh <= 0 || dw <= 0) return -1;
    const int K = kh * kw;
    if (K > ATTN_MAX_TAPS) return -1;
    const int span_h = H + 2 * ph - dh * (kh - 1) - 1;
    const int span_w = W + 2 * pw - dw * (kw - 1) - 1;
    if (span_h < 0 || span_w < 0) return -1;
    const int Ho = span_h / sh + 1, Wo = span_w / sw + 1;
    for (size_t n = 0; n < (size_t)B * H * W * G * D; ++n) grad_value[n] = 0.0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    #pragma omp parallel for schedule(dynamic, 1)
    for (int bg = 0; bg < B * G; ++bg) {
        const int b = bg / G, g = bg % G;
        for (int hw = 0; hw < Ho * Wo; ++hw) {
            const int ho = hw / Wo, wo = hw % Wo;
            const size_t row = ((size_t)b * Ho * Wo + hw) * G + g;   /* (b, ho, wo, g) */
            const float *wrow = weights + row * K;
            const float *orow = offsets + row * K * 2;
            const float *go = grad_out + row * D;
            double a[ATTN_MAX_TAPS], ga[ATTN_MAX_TAPS];
            double wmax = -INFINITY, wsum = 0.0;
            for (int k = 0; k < K; ++k) {
                a[k] = (double)wrow[k];
                if (a[k] > wmax) wmax = a[k];
            }
            if (softmax) {
                for (int k = 0; k < K; ++k) { a[k] = exp(a[k] - wmax); wsum += a[k]; }
                for (int k = 0; k < K; ++k) a[k] /= wsum;
            }
            for (int k = 0; k < K; ++k) {
                const int i = k / kw, j = k % kw;
                const float py = (float)(ho * sh - ph + i * dh) + orow[2 * k];
                const float px = (float)(wo * sw - pw + j * dw) + orow[2 * k + 1];
                const float fy0 = floorf(py), fx0 = floorf(px);
                const double ly = (double)py - (double)fy0;
                const double lx = (double)px - (double)fx0;
                const double rw[2] = {1.0 - ly, ly};                 /* row weights */
                const double cwx[2] = {1.0 - lx, lx};                /* column weights */
                const double dsgn[2] = {-1.0, 1.0};                  /* their derivatives */
                double g_a = 0.0, g_y = 0.0, g_x = 0.0;
                for (int e2 = 0; e2 < 4; ++e2) {
                    const int ay = e2 >> 1, ex = e2 & 1;
                    const double yy = (double)fy0 + ay, xx = (double)fx0 + ex;
                    if (!(yy >= 0.0 && yy <= H - 1 && xx >= 0.0 && xx <= W - 1)) continue;
                    const size_t at = (((size_t)b * H + (size_t)yy) * W + (size_t)xx) * G + g;
                    const float *v = value + at * D;
                    double *gv = grad_value + at * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += (double)go[d] * (double)v[d];
                    g_a += rw[ay] * cwx[ex] * dot;
                    g_y += dsgn[ay] * cwx[ex] * dot;
                    g_x += rw[ay] * dsgn[ex] * dot;
                    const double s = a[k] * rw[ay] * cwx[ex];
                    for (int d = 0; d < D; ++d) gv[d] += s * (double)go[d];
                }
                ga[k] = g_a;
                double *gofs = grad_offsets + (row * K + k) * 2;
                gofs[0] = a[k] * g_y;
                gofs[1] = a[k] * g_x;
            }
            double *gw = grad_weights + row * K;
            if (softmax) {
                double s_ag = 0.0;
                for (int k = 0; k < K; ++k) s_ag += a[k] * ga[k];
                for (int k = 0; k < K; ++k) gw[k] = a[k] * (ga[k] - s_ag);
            } else {
                for (int k = 0; k < K; ++k) gw[k] = ga[k];
            }
        }
    }
    return 0;
}
