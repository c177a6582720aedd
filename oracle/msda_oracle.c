/*
 * Oracle for the forward pass of multi-scale deformable attention (MSDA).
 *
 * TEST INFRASTRUCTURE ONLY, like dcn_oracle.c: the plain, slow CPU
 * definition the CUDA kernel is checked against; the product library never
 * links or calls it, and it shares no code with the CUDA sources.
 *
 * What it computes (page "deformops 3.0.1", section "Multi-scale deformable
 * attention": the functional form msda(value, shapes, starts, locations,
 * weights, method)).  With B batch, G heads, D channels per head, Q
 * queries, L levels and K points per level:
 *
 *   value     [B, S, G, D]        S = sum over levels of H_l * W_l; level l
 *                                 occupies rows starts[l] .. + H_l*W_l,
 *                                 row-major (row y*W_l + x)
 *   locations [B, Q, G, L, K, 2]  normalized to [0, 1]
 *   weights   [B, Q, G, L*K]      used as given, or (softmax) normalized
 *                                 jointly over the L*K entries of (b, q, g)
 *   out       [B, Q, G, D]
 *
 *   out[b,q,g,d] = sum_{l,k} a[b,q,g,l,k] * S_l(b, g, d, py, px)
 *
 * where S_l is the bilinear sample of level l at pixel coordinates
 *   px = loc[..., 0] * W_l - 0.5,   py = loc[..., 1] * H_l - 0.5
 * (readings: the last axis holds (x, y), and a normalized coordinate maps
 * pixel centres to (i + 0.5) / size -- the convention of the Deformable
 * DETR operator that the page's layer implements; the page states neither),
 * from corners (y0 + a, x0 + e), y0 = floor(py), x0 = floor(px), with
 * weights (1-ly)(1-lx), (1-ly)lx, ly(1-lx), ly lx, and every corner outside
 * [0, H_l-1] x [0, W_l-1] contributing 0.
 *
 * Precision: px, py are formed in fp32 (the locations are fp32), so that
 * floor() is decided in the kernel's precision; corner weights, the
 * softmax and all sums are fp64, in the order l -> k -> corner.
 */
#include <math.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MSDA_MAX_LEVELS 16

/* shapes: L pairs (H_l, W_l); starts: L row offsets.  softmax != 0
 * normalizes the weights.  Returns 0, or -1 on a bad argument. */
int oracle_msda_forward(const float *value, const int *shapes, const int *starts, int L,
                        const float *locations, const float *weights, int softmax,
                        double *out, int B, int S, int G, int D, int Q, int K, int nthreads)
{
    if (!value || !shapes || !starts || !locations || !weights || !out) return -1;
    if (B <= 0 || S <= 0 || G <= 0 || D <= 0 || Q <= 0 || K <= 0) return -1;
    if (L <= 0 || L > MSDA_MAX_LEVELS || K > 64) return -1;
    for (int l = 0; l < L; ++l) {
        const int H = shapes[2 * l], W = shapes[2 * l + 1];
        if (H <= 0 || W <= 0 || starts[l] < 0 || (long long)starts[l] + (long long)H * W > S)
            return -1;
    }
    const int LK = L * K;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    #pragma omp parallel for schedule(dynamic, 4)
    for (int bq = 0; bq < B * Q; ++bq) {
        const int b = bq / Q;
        for (int g = 0; g < G; ++g) {
            const size_t row = (size_t)bq * G + g;              /* (b, q, g) */
            const float *wrow = weights + row * LK;
            double a[MSDA_MAX_LEVELS * 64];
            double wmax = -INFINITY, wsum = 0.0;
            for (int t = 0; t < LK; ++t) {
                a[t] = (double)wrow[t];
                if (a[t] > wmax) wmax = a[t];
            }
            if (softmax) {
                for (int t = 0; t < LK; ++t) { a[t] = exp(a[t] - wmax); wsum += a[t]; }
                for (int t = 0; t < LK; ++t) a[t] /= wsum;
            }
            double *o = out + row * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int l = 0; l < L; ++l) {
                const int H = shapes[2 * l], W = shapes[2 * l + 1];
                for (int k = 0; k < K; ++k) {
                    const float *loc = locations + ((row * L + l) * K + k) * 2;
                    const float px = loc[0] * (float)W - 0.5f;
                    const float py = loc[1] * (float)H - 0.5f;
                    const float fx0 = floorf(px), fy0 = floorf(py);
                    const double lx = (double)px - (double)fx0;
                    const double ly = (double)py - (double)fy0;
                    const double wy[2] = {1.0 - ly, ly};
                    const double wx[2] = {1.0 - lx, lx};
                    const double aw = a[l * K + k];
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const int ay = e2 >> 1, ex = e2 & 1;
                        const double yy = (double)fy0 + ay, xx = (double)fx0 + ex;
                        if (!(yy >= 0.0 && yy <= H - 1 && xx >= 0.0 && xx <= W - 1)) continue;
                        const size_t s = (size_t)starts[l] + (size_t)yy * W + (size_t)xx;
                        const float *v = value + (((size_t)b * S + s) * G + g) * D;
                        const double cw = aw * wy[ay] * wx[ex];
                        for (int d = 0; d < D; ++d) o[d] += cw * (double)v[d];
                    }
                }
            }
        }
    }
    return 0;
}

/*
 * Backward of oracle_msda_forward: the chain rule applied to the definition
 * above, term by term.  The page's multi-scale attention backward writes
 * the value gradient by accumulation (section "DeformOps", "Zero-buffer
 * kernels"), and its float32 accumulator (section "Backend selection") is
 * the exact reading taken here: every gradient is returned in fp64 from
 * fp64 sums.  With go = grad_out[b,q,g,:], per (b, q, g) and point t=(l,k):
 *
 *   S_t[d]          = sum_c wy[c] wx[c] v_c[d]       (inside corners c only)
 *   dS_t/dpx [d]    = sum_c wy[c] sx[c] v_c[d],  sx = -1 (left), +1 (right)
 *   dS_t/dpy [d]    = sum_c sy[c] wx[c] v_c[d],  sy = -1 (top),  +1 (bottom)
 *   grad_a[t]       = <go, S_t>
 *   grad_value[c]  += a[t] wy[c] wx[c] go           (inside corners only)
 *   grad_loc[t]     = a[t] (<go, dS_t/dpx> W_l, <go, dS_t/dpy> H_l)
 *   grad_weights[t] = grad_a[t], or with softmax
 *                     a[t] (grad_a[t] - sum_s a[s] grad_a[s])
 *
 * Readings: px and py are formed in fp32 exactly as in the forward, and at
 * an integer coordinate the derivative is that of the cell floor() picks
 * (the right-hand one); a point whose corners are all outside has zero
 * gradient; the location gradient is with respect to the normalized
 * location (the factors W_l and H_l of px and py).
 *
 * grad_value [B,S,G,D], grad_locations [B,Q,G,L,K,2], grad_weights
 * [B,Q,G,L*K] are overwritten.  Parallel over (b, g) pairs: the value
 * gradient of one (b, g) receives only that pair's queries.
 */
int oracle_msda_backward(const float *value, const int *shapes, const int *starts, int L,
                         const float *locations, const float *weights, int softmax,
                         const float *grad_out, double *grad_value, double *grad_locations,
                         double *grad_weights, int B, int S, int G, int D, int Q, int K,
                         int nthreads)
{
    if (!value || !shapes || !starts || !locations || !weights || !grad_out) return -1;
    if (!grad_value || !grad_locations || !grad_weights) return -1;
    if (B <= 0 || S <= 0 || G <= 0 || D <= 0 || Q <= 0 || K <= 0) return -1;
    if (L <= 0 || L > MSDA_MAX_LEVELS || K > 64) return -1;
    for (int l = 0; l < L; ++l) {
        const int H = shapes[2 * l], W = shapes[2 * l + 1];
        if (H <= 0 || W <= 0 || starts[l] < 0 || (long long)starts[l] + (long long)H * W > S)
            return -1;
    }
    const int LK = L * K;
    for (size_t i = 0; i < (size_t)B * S * G * D; ++i) grad_value[i] = 0.0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    #pragma omp parallel for schedule(dynamic, 1)
    for (int bg = 0; bg < B * G; ++bg) {
        const int b = bg / G, g = bg % G;
        for (int q = 0; q < Q; ++q) {
            const size_t row = ((size_t)b * Q + q) * G + g;     /* (b, q, g) */
            const float *wrow = weights + row * LK;
            const float *go = grad_out + row * D;
            double a[MSDA_MAX_LEVELS * 64], ga[MSDA_MAX_LEVELS * 64];
            double wmax = -INFINITY, wsum = 0.0;
            for (int t = 0; t < LK; ++t) {
                a[t] = (double)wrow[t];
                if (a[t] > wmax) wmax = a[t];
            }
            if (softmax) {
                for (int t = 0; t < LK; ++t) { a[t] = exp(a[t] - wmax); wsum += a[t]; }
                for (int t = 0; t < LK; ++t) a[t] /= wsum;
            }
            for (int l = 0; l < L; ++l) {
                const int H = shapes[2 * l], W = shapes[2 * l + 1];
                for (int k = 0; k < K; ++k) {
                    const int t = l * K + k;
                    const float *loc = locations + ((row * L + l) * K + k) * 2;
                    const float px = loc[0] * (float)W - 0.5f;
                    const float py = loc[1] * (float)H - 0.5f;
                    const float fx0 = floorf(px), fy0 = floorf(py);
                    const double lx = (double)px - (double)fx0;
                    const double ly = (double)py - (double)fy0;
                    const double wy[2] = {1.0 - ly, ly};
                    const double wx[2] = {1.0 - lx, lx};
                    const double sgn[2] = {-1.0, 1.0};       /* d w[0]/dp, d w[1]/dp */
                    double g_a = 0.0, g_px = 0.0, g_py = 0.0;
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const int ay = e2 >> 1, ex = e2 & 1;
                        const double yy = (double)fy0 + ay, xx = (double)fx0 + ex;
                        if (!(yy >= 0.0 && yy <= H - 1 && xx >= 0.0 && xx <= W - 1)) continue;
                        const size_t s = (size_t)starts[l] + (size_t)yy * W + (size_t)xx;
                        const float *v = value + (((size_t)b * S + s) * G + g) * D;
                        double *gv = grad_value + (((size_t)b * S + s) * G + g) * D;
                        double dot = 0.0;                      /* <go, v_c> */
                        for (int d = 0; d < D; ++d) dot += (double)go[d] * (double)v[d];
                        g_a += wy[ay] * wx[ex] * dot;
                        g_px += wy[ay] * sgn[ex] * dot;
                        g_py += sgn[ay] * wx[ex] * dot;
                        const double cw = a[t] * wy[ay] * wx[ex];
                        for (int d = 0; d < D; ++d) gv[d] += cw * (double)go[d];
                    }
                    ga[t] = g_a;
                    double *gl = grad_locations + ((row * L + l) * K + k) * 2;
                    gl[0] = a[t] * g_px * (double)W;
                    gl[1] = a[t] * g_py * (double)H;
                }
            }
            double *gw = grad_weights + row * LK;
            if (softmax) {
                double s_ag = 0.0;
                for (int t = 0; t < LK; ++t) s_ag += a[t] * ga[t];
                for (int t = 0; t < LK; ++t) gw[t] = a[t] * (ga[t] - s_ag);
            } else {
                for (int t = 0; t < LK; ++t) gw[t] = ga[t];
            }
        }
    }
    return 0;
}
