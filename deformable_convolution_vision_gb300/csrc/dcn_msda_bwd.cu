// Multi-scale deformable attention (MSDA), backward, on CUDA cores.
//
// The gradients of the forward in dcn_msda.cu (page "deformops 3.0.1",
// section "Multi-scale deformable attention") for a cotangent go =
// grad_out[b,q,g,:], the chain rule term by term.  Per (b, q, g) and point
// t = (l, k), with the bilinear weights wy, wx of the forward and only the
// corners c inside level l:
//
//   grad_a[t]        = sum_c wy wx <go, v_c>
//   grad_value[c]   += a[t] wy wx go                  (fp32 reductions)
//   grad_loc[t]      = a[t] (W_l sum_c wy sx <go, v_c>,  H_l sum_c sy wx <go, v_c>)
//   grad_weights[t]  = grad_a[t], or with softmax a[t] (grad_a[t] - sum_s a[s] grad_a[s])
//
// sx, sy = -1 for the left/top corner, +1 for the right/bottom one (the
// derivative of the cell picked by floor(), i.e. the right-hand one at an
// integer coordinate).  The page's backward writes the value gradient with
// no intermediate sampling buffer (section "DeformOps", "Zero-buffer
// kernels"); so does this one, with fp32 reductions straight into
// grad_value -- the page's float32-accumulator mode (section "Backend
// selection"), which is exact where native half-precision atomics would
// round every partial sum.
//
// Layout of the work: a group of GRP lanes per (b, q, g); lane r takes the
// CH-channel chunks r, r + GRP, ... of the head (CH = 8 for 16-bit values,
// 4 for fp32, one 16-byte load per corner; or 1).  When the chunks and the
// lanes are as many (every head width the page's CUDA backend takes, with
// GRP <= 32), the cotangent stays in registers for all points, and with
// CH = 8 a lane reduces the channels 4r .. 4r+3 and 4(r+GRP) .. +3 instead
// of its own eight, so that the group's 16-byte reductions are contiguous:
// two lanes fill each 32-byte sector and L2 receives half as many
// reduction requests.  Every lane computes each point's corners and
// weights itself (the same addresses and arithmetic in the whole group),
// loads its chunks of the four corner rows and of go,
// accumulates its partial dot products, and reduces the three per-point
// sums across the group with shuffles.  The lane t % GRP writes point t's
// location gradient and its raw grad_a into grad_weights; with softmax the
// same lane later reads that entry back and replaces it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "dcn_rowload.cuh"
#include "dcn_sampling_ops.h"

namespace dcn {

namespace {


// grad_value[p .. p + CH) += s * g[0 .. CH): fp32 reductions (16 bytes each
// for CH a multiple of 4; p is then 16-byte aligned)
template <int CH>
__device__ __forceinline__ void red_scaled(float *p, float s, const float (&g)[CH]) {
    if constexpr (CH % 4 == 0) {
#pragma unroll
        for (int e = 0; e < CH; e += 4)
            asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                         :: "l"(p + e), "f"(s * g[e]), "f"(s * g[e + 1]), "f"(s * g[e + 2]),
                            "f"(s * g[e + 3]) : "memory");
    } else {
#pragma unroll
        for (int e = 0; e < CH; ++e) atomicAdd(p + e, s * g[e]);
    }
}

template <int GRP>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int m = GRP / 2; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}


// Three resident blocks per SM (at most 85 registers a thread): measured
// against one (128 registers) and four (64), it is the fastest at 5440
// queries (109 against 117 and 130 us) and within 4% of the best at 21760.
template <typename T, int CH, int GRP, bool kOneChunk>
__global__ void __launch_bounds__(256, 3)
msda_backward_kernel(MsdaBwdParams p) {
    static_assert((GRP & (GRP - 1)) == 0 && GRP <= 32, "row group");
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rows = static_cast<long long>(p.B) * p.Q * p.G;
    // lanes past the last row work on the last row (for the shuffles) and
    // write nothing
    const bool live = t < rows * GRP;
    const long long row = live ? t / GRP : rows - 1;     // (b, q, g)
    const int r = static_cast<int>(t % GRP);             // lane within the row group
    const int g = static_cast<int>(row % p.G);
    const int b = static_cast<int>(row / (static_cast<long long>(p.Q) * p.G));
    const int LK = p.L * p.K;
    const int nch = p.D / CH;                            // chunks of the head
    const float *__restrict__ wrow = p.weights + row * LK;
    const float *__restrict__ lrow = p.locations + row * LK * 2;
    const T *__restrict__ value = static_cast<const T *>(p.value);
    const T *__restrict__ go_row = static_cast<const T *>(p.grad_out) + row * p.D;
    float *__restrict__ gl_row = p.grad_locations + row * LK * 2;
    float *__restrict__ gw_row = p.grad_weights + row * LK;
    const int GD = p.G * p.D;

    // the forward's attention weights (fp32 softmax, largest logit first)
    float wmax = -INFINITY, wsum = 1.0f;
    if (p.softmax) {
        for (int i = r; i < LK; i += GRP) wmax = fmaxf(wmax, __ldg(wrow + i));
#pragma unroll
        for (int m = GRP / 2; m >= 1; m >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, m));
        wsum = 0.0f;
        for (int i = r; i < LK; i += GRP) wsum += expf(__ldg(wrow + i) - wmax);
        wsum = group_sum<GRP>(wsum);
    }
    const float inv = 1.0f / wsum;

    DCN_BAD_DECL;
    float s_ag = 0.0f;   // sum over points of a[t] * grad_a[t] (the same in every lane)
    // one chunk per lane: its cotangent once, in the load order (go_d, for
    // the dot products) and in the reduction order (go_r, see above)
    constexpr bool kSplit = kOneChunk && CH == 8;
    float go_d[CH], go_r[CH];
    if constexpr (kOneChunk) {
        row_load<T, CH>(go_row + r * CH, go_d);
        if constexpr (kSplit) {
            row_load4<T>(go_row + 4 * r, go_r);
            row_load4<T>(go_row + 4 * (r + GRP), go_r + 4);
        }
    }
    for (int l = 0; l < p.L; ++l) {
        const int H = p.H[l], W = p.W[l];
        const T *vlevel = value + (static_cast<size_t>(b) * p.S + p.start[l]) * GD + g * p.D;
        float *glevel = p.grad_value + (static_cast<size_t>(b) * p.S + p.start[l]) * GD + g * p.D;
        for (int k = 0; k < p.K; ++k) {
            const int i = l * p.K + k;
            const float lw = __ldg(wrow + i);
            const float a = p.softmax ? expf(lw - wmax) * inv : lw;
            const float2 loc = __ldg(reinterpret_cast<const float2 *>(lrow) + i);
            // the forward's pixel coordinates, cell and weights
            float px = __fsub_rn(__fmul_rn(loc.x, static_cast<float>(W)), 0.5f);
            float py = __fsub_rn(__fmul_rn(loc.y, static_cast<float>(H)), 0.5f);
            px = fminf(fmaxf(px, -2.0f), static_cast<float>(W + 1));
            py = fminf(fmaxf(py, -2.0f), static_cast<float>(H + 1));
            const float fx = floorf(px), fy = floorf(py);
            const float lx = px - fx, ly = py - fy;
            const int x0 = static_cast<int>(fx), y0 = static_cast<int>(fy);
            const float wy[2] = {1.0f - ly, ly};
            const float wx[2] = {1.0f - lx, lx};
            float ga = 0.0f, gpx = 0.0f, gpy = 0.0f;     // this lane's partial sums
            for (int c0 = r; c0 < nch; c0 += GRP) {
                float go[CH];
                if constexpr (kOneChunk) {
#pragma unroll
                    for (int e = 0; e < CH; ++e) go[e] = go_d[e];
                } else {
                    row_load<T, CH>(go_row + c0 * CH, go);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int ay = c >> 1, ex = c & 1;
                    const int yy = y0 + ay, xx = x0 + ex;
                    if (static_cast<unsigned>(yy) >= static_cast<unsigned>(H) ||
                        static_cast<unsigned>(xx) >= static_cast<unsigned>(W))
                        continue;
                    const size_t pix = static_cast<size_t>(yy * W + xx) * GD;
                    const size_t off = pix + c0 * CH;
                    float v[CH];
                    row_load<T, CH>(DCN_ROW(vlevel + off, CH), v);
                    float dot = 0.0f;
#pragma unroll
                    for (int e = 0; e < CH; ++e) dot = fmaf(go[e], v[e], dot);
                    const float cw = wy[ay] * wx[ex];
                    ga = fmaf(cw, dot, ga);
                    gpx = fmaf(ex ? wy[ay] : -wy[ay], dot, gpx);
                    gpy = fmaf(ay ? wx[ex] : -wx[ex], dot, gpy);
                    if (live) {
                        if constexpr (kSplit) {
                            const float sc = a * cw;
                            float lo[4] = {go_r[0], go_r[1], go_r[2], go_r[3]};
                            float hi[4] = {go_r[4], go_r[5], go_r[6], go_r[7]};
                            if (DCN_GROW_OK(glevel + pix + 4 * r, 4)) red_scaled<4>(glevel + pix + 4 * r, sc, lo);
                            if (DCN_GROW_OK(glevel + pix + 4 * (r + GRP), 4))
                                red_scaled<4>(glevel + pix + 4 * (r + GRP), sc, hi);
                        } else {
                            if (DCN_GROW_OK(glevel + off, CH)) red_scaled<CH>(glevel + off, a * cw, go);
                        }
                    }
                }
            }
            ga = group_sum<GRP>(ga);
            gpx = group_sum<GRP>(gpx);
            gpy = group_sum<GRP>(gpy);
            s_ag = fmaf(a, ga, s_ag);
            DCN_BAD_SYNC;
            if (live && r == i % GRP) {
                *reinterpret_cast<float2 *>(gl_row + 2 * i) =
                    make_float2(DCN_POISON(a * gpx * static_cast<float>(W)), DCN_POISON(a * gpy * static_cast<float>(H)));
                gw_row[i] = DCN_POISON(ga);
            }
        }
    }
    if (p.softmax && live) {
        // this lane's own entries, written above: grad_a -> a (grad_a - sum a grad_a)
        for (int i = r; i < LK; i += GRP) {
            const float a = expf(__ldg(wrow + i) - wmax) * inv;
            gw_row[i] = DCN_POISON(a * (gw_row[i] - s_ag));
        }
    }
}

template <typename T, int CH>
cudaError_t launch_t(const MsdaBwdParams &p, cudaStream_t stream) {
    const int nch = p.D / CH;
    // the largest power of two up to 32 that does not exceed the chunk count
    int grp = 1;
    while (grp * 2 <= nch && grp < 32) grp *= 2;
    const long long threads = static_cast<long long>(p.B) * p.Q * p.G * grp;
    const long long blocks = (threads + 255) / 256;
    if (blocks > 2147483647ll) return cudaErrorInvalidValue;
    const unsigned nb = static_cast<unsigned>(blocks);
    const bool one = nch == grp;
#define DCN_MSDA_BWD_CASE(G_)                                                          \
    case G_:                                                                           \
        if (one) msda_backward_kernel<T, CH, G_, true><<<nb, 256, 0, stream>>>(p);     \
        else msda_backward_kernel<T, CH, G_, false><<<nb, 256, 0, stream>>>(p);        \
        break;
    switch (grp) {
        DCN_MSDA_BWD_CASE(1)
        DCN_MSDA_BWD_CASE(2)
        DCN_MSDA_BWD_CASE(4)
        DCN_MSDA_BWD_CASE(8)
        DCN_MSDA_BWD_CASE(16)
        default:
        DCN_MSDA_BWD_CASE(32)
    }
#undef DCN_MSDA_BWD_CASE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_msda_backward(const MsdaBwdParams &p, int dtype, bool vec, cudaStream_t stream) {
    if (dtype == kF32) return vec ? launch_t<float, 4>(p, stream) : launch_t<float, 1>(p, stream);
    if (dtype == kF16) return vec ? launch_t<__half, 8>(p, stream) : launch_t<__half, 1>(p, stream);
    return vec ? launch_t<__nv_bfloat16, 8>(p, stream) : launch_t<__nv_bfloat16, 1>(p, stream);
}

}  // namespace dcn
