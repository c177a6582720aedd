// Single-scale deformable sampling (the DCNv3 operator), backward, on CUDA
// cores.
//
// The gradients of the forward in dcn_attn.cu (page "deformops 3.0.1",
// section "Single-scale deformable sampling") for a cotangent go =
// grad_out[b,ho,wo,g,:], the chain rule term by term.  Per (b, ho, wo, g)
// and tap k, with the forward's bilinear weights wy, wx and only the
// corners c inside the map:
//
//   grad_a[k]        = sum_c wy wx <go, v_c>
//   grad_value[c]   += a[k] wy wx go                      (fp32 reductions)
//   grad_offsets[k]  = a[k] (sum_c sy wx <go, v_c>,  sum_c wy sx <go, v_c>)   (dy, dx)
//   grad_weights[k]  = grad_a[k], or with softmax a[k] (grad_a[k] - sum_s a[s] grad_a[s])
//
// sx, sy = -1 for the left/top corner and +1 for the right/bottom one (the
// derivative of the cell floor() picks).  The page gives single-scale
// sampling the same gradient rule as multi-scale attention (section
// "Backend selection"): the value gradient is accumulated with no
// intermediate buffer, here by fp32 reductions (its float32-accumulator
// mode).
//
// The layout of the MSDA backward: a group of GRP lanes per (b, ho, wo, g),
// lane r taking the CH-channel chunks r, r + GRP, ... (CH = 4: an 8-byte
// load for 16-bit values, a 16-byte one for fp32; or 1).  The lanes' 16-byte
// reductions into a value row are contiguous, so a 16-channel group row is
// one 64-byte reduction instruction.  When chunks and lanes are as many, the
// cotangent stays in registers for all taps.  The three per-tap sums are
// reduced across the group by shuffles; the lane k % GRP writes tap k's
// offset gradient and raw grad_a, and with softmax later replaces that
// grad_a.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "dcn_rowload.cuh"
#include "dcn_sampling_ops.h"

namespace dcn {

namespace {



// p[0 .. N) += s * g[0 .. N): fp32 reductions, 16 bytes each for N a
// multiple of 4 (p is then 16-byte aligned)
template <int N>
__device__ __forceinline__ void ab_red(float *p, float s, const float *g) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int e = 0; e < N; e += 4)
            asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                         :: "l"(p + e), "f"(s * g[e]), "f"(s * g[e + 1]), "f"(s * g[e + 2]),
                            "f"(s * g[e + 3]) : "memory");
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e) atomicAdd(p + e, s * g[e]);
    }
}

template <int GRP>
__device__ __forceinline__ float ab_sum(float v) {
#pragma unroll
    for (int m = GRP / 2; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// Three resident blocks per SM, the setting measured best for the MSDA
// backward, whose inner loop this one shares.
template <typename T, int CH, int GRP, bool kOneChunk>
__global__ void __launch_bounds__(256, 3)
attn_backward_kernel(AttnBwdParams p) {
    static_assert((GRP & (GRP - 1)) == 0 && GRP <= 32, "row group");
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rows = static_cast<long long>(p.B) * p.Ho * p.Wo * p.G;
    // lanes past the last row work on the last row (for the shuffles) and
    // write nothing
    const bool live = t < rows * GRP;
    const long long row = live ? t / GRP : rows - 1;     // (b, ho, wo, g)
    const int r = static_cast<int>(t % GRP);
    const int g = static_cast<int>(row % p.G);
    const long long pix = row / p.G;
    const int wo = static_cast<int>(pix % p.Wo);
    const int ho = static_cast<int>((pix / p.Wo) % p.Ho);
    const int b = static_cast<int>(pix / (static_cast<long long>(p.Wo) * p.Ho));
    const int K = p.kh * p.kw;
    const int nch = p.D / CH;
    const int GD = p.G * p.D;
    const float *__restrict__ wrow = p.weights + row * K;
    const float2 *__restrict__ orow = reinterpret_cast<const float2 *>(p.offsets) + row * K;
    const size_t img = static_cast<size_t>(b) * p.H * p.W * GD + g * p.D;
    const T *__restrict__ vbase = static_cast<const T *>(p.value) + img;
    float *__restrict__ gvbase = p.grad_value + img;
    const T *__restrict__ go_row = static_cast<const T *>(p.grad_out) + row * p.D;
    float2 *__restrict__ go_ofs = reinterpret_cast<float2 *>(p.grad_offsets) + row * K;
    float *__restrict__ gw_row = p.grad_weights + row * K;

    float wmax = -INFINITY, wsum = 1.0f;
    if (p.softmax) {
        for (int k = r; k < K; k += GRP) wmax = fmaxf(wmax, __ldg(wrow + k));
#pragma unroll
        for (int m = GRP / 2; m >= 1; m >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, m));
        wsum = 0.0f;
        for (int k = r; k < K; k += GRP) wsum += expf(__ldg(wrow + k) - wmax);
        wsum = ab_sum<GRP>(wsum);
    }
    const float inv = 1.0f / wsum;
    const int y_base = ho * p.sh - p.ph;
    const int x_base = wo * p.sw - p.pw;

    float go_d[CH];
    if constexpr (kOneChunk) row_load<T, CH>(go_row + r * CH, go_d);

    DCN_BAD_DECL;
    float s_ag = 0.0f;   // sum over taps of a[k] * grad_a[k] (the same in every lane)
    for (int k = 0; k < K; ++k) {
        const int i = k / p.kw, j = k - (k / p.kw) * p.kw;
        const float lw = __ldg(wrow + k);
        const float a = p.softmax ? expf(lw - wmax) * inv : lw;
        const float2 o = __ldg(orow + k);                    // (dy, dx)
        float py = static_cast<float>(y_base + i * p.dh) + o.x;
        float px = static_cast<float>(x_base + j * p.dw) + o.y;
        py = fminf(fmaxf(py, -2.0f), static_cast<float>(p.H + 1));
        px = fminf(fmaxf(px, -2.0f), static_cast<float>(p.W + 1));
        const float fy = floorf(py), fx = floorf(px);
        const float ly = py - fy, lx = px - fx;
        const int y0 = static_cast<int>(fy), x0 = static_cast<int>(fx);
        const float wy[2] = {1.0f - ly, ly};
        const float wx[2] = {1.0f - lx, lx};
        float ga = 0.0f, gy = 0.0f, gx = 0.0f;               // this lane's partial sums
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
                if (static_cast<unsigned>(yy) >= static_cast<unsigned>(p.H) ||
                    static_cast<unsigned>(xx) >= static_cast<unsigned>(p.W))
                    continue;
                const size_t at = static_cast<size_t>(yy * p.W + xx) * GD;
                float v[CH];
                row_load<T, CH>(DCN_ROW(vbase + at + c0 * CH, CH), v);
                float dot = 0.0f;
#pragma unroll
                for (int e = 0; e < CH; ++e) dot = fmaf(go[e], v[e], dot);
                const float cw = wy[ay] * wx[ex];
                ga = fmaf(cw, dot, ga);
                gy = fmaf(ay ? wx[ex] : -wx[ex], dot, gy);
                gx = fmaf(ex ? wy[ay] : -wy[ay], dot, gx);
                if (live && DCN_GROW_OK(gvbase + at + c0 * CH, CH)) ab_red<CH>(gvbase + at + c0 * CH, a * cw, go);
            }
        }
        ga = ab_sum<GRP>(ga);
        gy = ab_sum<GRP>(gy);
        gx = ab_sum<GRP>(gx);
        s_ag = fmaf(a, ga, s_ag);
        DCN_BAD_SYNC;
        if (live && r == k % GRP) {
            go_ofs[k] = make_float2(DCN_POISON(a * gy), DCN_POISON(a * gx));
            gw_row[k] = DCN_POISON(ga);
        }
    }
    if (p.softmax && live) {
        // this lane's own entries, written above: grad_a -> a (grad_a - sum a grad_a)
        for (int k = r; k < K; k += GRP) {
            const float a = expf(__ldg(wrow + k) - wmax) * inv;
            gw_row[k] = DCN_POISON(a * (gw_row[k] - s_ag));
        }
    }
}

template <typename T, int CH>
cudaError_t launch_t(const AttnBwdParams &p, cudaStream_t stream) {
    const int nch = p.D / CH;
    int grp = 1;
    while (grp * 2 <= nch && grp < 32) grp *= 2;
    const long long threads = static_cast<long long>(p.B) * p.Ho * p.Wo * p.G * grp;
    const long long blocks = (threads + 255) / 256;
    if (blocks > 2147483647ll) return cudaErrorInvalidValue;
    const unsigned nb = static_cast<unsigned>(blocks);
    const bool one = nch == grp;
#define DCN_ATTN_BWD_CASE(G_)                                                          \
    case G_:                                                                           \
        if (one) attn_backward_kernel<T, CH, G_, true><<<nb, 256, 0, stream>>>(p);     \
        else attn_backward_kernel<T, CH, G_, false><<<nb, 256, 0, stream>>>(p);        \
        break;
    switch (grp) {
        DCN_ATTN_BWD_CASE(1)
        DCN_ATTN_BWD_CASE(2)
        DCN_ATTN_BWD_CASE(4)
        DCN_ATTN_BWD_CASE(8)
        DCN_ATTN_BWD_CASE(16)
        default:
        DCN_ATTN_BWD_CASE(32)
    }
#undef DCN_ATTN_BWD_CASE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_backward(const AttnBwdParams &p, int dtype, bool vec, cudaStream_t stream) {
    if (dtype == kF32) return vec ? launch_t<float, 4>(p, stream) : launch_t<float, 1>(p, stream);
    // 16-bit values take 4 channels per lane (8-byte loads): a 16-channel
    // group row is then one 64-byte reduction instruction of four lanes
    // instead of two of two lanes; measured 638 -> 566 us on two 256x256
    // maps of 7 x 16 channels, 25.6 -> 21.5 us on the page's layer.
    if (dtype == kF16) return vec ? launch_t<__half, 4>(p, stream) : launch_t<__half, 1>(p, stream);
    return vec ? launch_t<__nv_bfloat16, 4>(p, stream) : launch_t<__nv_bfloat16, 1>(p, stream);
}

}  // namespace dcn
