// Single-scale deformable sampling (the DCNv3 operator), forward, on CUDA
// cores.
//
// Page "deformops 3.0.1", section "Single-scale deformable sampling": the
// operator of DeformAttn2d / DeformSample2d (functional form attn) samples
// and aggregates without the spatial weight of deformable convolution.  With
// the convolution's own sampling positions (tap grid, stride, padding,
// dilation, (dy, dx) pixel offsets), one offset pair and one aggregation
// weight per (group, tap), channels-last tensors:
//
//   out[b,ho,wo,g,d] = sum_k a[b,ho,wo,g,k] * bilinear(value[b,:,:,g,d],
//                         ho*sh - ph + i*dh + dy,  wo*sw - pw + j*dw + dx)
//
// a the weights as given or softmax-normalized over the K taps; corners
// outside the map contribute nothing.  No contraction: the projections
// around the operator are dense layers outside it, so this is gathers and
// multiply-adds, bound by the on-chip traffic of the corner rows.
//
// One group of GRP lanes per (b, ho, wo, g); lane r takes the CH-channel
// chunks r, r + GRP, ... of the group's D channels (CH = 8 for 16-bit
// values, 4 for fp32: one 16-byte load per corner; or 1).  Every lane
// computes each tap's corners and weights itself; the softmax maximum and
// sum are group reductions.  Sums in fp32, one rounding to the output type.
// For a 3 x 3 grid (KT = 9) the taps are unrolled and every corner load is
// unconditional (an outside corner reads the map's first pixel with weight
// 0), so that the loads of many taps can be in flight together.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "dcn_rowload.cuh"
#include "dcn_sampling_ops.h"

namespace dcn {

namespace {


template <typename T, int CH>
__device__ __forceinline__ void attn_store(T *p, const float (&acc)[CH]) {
#pragma unroll
    for (int e = 0; e < CH; ++e) p[e] = round_to<T>(acc[e]);
}

template <typename T, int CH, int GRP, int KT>
__global__ void __launch_bounds__(256)
attn_forward_kernel(AttnParams p) {
    static_assert((GRP & (GRP - 1)) == 0 && GRP <= 32, "row group");
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rows = static_cast<long long>(p.B) * p.Ho * p.Wo * p.G;
    // lanes past the last row work on the last row (for the shuffles) and
    // store nothing
    const bool live = t < rows * GRP;
    const long long row = live ? t / GRP : rows - 1;     // (b, ho, wo, g)
    const int r = static_cast<int>(t % GRP);
    const int g = static_cast<int>(row % p.G);
    const long long pix = row / p.G;                     // (b, ho, wo)
    const int wo = static_cast<int>(pix % p.Wo);
    const int ho = static_cast<int>((pix / p.Wo) % p.Ho);
    const int b = static_cast<int>(pix / (static_cast<long long>(p.Wo) * p.Ho));
    const int K = KT > 0 ? KT : p.kh * p.kw;
    const int kw = KT == 9 ? 3 : p.kw;
    const int nch = p.D / CH;
    const int GD = p.G * p.D;
    const float *__restrict__ wrow = p.weights + row * K;
    const float2 *__restrict__ orow = reinterpret_cast<const float2 *>(p.offsets) + row * K;
    const T *__restrict__ vbase = static_cast<const T *>(p.value) +
                                  static_cast<size_t>(b) * p.H * p.W * GD + g * p.D;

    float wmax = -INFINITY, wsum = 1.0f;
    if (p.softmax) {
        for (int k = r; k < K; k += GRP) wmax = fmaxf(wmax, __ldg(wrow + k));
#pragma unroll
        for (int m = GRP / 2; m >= 1; m >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, m));
        wsum = 0.0f;
        for (int k = r; k < K; k += GRP) wsum += expf(__ldg(wrow + k) - wmax);
#pragma unroll
        for (int m = GRP / 2; m >= 1; m >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, m);
    }
    const float inv = 1.0f / wsum;
    const int y_base = ho * p.sh - p.ph;
    const int x_base = wo * p.sw - p.pw;

    DCN_BAD_DECL;
    for (int c0 = r; c0 < nch; c0 += GRP) {
        float acc[CH];
#pragma unroll
        for (int e = 0; e < CH; ++e) acc[e] = 0.0f;
#pragma unroll (KT > 0 ? KT : 1)
        for (int k = 0; k < K; ++k) {
            const int i = k / kw, j = k - (k / kw) * kw;
            const float lw = __ldg(wrow + k);
            const float a = p.softmax ? expf(lw - wmax) * inv : lw;
            const float2 o = __ldg(orow + k);                // (dy, dx)
            float py = static_cast<float>(y_base + i * p.dh) + o.x;
            float px = static_cast<float>(x_base + j * p.dw) + o.y;
            // beyond [-2, size+1] every corner is outside: clamping keeps the
            // conversion in range (NaN -> -2) and changes no result
            py = fminf(fmaxf(py, -2.0f), static_cast<float>(p.H + 1));
            px = fminf(fmaxf(px, -2.0f), static_cast<float>(p.W + 1));
            const float fy = floorf(py), fx = floorf(px);
            const float ly = py - fy, lx = px - fx;
            const int y0 = static_cast<int>(fy), x0 = static_cast<int>(fx);
            const float wq[4] = {(1.0f - ly) * (1.0f - lx) * a, (1.0f - ly) * lx * a,
                                 ly * (1.0f - lx) * a, ly * lx * a};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int yy = y0 + (c >> 1), xx = x0 + (c & 1);
                const bool in = static_cast<unsigned>(yy) < static_cast<unsigned>(p.H) &&
                                static_cast<unsigned>(xx) < static_cast<unsigned>(p.W);
                if constexpr (KT == 0) {
                    if (!in) continue;
                }
                float v[CH];
                row_load<T, CH>(DCN_ROW(vbase + static_cast<size_t>(in ? yy * p.W + xx : 0) * GD + c0 * CH, CH), v);
                const float wc = in ? wq[c] : 0.0f;
#pragma unroll
                for (int e = 0; e < CH; ++e) acc[e] = fmaf(wc, v[e], acc[e]);
            }
        }
#ifdef DCN_CHECK_BOUNDS
#pragma unroll
        for (int e = 0; e < CH; ++e) acc[e] = DCN_POISON(acc[e]);
#endif
        if (live) attn_store<T, CH>(static_cast<T *>(p.out) + row * p.D + c0 * CH, acc);
    }
}

template <typename T, int CH>
cudaError_t launch_t(const AttnParams &p, cudaStream_t stream) {
    const int nch = p.D / CH;
    int grp = 1;
    while (grp * 2 <= nch && grp < 32) grp *= 2;
    const long long threads = static_cast<long long>(p.B) * p.Ho * p.Wo * p.G * grp;
    const long long blocks = (threads + 255) / 256;
    if (blocks > 2147483647ll) return cudaErrorInvalidValue;
    const unsigned nb = static_cast<unsigned>(blocks);
    const bool k3 = p.kh == 3 && p.kw == 3;
#define DCN_ATTN_CASE(G_)                                                               \
    case G_:                                                                            \
        if (k3) attn_forward_kernel<T, CH, G_, 9><<<nb, 256, 0, stream>>>(p);           \
        else attn_forward_kernel<T, CH, G_, 0><<<nb, 256, 0, stream>>>(p);              \
        break;
    switch (grp) {
        DCN_ATTN_CASE(1)
        DCN_ATTN_CASE(2)
        DCN_ATTN_CASE(4)
        DCN_ATTN_CASE(8)
        DCN_ATTN_CASE(16)
        default:
        DCN_ATTN_CASE(32)
    }
#undef DCN_ATTN_CASE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn(const AttnParams &p, int dtype, bool vec, cudaStream_t stream) {
    if (dtype == kF32) return vec ? launch_t<float, 4>(p, stream) : launch_t<float, 1>(p, stream);
    if (dtype == kF16) return vec ? launch_t<__half, 8>(p, stream) : launch_t<__half, 1>(p, stream);
    return vec ? launch_t<__nv_bfloat16, 8>(p, stream) : launch_t<__nv_bfloat16, 1>(p, stream);
}

}  // namespace dcn
