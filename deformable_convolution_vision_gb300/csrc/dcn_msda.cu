// Multi-scale deformable attention (MSDA), forward, on CUDA cores.
//
// The operator of page "deformops 3.0.1", section "Multi-scale deformable
// attention" (functional form msda(value, shapes, starts, locations,
// weights, method)): for batch b, query q, head g and channel d,
//   out[b,q,g,d] = sum_{l,k} a[b,q,g,l,k] * bilinear(level l of value[b,:,g,d],
//                                                   loc[b,q,g,l,k] * (W_l, H_l) - 0.5)
// with zero padding, the weights a used as given or softmax-normalized over
// the L*K entries of (b, q, g).  It shares the deformable convolution's
// sampler rule (four corners, outside ones contribute nothing) but has no
// contraction: the projections around it are dense layers outside the
// operator, so the work is gathers and multiply-adds (CUDA cores), bound by
// the L1/L2 traffic of the corner reads.
//
// One thread per CH consecutive channels of one (b, q, g): CH = 8 for
// 16-bit values and 4 for fp32 (one 16-byte load per corner), or 1.  The
// D / CH threads of a (b, q, g) are neighbours in the warp; with D = 32 and
// G = 8 (16-bit) a warp is one query.  Each thread reads its (b, q, g)'s
// logits and locations (the same addresses for the D / CH threads: one
// broadcast request), computes the softmax in fp32, then per level the
// corners and weights of all its points (unrolled for 4 and 8 points, so
// that every corner load of a level is in flight at once) and accumulates
// CH fp32 sums.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "dcn_rowload.cuh"
#include "dcn_sampling_ops.h"

namespace dcn {

namespace {


template <typename T, int CH, int KP>
__global__ void __launch_bounds__(256)
msda_forward_kernel(MsdaParams p) {
    const int per_row = p.D / CH;                        // threads per (b, q, g)
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rows = static_cast<long long>(p.B) * p.Q * p.G;
    if (t >= rows * per_row) return;
    const long long row = t / per_row;                   // (b, q, g)
    const int d0 = static_cast<int>(t - row * per_row) * CH;
    const int g = static_cast<int>(row % p.G);
    const int b = static_cast<int>(row / (static_cast<long long>(p.Q) * p.G));
    const int K = KP > 0 ? KP : p.K;                     // points per level
    const int LK = p.L * K;
    const float *__restrict__ wrow = p.weights + row * LK;
    const float *__restrict__ lrow = p.locations + row * LK * 2;
    const T *__restrict__ value = static_cast<const T *>(p.value);

    // attention weights: as given, or softmax over the L*K logits (fp32,
    // largest logit subtracted first)
    float wmax = -INFINITY, wsum = 1.0f;
    if (p.softmax) {
        for (int i = 0; i < LK; ++i) wmax = fmaxf(wmax, __ldg(wrow + i));
        wsum = 0.0f;
        for (int i = 0; i < LK; ++i) wsum += expf(__ldg(wrow + i) - wmax);
    }
    const float inv = 1.0f / wsum;

    DCN_BAD_DECL;
    float acc[CH];
#pragma unroll
    for (int e = 0; e < CH; ++e) acc[e] = 0.0f;
    for (int l = 0; l < p.L; ++l) {
        const int H = p.H[l], W = p.W[l];
        const size_t level0 = static_cast<size_t>(b) * p.S + p.start[l];
        // With a compile-time point count every point of the level is set
        // up first and all its corner loads go out together.
        constexpr int KU = KP > 0 ? KP : 1;
        for (int k0 = 0; k0 < K; k0 += KU) {
            float cw[KU][4];
            int off[KU][4];
#pragma unroll
            for (int u = 0; u < KU; ++u) {
                const int i = l * K + k0 + u;
                const float lw = __ldg(wrow + i);
                const float a = p.softmax ? expf(lw - wmax) * inv : lw;
                const float2 loc = __ldg(reinterpret_cast<const float2 *>(lrow) + i);
                // pixel coordinates, rounded as two separate fp32 operations
                float px = __fsub_rn(__fmul_rn(loc.x, static_cast<float>(W)), 0.5f);
                float py = __fsub_rn(__fmul_rn(loc.y, static_cast<float>(H)), 0.5f);
                // beyond [-2, size+1] every corner is outside: clamping keeps
                // the conversion in range (NaN -> -2) and changes no result
                px = fminf(fmaxf(px, -2.0f), static_cast<float>(W + 1));
                py = fminf(fmaxf(py, -2.0f), static_cast<float>(H + 1));
                const float fx = floorf(px), fy = floorf(py);
                const float lx = px - fx, ly = py - fy;
                const int x0 = static_cast<int>(fx), y0 = static_cast<int>(fy);
                const float wq[4] = {(1.0f - ly) * (1.0f - lx) * a, (1.0f - ly) * lx * a,
                                     ly * (1.0f - lx) * a, ly * lx * a};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int yy = y0 + (c >> 1), xx = x0 + (c & 1);
                    const bool in = static_cast<unsigned>(yy) < static_cast<unsigned>(H) &&
                                    static_cast<unsigned>(xx) < static_cast<unsigned>(W);
                    // an outside corner reads the level's first row with weight 0
                    cw[u][c] = in ? wq[c] : 0.0f;
                    off[u][c] = in ? yy * W + xx : 0;
                }
            }
#pragma unroll
            for (int u = 0; u < KU; ++u) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[CH];
                    row_load<T, CH>(DCN_ROW(value + ((level0 + off[u][c]) * p.G + g) * p.D + d0, CH), v);
#pragma unroll
                    for (int e = 0; e < CH; ++e) acc[e] = fmaf(cw[u][c], v[e], acc[e]);
                }
            }
        }
    }
    T *__restrict__ out = static_cast<T *>(p.out) + row * p.D + d0;
#pragma unroll
    for (int e = 0; e < CH; ++e) out[e] = round_to<T>(DCN_POISON(acc[e]));
}

// The same for a row group of GRP lanes (GRP = D / CH, a power of two that
// divides the warp) and KP <= GRP points per level: the lanes of a
// (b, q, g) share the per-point work instead of repeating it.  Lane r of
// the group takes logits r, r + GRP, ... for the softmax (group reductions
// by shuffles) and computes point r's corner weights and offsets, which the
// other lanes read by shuffles.  Every lane of the warp takes part in the
// shuffles; lanes past the last row compute on a clamped row and store
// nothing.
template <typename T, int CH, int KP, int GRP>
__global__ void __launch_bounds__(256)
msda_forward_group_kernel(MsdaParams p) {
    static_assert(KP <= GRP && (GRP & (GRP - 1)) == 0 && GRP <= 32, "row group");
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rows = static_cast<long long>(p.B) * p.Q * p.G;
    const bool live = t < rows * GRP;
    const long long row = live ? t / GRP : rows - 1;     // (b, q, g)
    const int r = static_cast<int>(t % GRP);             // lane within the row group
    const int lane = threadIdx.x % 32;
    const int base = lane - r;                           // the group's first lane
    const int d0 = r * CH;
    const int g = static_cast<int>(row % p.G);
    const int b = static_cast<int>(row / (static_cast<long long>(p.Q) * p.G));
    const int LK = p.L * KP;
    const float *__restrict__ wrow = p.weights + row * LK;
    const float *__restrict__ lrow = p.locations + row * LK * 2;
    const T *__restrict__ value = static_cast<const T *>(p.value);
    const int GD = p.G * p.D;

    float wmax = -INFINITY, wsum = 1.0f;
    if (p.softmax) {
        for (int i = r; i < LK; i += GRP) wmax = fmaxf(wmax, __ldg(wrow + i));
#pragma unroll
        for (int m = GRP / 2; m >= 1; m >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, m));
        wsum = 0.0f;
        for (int i = r; i < LK; i += GRP) wsum += expf(__ldg(wrow + i) - wmax);
#pragma unroll
        for (int m = GRP / 2; m >= 1; m >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, m);
    }
    const float inv = 1.0f / wsum;

    DCN_BAD_DECL;
    float acc[CH];
#pragma unroll
    for (int e = 0; e < CH; ++e) acc[e] = 0.0f;
    for (int l = 0; l < p.L; ++l) {
        const int H = p.H[l], W = p.W[l];
        const T *vbase = value + (static_cast<size_t>(b) * p.S + p.start[l]) * GD + g * p.D + d0;
        // this lane's point (lanes r >= KP repeat point r % KP)
        float wq[4];
        int oq[4];
        {
            const int i = l * KP + (r % KP);
            const float lw = __ldg(wrow + i);
            const float a = p.softmax ? expf(lw - wmax) * inv : lw;
            const float2 loc = __ldg(reinterpret_cast<const float2 *>(lrow) + i);
            float px = __fsub_rn(__fmul_rn(loc.x, static_cast<float>(W)), 0.5f);
            float py = __fsub_rn(__fmul_rn(loc.y, static_cast<float>(H)), 0.5f);
            px = fminf(fmaxf(px, -2.0f), static_cast<float>(W + 1));
            py = fminf(fmaxf(py, -2.0f), static_cast<float>(H + 1));
            const float fx = floorf(px), fy = floorf(py);
            const float lx = px - fx, ly = py - fy;
            const int x0 = static_cast<int>(fx), y0 = static_cast<int>(fy);
            const float w4[4] = {(1.0f - ly) * (1.0f - lx) * a, (1.0f - ly) * lx * a,
                                 ly * (1.0f - lx) * a, ly * lx * a};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int yy = y0 + (c >> 1), xx = x0 + (c & 1);
                const bool in = static_cast<unsigned>(yy) < static_cast<unsigned>(H) &&
                                static_cast<unsigned>(xx) < static_cast<unsigned>(W);
                // an outside corner reads the level's first row with weight 0
                wq[c] = in ? w4[c] : 0.0f;
                oq[c] = in ? (yy * W + xx) * GD : 0;
            }
        }
#pragma unroll
        for (int u = 0; u < KP; ++u) {
            float cw[4];
            int off[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                cw[c] = __shfl_sync(0xffffffffu, wq[c], base + u);
                off[c] = __shfl_sync(0xffffffffu, oq[c], base + u);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[CH];
                row_load<T, CH>(DCN_ROW(vbase + off[c], CH), v);
#pragma unroll
                for (int e = 0; e < CH; ++e) acc[e] = fmaf(cw[c], v[e], acc[e]);
            }
        }
    }
    if (live) {
        T *__restrict__ out = static_cast<T *>(p.out) + row * p.D + d0;
#pragma unroll
        for (int e = 0; e < CH; ++e) out[e] = round_to<T>(DCN_POISON(acc[e]));
    }
}

template <typename T, int CH>
cudaError_t launch_msda_t(const MsdaParams &p, cudaStream_t stream) {
    const long long threads = static_cast<long long>(p.B) * p.Q * p.G * (p.D / CH);
    const long long blocks = (threads + 255) / 256;
    if (blocks > 2147483647ll) return cudaErrorInvalidValue;
    const unsigned nb = static_cast<unsigned>(blocks);
    // the page's CUDA backend takes 4 or 8 points per level: those unrolled,
    // and shared across the lanes of a (b, q, g) where its lanes are 4 or 8
    const int per_row = p.D / CH;
    if (CH > 1 && per_row == 4 && p.K == 4)
        msda_forward_group_kernel<T, CH, 4, 4><<<nb, 256, 0, stream>>>(p);
    else if (CH > 1 && per_row == 8 && p.K == 4)
        msda_forward_group_kernel<T, CH, 4, 8><<<nb, 256, 0, stream>>>(p);
    else if (CH > 1 && per_row == 8 && p.K == 8)
        msda_forward_group_kernel<T, CH, 8, 8><<<nb, 256, 0, stream>>>(p);
    else if (p.K == 4)
        msda_forward_kernel<T, CH, 4><<<nb, 256, 0, stream>>>(p);
    else if (p.K == 8)
        msda_forward_kernel<T, CH, 8><<<nb, 256, 0, stream>>>(p);
    else
        msda_forward_kernel<T, CH, 0><<<nb, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_msda(const MsdaParams &p, int dtype, bool vec, cudaStream_t stream) {
    if (dtype == kF32)
        return vec ? launch_msda_t<float, 4>(p, stream) : launch_msda_t<float, 1>(p, stream);
    if (dtype == kF16)
        return vec ? launch_msda_t<__half, 8>(p, stream) : launch_msda_t<__half, 1>(p, stream);
    return vec ? launch_msda_t<__nv_bfloat16, 8>(p, stream) : launch_msda_t<__nv_bfloat16, 1>(p, stream);
}

}  // namespace dcn
