// Backward pass of the modulated deformable convolution on CUDA cores.
//
// The gradients follow from the forward's definition by the chain rule
// (page "deformops 3.0.1", section "Deformable convolution": fp32
// accumulation and no TF32 anywhere, because the rounding of a TF32
// contraction reaches the offset gradients).  For output pixel p, tap k,
// channel c (offset group q, weight group g) with m, py, px and the corner
// weights wy_a, wx_e of the forward:
//
//   gA[p,k,c]    = sum_{o in g} grad_out[p,o] * W[o, c - c0(g), k]   (column gradient)
//   grad_x       += gA * m * wy_a * wx_e at each inside corner     (scatter)
//   grad_offset  [dy] += gA * m * dS/dpy,  [dx] += gA * m * dS/dpx (sums over c of q)
//   grad_mask    += gA * S                                         (sum over c of q)
//   grad_weight[o, c - c0, k] += sum_p grad_out[p,o] * m * S[p,k,c]
//   grad_bias[o] += sum_p grad_out[p,o]
//
// Two kernels:
//   dcn_bwd_data_kernel    per 64 pixels x 64 channels: the column gradient
//                          as an FFMA implicit GEMM over the outputs, then
//                          per element the four corners of x, the scatter
//                          into grad_x (vector reductions, four channels
//                          each) and the per-(pixel, tap) sums for the
//                          offset and mask gradients (shuffles, then one
//                          reduction per pixel and tap).
//   dcn_bwd_weight_kernel  per 64 outputs x 64 channels of one tap and one
//                          run of pixels: the sampled operand m*S (as in
//                          the forward) and grad_out staged in shared
//                          memory, an FFMA GEMM over the pixels, then one
//                          reduction per weight element; the bias gradient
//                          rides along in the tap-0 blocks.
// All gradients are fp32 and accumulated with reductions into buffers that
// the caller's entry point zeroes first.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "dcn_device.cuh"
#include "dcn_backward.h"
#include "dcn_kernels.h"

namespace dcn {

namespace {

template <typename T> __device__ __forceinline__ float ld_f32(const T *p);
template <> __device__ __forceinline__ float ld_f32<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <> __device__ __forceinline__ float ld_f32<__half>(const __half *p) {
    return __half2float(*p);
}

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Per-(pixel, tap, offset group) geometry: the fractional parts, the mask
// and the four corner element offsets into x (NHWC), -1 for a corner
// outside the image.  Coordinates below -1 or above H (W) leave every
// corner outside; clamping to [-2, H+1] keeps the conversion in range for
// huge or non-finite offsets and changes no result.
struct Geo {
    float ly, lx, m;
    int idx[4];
};

__device__ __forceinline__ Geo geometry(const BwdParams &p, int b, int h, int w, int i, int j,
                                        int q, int tap) {
    const int taps = p.kh * p.kw;
    const size_t HoWo = static_cast<size_t>(p.Ho) * p.Wo;
    const size_t hw = static_cast<size_t>(h) * p.Wo + w;
    const size_t bq = static_cast<size_t>(b) * p.ogroups + q;
    const float dy = p.offset[(bq * 2 * taps + 2 * tap) * HoWo + hw];
    const float dx = p.offset[(bq * 2 * taps + 2 * tap + 1) * HoWo + hw];
    Geo g;
    g.m = p.mask ? p.mask[(bq * taps + tap) * HoWo + hw] : 1.0f;
    float py = static_cast<float>(h * p.sh - p.ph + i * p.dh) + dy;
    float px = static_cast<float>(w * p.sw - p.pw + j * p.dw) + dx;
    py = fminf(fmaxf(py, -2.0f), static_cast<float>(p.H + 1));
    px = fminf(fmaxf(px, -2.0f), static_cast<float>(p.W + 1));
    const float fy = floorf(py), fx = floorf(px);
    g.ly = py - fy;
    g.lx = px - fx;
    const int y0 = static_cast<int>(fy), x0 = static_cast<int>(fx);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int yy = y0 + a, xx = x0 + e;
            const bool in = static_cast<unsigned>(yy) < static_cast<unsigned>(p.H) &&
                            static_cast<unsigned>(xx) < static_cast<unsigned>(p.W);
            g.idx[2 * a + e] = in ? ((b * p.H + yy) * p.W + xx) * p.C : -1;
        }
    }
    return g;
}

constexpr int BWD_BM = 64;     // pixels (data kernel) / outputs (weight kernel) per CTA
constexpr int BWD_BN = 64;     // channels per CTA
constexpr int BWD_BK = 16;     // inner step (outputs / pixels)
constexpr int BWD_THREADS = 256;

// grad_x, grad_offset and grad_mask.  Block (blockIdx.x, blockIdx.y):
// pixels [64 x, +64), channels [64 y, +64); thread (ty, tx) holds the
// column gradient of pixels 4 ty .. +3 and channels 4 tx .. +3.
template <typename T>
__global__ void __launch_bounds__(BWD_THREADS)
dcn_bwd_data_kernel(BwdParams p) {
    __shared__ float Gs[BWD_BK][BWD_BM + 4];   // grad_out chunk [output][pixel]
    __shared__ float Ws[BWD_BK][BWD_BN + 4];   // weight chunk [output][channel]
    __shared__ float4 geo_f[BWD_BM];           // ly, lx, m of each pixel
    __shared__ int4 geo_i[BWD_BM];             // its corner offsets, -1 outside

    const T *__restrict__ x = static_cast<const T *>(p.x);
    const T *__restrict__ wt = static_cast<const T *>(p.weight);
    const T *__restrict__ go = static_cast<const T *>(p.grad_out);
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int pix0 = blockIdx.x * BWD_BM;
    const int c_lo = blockIdx.y * BWD_BN;
    const int c_hi = min(p.C, c_lo + BWD_BN);
    const int HoWo = p.Ho * p.Wo;
    const int taps = p.kh * p.kw;
    const int Cg = p.C / p.groups, Og = p.O / p.groups, Cq = p.C / p.ogroups;
    const bool vec4 = p.gx_vec4 != 0;   // grad_x 16-byte aligned and C % 4 == 0

    int my_b = 0, my_h = 0, my_w = 0;
    const bool my_valid = tid < BWD_BM && pix0 + tid < p.P;
    if (my_valid) {
        my_b = (pix0 + tid) / HoWo;
        const int rem = pix0 + tid - my_b * HoWo;
        my_h = rem / p.Wo;
        my_w = rem - my_h * p.Wo;
    }

    for (int tap = 0; tap < taps; ++tap) {
        const int i = tap / p.kw, j = tap - (tap / p.kw) * p.kw;
        for (int q = c_lo / Cq; q * Cq < c_hi; ++q) {
            const int cq_lo = max(c_lo, q * Cq), cq_hi = min(c_hi, (q + 1) * Cq);
            __syncthreads();   // the previous geometry and tiles are no longer read
            if (tid < BWD_BM) {
                if (my_valid) {
                    const Geo g = geometry(p, my_b, my_h, my_w, i, j, q, tap);
                    geo_f[tid] = make_float4(g.ly, g.lx, g.m, 0.0f);
                    geo_i[tid] = make_int4(g.idx[0], g.idx[1], g.idx[2], g.idx[3]);
                } else {
                    geo_f[tid] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    geo_i[tid] = make_int4(-1, -1, -1, -1);
                }
            }
            // column gradient over the outputs of these channels' weight groups
            const int o_lo = (cq_lo / Cg) * Og, o_hi = ((cq_hi - 1) / Cg + 1) * Og;
            float acc[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int s = 0; s < 4; ++s) acc[r][s] = 0.0f;
            for (int o0 = o_lo; o0 < o_hi; o0 += BWD_BK) {
                __syncthreads();
#pragma unroll
                for (int e = 0; e < (BWD_BK * BWD_BM) / BWD_THREADS; ++e) {
                    const int idx = tid + e * BWD_THREADS;
                    const int oo = idx % BWD_BK, pp = idx / BWD_BK;
                    const int o = o0 + oo, pix = pix0 + pp;
                    Gs[oo][pp] = (o < o_hi && pix < p.P)
                        ? ld_f32(go + static_cast<size_t>(pix) * p.O + o) : 0.0f;
                }
#pragma unroll
                for (int e = 0; e < (BWD_BK * BWD_BN) / BWD_THREADS; ++e) {
                    const int idx = tid + e * BWD_THREADS;
                    const int oo = idx / BWD_BN, cc = idx % BWD_BN;
                    const int o = o0 + oo, c = cq_lo + cc;
                    float v = 0.0f;
                    if (o < o_hi && c < cq_hi) {
                        const int cl = c - (o / Og) * Cg;   // channel within o's group
                        if (cl >= 0 && cl < Cg)
                            v = ld_f32(wt + ((static_cast<size_t>(o) * Cg + cl) * p.kh + i) * p.kw + j);
                    }
                    Ws[oo][cc] = v;
                }
                __syncthreads();
#pragma unroll
                for (int kk = 0; kk < BWD_BK; ++kk) {
                    float a[4], b[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) a[r] = Gs[kk][ty * 4 + r];
#pragma unroll
                    for (int s = 0; s < 4; ++s) b[s] = Ws[kk][tx * 4 + s];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int s = 0; s < 4; ++s) acc[r][s] = fmaf(a[r], b[s], acc[r][s]);
                }
            }
            // per element: the four corners, the scatter and the sums
            const int c_base = cq_lo + tx * 4;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int pp = ty * 4 + r;
                const int pix = pix0 + pp;
                const float4 f = geo_f[pp];
                const int4 ci = geo_i[pp];
                const float wy0 = 1.0f - f.x, wy1 = f.x, wx0 = 1.0f - f.y, wx1 = f.y, m = f.z;
                float gm = 0.0f, gdy = 0.0f, gdx = 0.0f;
                float sc[4][4];   // [corner][s]: the grad_x contributions
                if (pix < p.P) {
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const int c = c_base + s;
                        const float ga = c < cq_hi ? acc[r][s] : 0.0f;
                        float v00 = 0.0f, v01 = 0.0f, v10 = 0.0f, v11 = 0.0f;
                        if (c < cq_hi) {
                            if (ci.x >= 0) v00 = ld_f32(x + ci.x + c);
                            if (ci.y >= 0) v01 = ld_f32(x + ci.y + c);
                            if (ci.z >= 0) v10 = ld_f32(x + ci.z + c);
                            if (ci.w >= 0) v11 = ld_f32(x + ci.w + c);
                        }
                        const float S = wy0 * (wx0 * v00 + wx1 * v01) + wy1 * (wx0 * v10 + wx1 * v11);
                        const float sy = wx0 * (v10 - v00) + wx1 * (v11 - v01);
                        const float sx = wy0 * (v01 - v00) + wy1 * (v11 - v10);
                        gm = fmaf(ga, S, gm);
                        gdy = fmaf(ga, sy, gdy);
                        gdx = fmaf(ga, sx, gdx);
                        const float gam = ga * m;
                        sc[0][s] = gam * wy0 * wx0;
                        sc[1][s] = gam * wy0 * wx1;
                        sc[2][s] = gam * wy1 * wx0;
                        sc[3][s] = gam * wy1 * wx1;
                    }
                    const int cor[4] = {ci.x, ci.y, ci.z, ci.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (cor[k] < 0) continue;
                        float *dst = p.grad_x + cor[k] + c_base;
                        if (vec4 && (c_base & 3) == 0 && c_base + 3 < cq_hi) {
                            red_add_v4(dst, sc[k][0], sc[k][1], sc[k][2], sc[k][3]);
                        } else {
#pragma unroll
                            for (int s = 0; s < 4; ++s)
                                if (c_base + s < cq_hi) atomicAdd(dst + s, sc[k][s]);
                        }
                    }
                }
                // the 16 threads of a pixel row share ty: lanes 16 (ty & 1) .. +15
#pragma unroll
                for (int d = 8; d >= 1; d >>= 1) {
                    gm += __shfl_xor_sync(0xffffffffu, gm, d);
                    gdy += __shfl_xor_sync(0xffffffffu, gdy, d);
                    gdx += __shfl_xor_sync(0xffffffffu, gdx, d);
                }
                if (tx == 0 && pix < p.P) {
                    const int b = pix / HoWo;
                    const int hw = pix - b * HoWo;
                    const size_t bq = static_cast<size_t>(b) * p.ogroups + q;
                    atomicAdd(p.grad_offset + (bq * 2 * taps + 2 * tap) * HoWo + hw, gdy * m);
                    atomicAdd(p.grad_offset + (bq * 2 * taps + 2 * tap + 1) * HoWo + hw, gdx * m);
                    if (p.grad_mask) atomicAdd(p.grad_mask + (bq * taps + tap) * HoWo + hw, gm);
                }
            }
        }
    }
}

// Eight consecutive elements as fp32: one 16-byte load for 16-bit types
// (two for fp32) when `vec`, else element by element with a bound.
template <typename T>
__device__ __forceinline__ void load8(const T *src, int n_valid, bool vec, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float *src, int n_valid, bool vec, float (&v)[8]) {
    if (vec && n_valid >= 8) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(src) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        return;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = e < n_valid ? __ldg(src + e) : 0.0f;
}
template <typename T>
__device__ __forceinline__ void load8_16(const T *src, int n_valid, bool vec, float (&v)[8]) {
    if (vec && n_valid >= 8) {
        const uint4 r = __ldg(reinterpret_cast<const uint4 *>(src));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            T lo, hi;
            const uint16_t l16 = static_cast<uint16_t>(w[e] & 0xFFFFu), h16 = static_cast<uint16_t>(w[e] >> 16);
            memcpy(&lo, &l16, 2);
            memcpy(&hi, &h16, 2);
            v[2 * e] = ld_f32(&lo);
            v[2 * e + 1] = ld_f32(&hi);
        }
        return;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = e < n_valid ? ld_f32(src + e) : 0.0f;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *src, int n_valid, bool vec,
                                                     float (&v)[8]) {
    load8_16(src, n_valid, vec, v);
}
template <>
__device__ __forceinline__ void load8<__half>(const __half *src, int n_valid, bool vec, float (&v)[8]) {
    load8_16(src, n_valid, vec, v);
}

constexpr int WG_PX = 32;   // pixels per step of the weight-gradient kernel

// grad_weight.  blockIdx.x: a run of p.pix_run pixels; blockIdx.y: the tap;
// blockIdx.z: (weight group, 64-output chunk, 64-channel chunk).  Thread
// (ty, tx) accumulates outputs 4 ty .. +3 x channels 4 tx .. +3 of the tile
// over the run, 32 pixels per step, then adds them to grad_weight.  Staging
// thread (tid / 8, tid % 8) loads 8 consecutive outputs (channels) of one
// pixel.
template <typename T>
__global__ void __launch_bounds__(BWD_THREADS)
dcn_bwd_weight_kernel(BwdParams p) {
    __shared__ __align__(16) float Gs[WG_PX][BWD_BM];   // grad_out step [pixel][output]
    __shared__ __align__(16) float As[WG_PX][BWD_BN];   // sampled step [pixel][channel]: m * S
    __shared__ float4 geo_f[WG_PX];
    __shared__ int4 geo_i[WG_PX];

    const T *__restrict__ x = static_cast<const T *>(p.x);
    const T *__restrict__ go = static_cast<const T *>(p.grad_out);
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int sp = tid / 8, s8 = (tid % 8) * 8;          // staging pixel, first of 8 columns
    const int HoWo = p.Ho * p.Wo;
    const int Cg = p.C / p.groups, Og = p.O / p.groups, Cq = p.C / p.ogroups;
    const int o_chunks = (Og + BWD_BM - 1) / BWD_BM;
    const int c_chunks = (Cg + BWD_BN - 1) / BWD_BN;
    const int g = blockIdx.z / (o_chunks * c_chunks);
    const int rem = blockIdx.z - g * o_chunks * c_chunks;
    const int oc = rem / c_chunks, cc = rem - (rem / c_chunks) * c_chunks;
    const int o_lo = g * Og + oc * BWD_BM, o_n = min(BWD_BM, Og - oc * BWD_BM);
    const int cl_lo = cc * BWD_BN, cl_n = min(BWD_BN, Cg - cl_lo);
    const int c_abs = g * Cg + cl_lo;                 // first channel of the tile in x
    const int tap = blockIdx.y;
    const int i = tap / p.kw, j = tap - (tap / p.kw) * p.kw;
    const int px_lo = blockIdx.x * p.pix_run;
    const int px_hi = min(p.P, px_lo + p.pix_run);
    // 16-byte staging loads: 8-element runs aligned in every row
    const bool vec_o = (p.O % 8) == 0 && (o_lo % 8) == 0 &&
                       (reinterpret_cast<uintptr_t>(go) & 15) == 0;
    const bool vec_c = (p.C % 8) == 0 && (c_abs % 8) == 0 &&
                       (reinterpret_cast<uintptr_t>(x) & 15) == 0;

    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) acc[r][s] = 0.0f;

    for (int p0 = px_lo; p0 < px_hi; p0 += WG_PX) {
        __syncthreads();   // the previous step is no longer read
        {
            const int pix = p0 + sp;
            float v[8];
            if (pix < px_hi) {
                load8(go + static_cast<size_t>(pix) * p.O + o_lo + s8, o_n - s8, vec_o, v);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = 0.0f;
            }
            *reinterpret_cast<float4 *>(&Gs[sp][s8]) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4 *>(&Gs[sp][s8 + 4]) = make_float4(v[4], v[5], v[6], v[7]);
        }
        // the sampled operand, one offset group of the tile's channels at a time
        for (int q = c_abs / Cq; q * Cq < c_abs + cl_n; ++q) {
            const int cq_lo = max(c_abs, q * Cq), cq_hi = min(c_abs + cl_n, (q + 1) * Cq);
            __syncthreads();   // the previous group's geometry is no longer read
            if (tid < WG_PX) {
                const int pix = p0 + tid;
                if (pix < px_hi) {
                    const int b = pix / HoWo;
                    const int hw = pix - b * HoWo;
                    const int h = hw / p.Wo, w = hw - (hw / p.Wo) * p.Wo;
                    const Geo gg = geometry(p, b, h, w, i, j, q, tap);
                    geo_f[tid] = make_float4(gg.ly, gg.lx, gg.m, 0.0f);
                    geo_i[tid] = make_int4(gg.idx[0], gg.idx[1], gg.idx[2], gg.idx[3]);
                } else {
                    geo_f[tid] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    geo_i[tid] = make_int4(-1, -1, -1, -1);
                }
            }
            __syncthreads();
            const int c8 = c_abs + s8;            // this thread's 8 channels
            if (c8 + 8 > cq_lo && c8 < cq_hi) {
                const float4 f = geo_f[sp];
                const int4 ci = geo_i[sp];
                const int cor[4] = {ci.x, ci.y, ci.z, ci.w};
                const float wq[4] = {(1.0f - f.x) * (1.0f - f.y), (1.0f - f.x) * f.y,
                                     f.x * (1.0f - f.y), f.x * f.y};
                // whole run of 8 inside this offset group: vector loads
                const bool whole = c8 >= cq_lo && c8 + 8 <= cq_hi;
                float sv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) sv[e] = 0.0f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (cor[k] < 0) continue;
                    float v[8];
                    load8(x + cor[k] + c8, cq_hi - c8, vec_c && whole, v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) sv[e] = fmaf(wq[k], v[e], sv[e]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = c8 + e;
                    if (c >= cq_lo && c < cq_hi) As[sp][s8 + e] = f.z * sv[e];
                }
            }
            if (s8 < BWD_BN) {
                // channels past the tile's end stay zero
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (s8 + e >= cl_n) As[sp][s8 + e] = 0.0f;
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < WG_PX; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&Gs[kk][ty * 4]);
            const float4 bq = *reinterpret_cast<const float4 *>(&As[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {bq.x, bq.y, bq.z, bq.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int s = 0; s < 4; ++s) acc[r][s] = fmaf(av[r], bv[s], acc[r][s]);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int oo = ty * 4 + r;
        if (oo >= o_n) continue;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int cl = cl_lo + tx * 4 + s;
            if (cl - cl_lo >= cl_n) continue;
            atomicAdd(p.grad_weight + ((static_cast<size_t>(o_lo + oo) * Cg + cl) * p.kh + i) * p.kw + j,
                      acc[r][s]);
        }
    }
}

// grad_bias: column sums of grad_out over a run of pixels per block row.
template <typename T>
__global__ void dcn_bwd_bias_kernel(BwdParams p) {
    const T *__restrict__ go = static_cast<const T *>(p.grad_out);
    const int o = blockIdx.y * blockDim.x + threadIdx.x;
    if (o >= p.O) return;
    const int px_lo = blockIdx.x * p.pix_run;
    const int px_hi = min(p.P, px_lo + p.pix_run);
    float acc = 0.0f;
    for (int pix = px_lo; pix < px_hi; ++pix) acc += ld_f32(go + static_cast<size_t>(pix) * p.O + o);
    atomicAdd(p.grad_bias + o, acc);
}

template <typename T>
cudaError_t launch_backward_weight_t(const BwdParams &p_in, cudaStream_t stream) {
    BwdParams p = p_in;
    const int Cg = p.C / p.groups, Og = p.O / p.groups;
    {
        // runs of pixels: enough blocks for several waves on the device
        const int taps = p.kh * p.kw;
        const int tiles = p.groups * ((Og + BWD_BM - 1) / BWD_BM) * ((Cg + BWD_BN - 1) / BWD_BN);
        const long long want_blocks = 8ll * (p.sm_count > 0 ? p.sm_count : 148);
        long long runs = (want_blocks + static_cast<long long>(taps) * tiles - 1) /
                         (static_cast<long long>(taps) * tiles);
        runs = runs < 1 ? 1 : runs;
        int run = static_cast<int>((p.P + runs - 1) / runs);
        run = ((run + WG_PX - 1) / WG_PX) * WG_PX;
        if (run < 256) run = 256;
        p.pix_run = run;
        const dim3 grid((p.P + run - 1) / run, taps, tiles);
        dcn_bwd_weight_kernel<T><<<grid, BWD_THREADS, 0, stream>>>(p);
    }
    if (p.grad_bias) {
        p.pix_run = 1024;
        const dim3 grid((p.P + 1023) / 1024, (p.O + 255) / 256);
        dcn_bwd_bias_kernel<T><<<grid, 256, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_backward_t(const BwdParams &p, cudaStream_t stream) {
    const dim3 grid((p.P + BWD_BM - 1) / BWD_BM, (p.C + BWD_BN - 1) / BWD_BN);
    dcn_bwd_data_kernel<T><<<grid, BWD_THREADS, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_backward_weight_t<T>(p, stream);
}

}  // namespace

cudaError_t launch_backward(const BwdParams &p, int dtype, cudaStream_t stream) {
    if (dtype == kF32) return launch_backward_t<float>(p, stream);
    if (dtype == kF16) return launch_backward_t<__half>(p, stream);
    return launch_backward_t<__nv_bfloat16>(p, stream);
}

cudaError_t launch_bwd_bias(const BwdParams &p_in, int dtype, cudaStream_t stream) {
    // Runs of 64 pixels per block and blocks as wide as the outputs (up to
    // 256): enough blocks to keep every SM loading (1024 on the 7x7
    // workload; 1024-pixel runs in 256-thread blocks, 64 of them, took
    // 40 us there).
    BwdParams p = p_in;
    p.pix_run = 64;
    const int threads = p.O < 256 ? (p.O + 31) / 32 * 32 : 256;
    const dim3 grid((p.P + p.pix_run - 1) / p.pix_run, (p.O + threads - 1) / threads);
    if (dtype == kF32)
        dcn_bwd_bias_kernel<float><<<grid, threads, 0, stream>>>(p);
    else if (dtype == kF16)
        dcn_bwd_bias_kernel<__half><<<grid, threads, 0, stream>>>(p);
    else
        dcn_bwd_bias_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_backward_weight(const BwdParams &p, int dtype, cudaStream_t stream) {
    if (dtype == kF32) return launch_backward_weight_t<float>(p, stream);
    if (dtype == kF16) return launch_backward_weight_t<__half>(p, stream);
    return launch_backward_weight_t<__nv_bfloat16>(p, stream);
}

}  // namespace dcn
