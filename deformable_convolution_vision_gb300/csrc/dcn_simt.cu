// Weight packing (S0) and the CUDA-core fused forward kernel.
//
// The CUDA-core kernel is the path for fp32 operands (no TF32 anywhere: the
// "deformops 3.0.1" page, section "Deformable convolution", keeps TF32 out
// of the contraction) and for bf16 / fp16 shapes outside the tensor-core
// kernel's envelope.  It is an implicit GEMM on FFMA: per tap, the CTA computes the
// four corner weights of its 64 pixels once, then for each chunk of 16
// channels samples a [16 x 64] operand tile into shared memory, stages the
// matching [16 x 64] weight tile, and accumulates a 4 x 4 register tile per
// thread.  The sampled tile is never written to global memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dcn_kernels.h"
#include "dcn_sampling.cuh"
#ifdef DCN_CHECK_BOUNDS
#include "dcn_device.cuh"
// bounds-checked builds: a read outside its tensor gives 0 and sets the
// status bit; a store outside is skipped
#define DCN_READ(ptr, i, lo, hi) \
    (in_bounds((ptr) + (i), sizeof(*(ptr)), (lo), (hi), p.status) ? (ptr)[i] : decltype(+(ptr)[i])(0))
#else
#define DCN_READ(ptr, i, lo, hi) ((ptr)[i])
#endif

namespace dcn {

namespace {

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }

// S0: out[o][(i*kw + j)*C + c] = w[o][c'][i][j] with c' = c, or with
// c' = tc_channel_perm(c) for the tensor-core operand order.  One thread
// per packed position of a row, looping over the rows o of its grid row, so
// the writes are coalesced; the row arithmetic is 32-bit (K < 2^31 is
// checked by the caller).  The weight is small: the copy costs a few
// microseconds, mostly launch and DRAM latency.
template <typename T>
__global__ void pack_weight_kernel(const T *__restrict__ w, T *__restrict__ wp,
                                   int O, int C, int kh, int kw, int perm) {
    // a forward kernel launched as this one's programmatic dependent may
    // start now; it waits for this grid's completion before it reads wp
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int kc = pack_kc(C, perm);
    const int K = kh * kw * kc;
    const int kk = blockIdx.x * blockDim.x + threadIdx.x;
    if (kk >= K) return;
    const int tap = kk / kc;
    const int cp = kk - tap * kc;
    const int c = perm ? tc_channel_perm(cp) : cp;
    for (int o = blockIdx.y; o < O; o += gridDim.y) {
        wp[static_cast<size_t>(o) * K + kk] =
            c < C ? w[(static_cast<size_t>(o) * C + c) * (kh * kw) + tap] : T();
    }
}

constexpr int SIMT_BM = 64;    // output pixels per CTA
constexpr int SIMT_BN = 64;    // output channels per CTA
constexpr int SIMT_BK = 16;    // channels per inner step
constexpr int SIMT_THREADS = 256;

template <typename T>
__global__ void __launch_bounds__(SIMT_THREADS)
dcn_simt_kernel(Params p) {
    __shared__ float As[SIMT_BK][SIMT_BM + 4];
    __shared__ float Bs[SIMT_BK][SIMT_BN + 4];
    __shared__ float4 cw_s[SIMT_BM];
    __shared__ int4 ci_s[SIMT_BM];

    const T *__restrict__ x = static_cast<const T *>(p.x);
    const T *__restrict__ wp = static_cast<const T *>(p.wpack);
    const int tid = threadIdx.x;
    const int pix0 = blockIdx.x * SIMT_BM;
    const int o0 = blockIdx.y * SIMT_BN;
    const int ty = tid / 16;   // pixel group: pixels ty*4 .. ty*4+3
    const int tx = tid % 16;   // channel group: outputs tx*4 .. tx*4+3
    const int HoWo = p.Ho * p.Wo;
    const int taps = p.kh * p.kw;
    const int Cg = p.C / p.groups;     // input channels per weight group
    const int Og = p.O / p.groups;     // output channels per weight group
    const int Cq = p.C / p.ogroups;    // channels per offset group
    // the channels this block's outputs contract over: their weight groups
    const int o_last = min(o0 + SIMT_BN, p.O) - 1;
    const int c_lo = (o0 / Og) * Cg;
    const int c_hi = (o_last / Og + 1) * Cg;

    // the pixel whose corner weights this thread computes (tid < SIMT_BM)
    const int my_pix = pix0 + tid;
    int my_b = 0, my_h = 0, my_w = 0;
    if (tid < SIMT_BM && my_pix < p.P) {
        my_b = my_pix / HoWo;
        const int rem = my_pix - my_b * HoWo;
        my_h = rem / p.Wo;
        my_w = rem - my_h * p.Wo;
    }

    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;

    for (int tap = 0; tap < taps; ++tap) {
        const int i = tap / p.kw;
        const int j = tap - i * p.kw;
        // the block's channels, one offset group at a time (each has its
        // own offsets and mask, so its own corner table)
        for (int q = c_lo / Cq; q * Cq < c_hi; ++q) {
            const int cq_lo = max(c_lo, q * Cq);
            const int cq_hi = min(c_hi, (q + 1) * Cq);
            __syncthreads();  // the previous corner table is no longer read
            if (tid < SIMT_BM) {
                TapCorners t;
                if (my_pix < p.P) {
                    const size_t hw = static_cast<size_t>(my_h) * p.Wo + my_w;
                    const size_t bq = static_cast<size_t>(my_b) * p.ogroups + q;
                    const size_t plane = static_cast<size_t>(p.plane);
                    const size_t ob = bq * 2 * taps * plane + hw;
                    const float dy = DCN_READ(p.offset, ob + static_cast<size_t>(2 * tap) * plane, p.off_lo, p.off_hi);
                    const float dx = DCN_READ(p.offset, ob + static_cast<size_t>(2 * tap + 1) * plane, p.off_lo, p.off_hi);
                    const float m = p.mask ? DCN_READ(p.mask, (bq * taps + tap) * plane + hw, p.mask_lo, p.mask_hi) : 1.0f;
                    tap_corners(dy, dx, m, (p.h0 + my_h) * p.sh - p.ph + i * p.dh, my_w * p.sw - p.pw + j * p.dw,
                                my_b, p.H, p.W, p.x_cstride, t);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) { t.w[e] = 0.0f; t.idx[e] = 0; }
                }
                cw_s[tid] = make_float4(t.w[0], t.w[1], t.w[2], t.w[3]);
                ci_s[tid] = make_int4(t.idx[0], t.idx[1], t.idx[2], t.idx[3]);
            }
            __syncthreads();

            for (int c0 = cq_lo; c0 < cq_hi; c0 += SIMT_BK) {
                // sampled operand: 16 channels x 64 pixels; consecutive threads
                // take consecutive channels of one pixel (coalesced in NHWC)
#pragma unroll
                for (int e = 0; e < (SIMT_BK * SIMT_BM) / SIMT_THREADS; ++e) {
                    const int idx = tid + e * SIMT_THREADS;
                    const int kk = idx % SIMT_BK;
                    const int pp = idx / SIMT_BK;
                    const int c = c0 + kk;
                    float v = 0.0f;
                    if (c < cq_hi) {
                        const float4 cw = cw_s[pp];
                        const int4 ci = ci_s[pp];
                        if (cw.x != 0.0f) v += cw.x * to_f32<T>(DCN_READ(x, ci.x + c, p.x_lo, p.x_hi));
                        if (cw.y != 0.0f) v += cw.y * to_f32<T>(DCN_READ(x, ci.y + c, p.x_lo, p.x_hi));
                        if (cw.z != 0.0f) v += cw.z * to_f32<T>(DCN_READ(x, ci.z + c, p.x_lo, p.x_hi));
                        if (cw.w != 0.0f) v += cw.w * to_f32<T>(DCN_READ(x, ci.w + c, p.x_lo, p.x_hi));
                    }
                    As[kk][pp] = v;
                }
                // weight tile: 16 channels x 64 outputs; an output's weight is
                // 0 for channels outside its group
#pragma unroll
                for (int e = 0; e < (SIMT_BK * SIMT_BN) / SIMT_THREADS; ++e) {
                    const int idx = tid + e * SIMT_THREADS;
                    const int kk = idx % SIMT_BK;
                    const int oo = idx / SIMT_BK;
                    const int c = c0 + kk;
                    const int o = o0 + oo;
                    float v = 0.0f;
                    if (c < cq_hi && o < p.O) {
                        const int cl = c - (o / Og) * Cg;   // channel within the output's group
                        if (cl >= 0 && cl < Cg) {
                            const int cp = p.wperm ? tc_channel_perm(cl) : cl;   // packed position
                            v = to_f32<T>(wp[static_cast<size_t>(o) * p.K + static_cast<size_t>(tap) * p.kc + cp]);
                        }
                    }
                    Bs[kk][oo] = v;
                }
                __syncthreads();
#pragma unroll
                for (int kk = 0; kk < SIMT_BK; ++kk) {
                    float a[4], b[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) a[r] = As[kk][ty * 4 + r];
#pragma unroll
                    for (int r = 0; r < 4; ++r) b[r] = Bs[kk][tx * 4 + r];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int s = 0; s < 4; ++s) acc[r][s] = fmaf(a[r], b[s], acc[r][s]);
                }
                __syncthreads();
            }
        }
    }

    // S5 epilogue: bias in fp32, cast, channels-last store
    T *__restrict__ out = static_cast<T *>(p.out);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int pix = pix0 + ty * 4 + r;
        if (pix >= p.P) continue;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int o = o0 + tx * 4 + s;
            if (o >= p.O) continue;
            const float bv = p.bias ? p.bias[o] : 0.0f;
            T *dst = out + static_cast<size_t>(pix) * p.out_stride + o;
#ifdef DCN_CHECK_BOUNDS
            if (!in_bounds(dst, sizeof(T), p.out_lo, p.out_hi, p.status)) continue;
#endif
            *dst = from_f32<T>(acc[r][s] + bv);
        }
    }
}

}  // namespace

cudaError_t launch_pack_weight(const void *weight, void *wpack, int O, int C, int kh, int kw,
                               int dtype, int perm, cudaStream_t stream) {
    // C: the weight's channel count, C_in / groups
    if (perm && C % 16 != 0) return cudaErrorInvalidValue;
    const int K = kh * kw * pack_kc(C, perm);
    const int threads = 256;
    const dim3 grid((K + threads - 1) / threads, O < 65535 ? O : 65535);
    if (dtype == kF32) {
        pack_weight_kernel<float><<<grid, threads, 0, stream>>>(
            static_cast<const float *>(weight), static_cast<float *>(wpack), O, C, kh, kw, perm);
    } else {
        // bf16 and fp16: the permutation moves 16-bit words
        pack_weight_kernel<uint16_t><<<grid, threads, 0, stream>>>(
            static_cast<const uint16_t *>(weight), static_cast<uint16_t *>(wpack),
            O, C, kh, kw, perm);
    }
    return cudaGetLastError();
}

cudaError_t launch_simt(const Params &p, int dtype, cudaStream_t stream) {
    dim3 grid((p.P + SIMT_BM - 1) / SIMT_BM, (p.O + SIMT_BN - 1) / SIMT_BN);
    if (dtype == kF32)
        dcn_simt_kernel<float><<<grid, SIMT_THREADS, 0, stream>>>(p);
    else if (dtype == kF16)
        dcn_simt_kernel<__half><<<grid, SIMT_THREADS, 0, stream>>>(p);
    else
        dcn_simt_kernel<__nv_bfloat16><<<grid, SIMT_THREADS, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dcn
