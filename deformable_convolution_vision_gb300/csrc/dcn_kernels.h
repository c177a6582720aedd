// Internal interface between the C ABI (dcn_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace dcn {

// Everything a forward kernel needs, passed by value.  Device pointers.
struct Params {
    const void *x;        // [B, H, W, C] channels-last
    const float *offset;  // [B, 2*kh*kw, Ho, Wo]
    const float *mask;    // [B, kh*kw, Ho, Wo] or nullptr
    const void *wpack;    // [O][kh*kw*C], tap-major / channel-minor (see wperm)
    const float *bias;    // [O] or nullptr
    void *out;            // [B, Ho, Wo, O] channels-last
    int B, C, H, W, O, kh, kw, pad, Ho, Wo;
    int P;                // B * Ho * Wo output pixels
    int K;                // kh * kw * C
    unsigned *status;     // device status word (timeout bit)
    unsigned long long timeout_ns;  // bound of every barrier wait
    int sample_f32;       // tensor-core path: 1 = fp32 bilinear combine, 0 = bf16
    // tensor-core path, stream-K scheduling (partial == nullptr: one tile per CTA)
    float *partial;       // fp32 partial tiles, one [O/16][128][16] slot per CTA
    unsigned *flags;      // one word per CTA: set to `epoch` once its partial is stored
    unsigned epoch;       // this launch's flag value (never 0)
    int sm_count;         // SMs of the device
    int units_per_cta;    // set by the launcher
    int wperm;            // 1: wpack's channels are in tc_channel_perm order
};

// Channel order of the tensor-core operand inside each 64-channel block:
// the bit fields c[2:3] and c[4:5] swapped.  Packed-weight position c holds
// channel tc_channel_perm(c); the map is its own inverse.  It matches the
// order in which the samplers' 16x256b TMEM stores lay a 64-channel row
// into 32 columns (thread quarter j holds channels 16j .. 16j+15 and writes
// them to columns 2j, 2j+1, 8+2j, 9+2j, ...).
__host__ __device__ constexpr int tc_channel_perm(int c) {
    return (c & ~0x3C) | ((c & 0x0C) << 2) | ((c & 0x30) >> 2);
}

enum Dtype { kF32 = 0, kBF16 = 1 };

// S0: weight [O, C, kh, kw] -> packed [O][(i*kw + j)*C + c'], where
// c' = c, or c' = tc_channel_perm(c) with perm != 0 (C % 64 == 0 only).
cudaError_t launch_pack_weight(const void *weight, void *wpack, int O, int C, int kh, int kw,
                               int dtype, int perm, cudaStream_t stream);

// CUDA-core fused sample + contraction + epilogue (fp32 or bf16 operands).
cudaError_t launch_simt(const Params &p, int dtype, cudaStream_t stream);

// tcgen05 fused implicit GEMM (bf16 operands).  `wmap` is a 2-D tensor map
// over the packed bf16 weight, box {64, O}, 128-byte swizzle.
bool tc_supported(int C, int O);
// Whether a weight for this (dtype, C, O) is packed in tc_channel_perm order.
inline bool tc_pack_permuted(int dtype, int C, int O) { return dtype == kBF16 && tc_supported(C, O); }
cudaError_t launch_tc(const Params &p, const CUtensorMap &wmap, cudaStream_t stream);

// One-thread kernel whose barrier wait runs out after timeout_ns.
cudaError_t launch_selftest_timeout(unsigned *status, unsigned long long timeout_ns,
                                    cudaStream_t stream);

}  // namespace dcn
