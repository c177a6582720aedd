// Declarations of the CUDA-core sampling operators that share the
// deformable convolution's bilinear sampler: multi-scale deformable
// attention and single-scale deformable sampling, forward and backward.
// Kept apart from dcn_kernels.h (the convolution's kernels) so that the two
// families build from separate declarations.
#pragma once

#include "dcn_kernels.h"

namespace dcn {

// Multi-scale deformable attention forward (device pointers; the level
// table by value).
constexpr int kMsdaMaxLevels = 8;
struct MsdaParams {
    const void *value;        // [B, S, G, D], the operand dtype
    const float *locations;   // [B, Q, G, L, K, 2], normalized (x, y)
    const float *weights;     // [B, Q, G, L*K]
    void *out;                // [B, Q, G, D], the operand dtype
    int B, S, G, D, Q, K, L;
    int softmax;              // 1: normalize the weights over L*K
    int H[kMsdaMaxLevels], W[kMsdaMaxLevels], start[kMsdaMaxLevels];
#ifdef DCN_CHECK_BOUNDS
    // bounds-checked builds: the byte ranges of the tensors the corner rows
    // are read from (and reduced into)
    const void *v_lo, *v_hi;
    const void *gv_lo, *gv_hi;
#endif
};
// vec: D a multiple of 8 (16-bit) or 4 (fp32) and value/out 16-byte aligned.
cudaError_t launch_msda(const MsdaParams &p, int dtype, bool vec, cudaStream_t stream);

// MSDA backward: the forward's operands plus the cotangent, fp32 gradients.
// grad_value must be zero on entry (the kernel accumulates into it).
struct MsdaBwdParams {
    const void *value;        // [B, S, G, D], the operand dtype
    const float *locations;   // [B, Q, G, L, K, 2]
    const float *weights;     // [B, Q, G, L*K]
    const void *grad_out;     // [B, Q, G, D], the operand dtype
    float *grad_value;        // [B, S, G, D]
    float *grad_locations;    // [B, Q, G, L, K, 2]
    float *grad_weights;      // [B, Q, G, L*K]
    int B, S, G, D, Q, K, L;
    int softmax;
    int H[kMsdaMaxLevels], W[kMsdaMaxLevels], start[kMsdaMaxLevels];
#ifdef DCN_CHECK_BOUNDS
    // bounds-checked builds: the byte ranges of the tensors the corner rows
    // are read from (and reduced into)
    const void *v_lo, *v_hi;
    const void *gv_lo, *gv_hi;
#endif
};
// vec: D a multiple of 8 (16-bit) or 4 (fp32); value, grad_out and
// grad_value 16-byte aligned.
cudaError_t launch_msda_backward(const MsdaBwdParams &p, int dtype, bool vec, cudaStream_t stream);

// Single-scale deformable sampling (DCNv3), forward.
struct AttnParams {
    const void *value;        // [B, H, W, G, D], the operand dtype
    const float *offsets;     // [B, Ho, Wo, G, K, 2], (dy, dx), 8-byte aligned
    const float *weights;     // [B, Ho, Wo, G, K]
    void *out;                // [B, Ho, Wo, G, D], the operand dtype
    int B, H, W, G, D, Ho, Wo;
    int kh, kw, sh, sw, ph, pw, dh, dw;
    int softmax;              // 1: normalize the weights over the K taps
#ifdef DCN_CHECK_BOUNDS
    // bounds-checked builds: the byte ranges of the tensors the corner rows
    // are read from (and reduced into)
    const void *v_lo, *v_hi;
    const void *gv_lo, *gv_hi;
#endif
};
// vec: D a multiple of 8 (16-bit) or 4 (fp32) and value/out 16-byte aligned.
cudaError_t launch_attn(const AttnParams &p, int dtype, bool vec, cudaStream_t stream);

// Its backward: fp32 gradients; grad_value must be zero on entry.
struct AttnBwdParams {
    const void *value;        // [B, H, W, G, D], the operand dtype
    const float *offsets;     // [B, Ho, Wo, G, K, 2]
    const float *weights;     // [B, Ho, Wo, G, K]
    const void *grad_out;     // [B, Ho, Wo, G, D], the operand dtype
    float *grad_value;        // [B, H, W, G, D]
    float *grad_offsets;      // [B, Ho, Wo, G, K, 2], 8-byte aligned
    float *grad_weights;      // [B, Ho, Wo, G, K]
    int B, H, W, G, D, Ho, Wo;
    int kh, kw, sh, sw, ph, pw, dh, dw;
    int softmax;
#ifdef DCN_CHECK_BOUNDS
    // bounds-checked builds: the byte ranges of the tensors the corner rows
    // are read from (and reduced into)
    const void *v_lo, *v_hi;
    const void *gv_lo, *gv_hi;
#endif
};
// vec: D a multiple of 4; value and grad_out 8-byte (16-bit) or 16-byte
// (fp32) aligned, grad_value 16-byte aligned.
cudaError_t launch_attn_backward(const AttnBwdParams &p, int dtype, bool vec, cudaStream_t stream);

}  // namespace dcn
