// Declarations of the convolution's backward kernels: the CUDA-core path,
// the tensor-core column gradient with its scatter, and the tensor-core
// weight gradient.  Kept apart from dcn_kernels.h (the forward's kernels)
// so that the two build from separate declarations.
#pragma once

#include "dcn_kernels.h"

namespace dcn {

// Everything the backward kernels need (device pointers).  x, weight and
// grad_out are in the operand dtype; the gradients are fp32 and must be
// zero on entry (the kernels add into them).
struct BwdParams {
    const void *x;          // [B, H, W, C] channels-last
    const float *offset;    // [B, 2*ogroups*kh*kw, Ho, Wo]
    const float *mask;      // [B, ogroups*kh*kw, Ho, Wo] or nullptr (all ones)
    const void *weight;     // [O, C/groups, kh, kw]
    const void *grad_out;   // [B, Ho, Wo, O] channels-last
    float *grad_x;          // [B, H, W, C] channels-last
    float *grad_offset;     // like offset
    float *grad_mask;       // like mask, or nullptr (not wanted)
    float *grad_weight;     // like weight
    float *grad_bias;       // [O] or nullptr (not wanted)
    int B, C, H, W, O, kh, kw;
    int sh, sw, ph, pw, dh, dw;
    int groups, ogroups;
    int Ho, Wo, P;
    int sm_count;
    int gx_vec4;            // grad_x 16-byte aligned and C % 4 == 0
    int pix_run;            // set by the launcher
    // tensor-core column-gradient kernel only
    unsigned *status;       // device status word (timeout bit)
    unsigned long long timeout_ns;
    int f16;                // 1: fp16 operands, 0: bf16
#ifdef DCN_CHECK_BOUNDS
    // bounds-checked builds: the byte ranges of the tensors the tensor-core
    // backward kernels read and add into
    const void *x_lo, *x_hi, *off_lo, *off_hi, *mask_lo, *mask_hi;
    const void *gx_lo, *gx_hi, *goff_lo, *goff_hi, *gmask_lo, *gmask_hi, *gw_lo, *gw_hi;
#endif
};

// Channel order of the tensor-core backward's weight operand inside each
// 64-channel block: row n of the packed block holds channel
// 16 * ((n >> 1) & 3) + 2 * (n >> 3) + (n & 1).  With it the 16x256b TMEM
// load of the fp32 column gradient gives thread quarter j the channels
// 16j .. 16j+15 (columns 2j, 2j+1, 8+2j, 9+2j, ...).
__host__ __device__ constexpr int bwd_channel_perm(int n) {
    return (n & ~63) | (16 * ((n >> 1) & 3) + 2 * ((n >> 3) & 7) + (n & 1));
}

// weight [O, C, kh, kw] (16-bit) -> packed [kh*kw*C][O]: row tap*C + c'
// holds weight[:, c, i, j] with c' = bwd_channel_perm(c) inside each
// 64-channel block (C % 64 == 0).
cudaError_t launch_pack_weight_bwd(const void *weight, void *wpack_t, int O, int C, int kh,
                                   int kw, cudaStream_t stream);

// Whether the tensor-core column-gradient kernel takes the problem: 16-bit
// operands, one weight group, C % 64 == 0, channels per offset group a
// multiple of 64, O % 64 == 0 and O <= 256.
bool bwd_tc_supported(int C, int O, int groups, int offset_groups);

// grad_x, grad_offset and grad_mask on tensor cores: the column gradient
// of a 128-pixel tile (grad_out tile via `gmap`, a 4-D tensor map over
// grad_out [B][Ho][Wo][O], box {64, 16, 8, 1}) against the packed weight
// of each (tap, 64-channel block) (via `wmap`, 2-D over [kh*kw*C][O], box
// {64, 64}), fp32 in tensor memory, then the bilinear scatter and sums.
cudaError_t launch_bwd_data_tc(const BwdParams &p, const CUtensorMap &gmap,
                               const CUtensorMap &wmap, cudaStream_t stream);
// grad_weight and grad_bias on CUDA cores (the second half of launch_backward).
cudaError_t launch_backward_weight(const BwdParams &p, int dtype, cudaStream_t stream);
// grad_weight on tensor cores (16-bit operands, one weight group, C and
// C/offset_groups multiples of 64, O a multiple of 64 up to 256): the
// sampled operand of each 128-pixel tile contracted with the grad_out tile
// (`gmap`, the column-gradient kernel's map) in shared memory, fp32 in
// tensor memory, added into grad_weight (which must be zeroed first).
// The grid is (row blocks of 128 (tap, channel) rows) x (pixel ranges), the
// ranges as many as p.sm_count allows (one at least).
cudaError_t launch_bwd_wgrad_tc(const BwdParams &p, const CUtensorMap &gmap, cudaStream_t stream);
int bwd_wgrad_row_blocks(const BwdParams &p);
// grad_bias alone (column sums of grad_out).
cudaError_t launch_bwd_bias(const BwdParams &p, int dtype, cudaStream_t stream);

// The backward pass: grad_x, grad_offset and grad_mask (one kernel),
// grad_weight (one kernel), grad_bias (one kernel, when wanted).
cudaError_t launch_backward(const BwdParams &p, int dtype, cudaStream_t stream);

}  // namespace dcn
