// Internal interface between the C ABI (dcn_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace dcn {

// Everything a forward kernel needs, passed by value.  Device pointers.
//
// The CUDA-core kernel reads the whole problem.  A tensor-core launch sees
// one weight group and one chunk of at most 256 of its output channels: C
// is then the group's channel count, O the chunk's output count, and the
// pointers are advanced to the group / chunk (x to its first channel,
// offset and mask to its first offset group, wpack, bias and out to its
// first output channel), with x_cstride and out_stride the full row
// strides.
struct Params {
    const void *x;        // [B, H, W, x_cstride] channels-last
    const float *offset;  // [B, 2*ogroups*kh*kw, Ho, Wo]
    const float *mask;    // [B, ogroups*kh*kw, Ho, Wo] or nullptr
    const void *wpack;    // [O][kh*kw*(C/groups)], tap-major / channel-minor (see wperm)
    const float *bias;    // [O] or nullptr
    void *out;            // [B, Ho, Wo, out_stride] channels-last
    int B, C, H, W, O, kh, kw;
    int sh, sw, ph, pw, dh, dw;  // stride, padding, dilation (h, w)
    int groups;           // weight groups (CUDA-core kernel; 1 in a tensor-core launch)
    int ogroups;          // offset groups (CUDA-core kernel)
    int Ho, Wo;           // output rows and columns of this launch
    int h0;               // absolute output row of the launch's first row (its
                          // sampling coordinates use h0 + row); 0 for a whole image
    int plane;            // elements between consecutive offset/mask planes:
                          // Ho * Wo, or the whole image's for a band of rows
    int P;                // B * Ho * Wo output pixels
    int K;                // packed weight row length: kh * kw * kc
    int kc;               // packed positions per tap: C / groups, or (tensor-core
                          // order) C / groups rounded up to a multiple of 64
    int x_cstride;        // elements between neighbouring pixels of x
    int out_stride;       // elements between neighbouring pixels of out
    // tensor-core launch view of the offset groups: og_count groups of
    // C / og_count channels each, from the first one the pointers address;
    // batch strides of offset and mask in planes (2*ogroups*kh*kw, ogroups*kh*kw)
    int og_count;
    int off_bstride, mask_bstride;
    unsigned *status;     // device status word (timeout bit)
    unsigned long long timeout_ns;  // bound of every barrier wait
#ifdef DCN_CHECK_BOUNDS
    // bounds-checked builds: the byte ranges of the caller's tensors
    const void *x_lo, *x_hi, *off_lo, *off_hi, *mask_lo, *mask_hi, *out_lo, *out_hi;
#endif
    int sample_f32;       // tensor-core path: 1 = fp32 bilinear combine, 0 = operand type
    int f16;              // tensor-core path: 1 = fp16 operands, 0 = bf16
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

enum Dtype { kF32 = 0, kBF16 = 1, kF16 = 2 };

// S0: weight [O, Cg, kh, kw] -> packed [O][(i*kw + j)*kc + pos].  perm == 0:
// kc = Cg and position pos holds channel pos.  perm != 0 (the tensor-core
// operand order, Cg % 16 == 0): kc = Cg rounded up to a multiple of 64,
// position pos holds channel tc_channel_perm(pos), and zero where that is
// >= Cg (the padding of a tap's last 64-channel block).
cudaError_t launch_pack_weight(const void *weight, void *wpack, int O, int Cg, int kh, int kw,
                               int dtype, int perm, cudaStream_t stream);
#ifdef DCN_CHECK_BOUNDS
// Bounds-checked builds: the byte ranges of the tensors a forward launch
// reads and writes, from its (possibly banded) view.
inline void set_bounds(Params &p, size_t es) {
    const char *x = static_cast<const char *>(p.x);
    p.x_lo = x;
    p.x_hi = x + static_cast<size_t>(p.B) * p.H * p.W * p.x_cstride * es;
    const size_t img = static_cast<size_t>(p.Ho) * p.Wo;   // one plane's pixels in this view
    const size_t plane = static_cast<size_t>(p.plane);
    p.off_lo = p.offset;
    p.off_hi = p.offset + (static_cast<size_t>(p.B) * p.off_bstride - 1) * plane + img;
    p.mask_lo = p.mask;
    p.mask_hi = p.mask ? p.mask + (static_cast<size_t>(p.B) * p.mask_bstride - 1) * plane + img : nullptr;
    char *out = static_cast<char *>(p.out);
    p.out_lo = out;
    p.out_hi = out + static_cast<size_t>(p.B) * img * p.out_stride * es;
}
#endif

// Packed positions per tap for a pack of Cg channels.
__host__ __device__ inline int pack_kc(int Cg, int perm) { return perm ? (Cg + 63) / 64 * 64 : Cg; }

// CUDA-core fused sample + contraction + epilogue (fp32, bf16 or fp16 operands).
cudaError_t launch_simt(const Params &p, int dtype, cudaStream_t stream);

// tcgen05 fused implicit GEMM (bf16 or fp16 operands, Params::f16), one
// launch = one weight group x one chunk of its output channels (see
// Params).  `wmap` is a 2-D tensor map over the chunk's rows of the packed
// 16-bit weight, box {64, O}, 128-byte swizzle.
//   tc_supported: the channel and output counts of one launch;
//   tc_max_virtual_taps: bound on kh*kw*og_count (a per-CTA table).
bool tc_supported(int C, int O);
constexpr int tc_max_virtual_taps = 512;
// Whether a weight whose groups have Cg channels is packed in
// tc_channel_perm order (a 16-bit type, Cg a multiple of 16).
inline bool tc_pack_permuted(int dtype, int Cg) { return (dtype == kBF16 || dtype == kF16) && Cg % 16 == 0; }
// after_pack: the launch directly follows this call's launch_pack_weight on
// the same stream.  It is then a programmatic dependent launch: the CTAs
// start while the pack runs (the pack lets them launch at once) and only the
// weight loads wait for the pack to finish (griddepcontrol.wait); x, offset
// and mask were complete before the pack started.
cudaError_t launch_tc(const Params &p, const CUtensorMap &wmap, cudaStream_t stream,
                      bool after_pack = false);

// Batched 2-D transpose [B][R][S] -> [B][S][R] of 2- or 4-byte elements.
cudaError_t launch_transpose(const void *src, void *dst, int B, int R, int S, int esize,
                             cudaStream_t stream);

// One-thread kernel whose barrier wait runs out after timeout_ns.
cudaError_t launch_selftest_timeout(unsigned *status, unsigned long long timeout_ns,
                                    cudaStream_t stream);

}  // namespace dcn
