/*
 * dcn.h -- C ABI of the GB300 (sm_103a) deformable sampling library: the
 * modulated deformable convolution forward pass (below; its general form,
 * dcn_forward_ex, further down), its backward, multi-scale deformable
 * attention and single-scale deformable sampling (forward and backward),
 * and NCHW/NHWC layout copies.  Each function states its own operation.
 *
 * The convolution (page "litert-community/Idol ... deform_conv.py", module
 * docstring and the four-corner loop of deform_conv2d_gather; page
 * "deformops 3.0.1", section "Deformable convolution"): torchvision
 * deform_conv2d with stride 1, dilation 1, one offset group and one weight
 * group.  For image b, output channel o and output pixel (h, w):
 *
 *   out[b,h,w,o] = bias[o] + sum_{i,j,c} weight[o,c,i,j] * m * S(b,c,py,px)
 *   k = i*kw + j,  dy = offset[b,2k,h,w],  dx = offset[b,2k+1,h,w],
 *   m = mask[b,k,h,w] (1 without a mask),
 *   py = (h - pad + i) + dy,  px = (w - pad + j) + dx   (fp32),
 *   S  = bilinear sample of channel c at (py, px); each of the four corners
 *        that falls outside [0,H-1] x [0,W-1] contributes 0.
 *
 *   Ho = H + 2*pad - kh + 1,  Wo = W + 2*pad - kw + 1.
 *
 * Layouts (dense, no padding between rows; all pointers are DEVICE pointers
 * unless the function name ends in _host):
 *   x      [B, H, W, C]       channels-last, element type `dtype`
 *   offset [B, 2*kh*kw, Ho, Wo] fp32; channel 2k holds dy_k, 2k+1 holds dx_k
 *   mask   [B, kh*kw, Ho, Wo] fp32, or NULL for "all ones" (DCN v1)
 *   weight [O, C, kh, kw]     element type `dtype` (torchvision layout)
 *   bias   [O]                fp32, or NULL for zero
 *   out    [B, Ho, Wo, O]     channels-last, element type `dtype`
 *
 * Numerics: sampling coordinates and corner weights are fp32.  The bilinear
 * combine of the four corners runs in the input dtype by default, as the
 * page's own gather decomposition does (its corner weights and sums are in
 * x.dtype): for bf16 (fp16) the weights are rounded to bf16 (fp16) and
 * each fused multiply-add rounds once to that type; dcn_set_sample_precision
 * selects an fp32 combine instead.  The contraction accumulates in fp32 for
 * every dtype (no TF32).  The 16-bit paths round each interpolated sample to
 * the operand type before the tensor-core contraction and round the fp32
 * result (after bias) to it at the end.  fp16 has the narrower range: the
 * caller keeps inputs, samples and outputs inside it (|v| < 65504).
 *
 * Ownership: the caller owns every tensor and the stream.  A handle owns a
 * small device workspace (the packed weight, a status word and, for
 * dcn_forward_host, device staging buffers) that grows on demand, in stream
 * order, and is released by dcn_destroy.  Calls that share a handle must be
 * ordered on one stream; use one handle per stream for concurrent streams.
 *
 * Errors: every function validates its arguments before launching anything
 * and returns a dcn_status_t; a failed check launches nothing.  Launches are
 * asynchronous; a device-side failure (a bounded wait that ran out) sets the
 * handle's status word, which dcn_sync_status reports.
 */
#ifndef DCN_H
#define DCN_H

#if defined(__GNUC__)
#define DCN_API __attribute__((visibility("default")))
#else
#define DCN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dcn_handle_s *dcn_handle_t;

/* Element type of x, weight and out. */
typedef enum {
    DCN_F32 = 0,   /* fp32 operands, CUDA-core FFMA path */
    DCN_BF16 = 1,  /* bf16 operands, tcgen05 tensor-core path where the shape allows */
    DCN_F16 = 2    /* fp16 operands, the same paths as bf16 (tcgen05 kind::f16 with fp16 A and B) */
} dcn_dtype_t;

typedef enum {
    DCN_OK = 0,
    DCN_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, misaligned pointer, size overflow */
    DCN_ERR_UNSUPPORTED = 2,  /* a forced path that cannot run this shape, or a device that is not sm_103 */
    DCN_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    DCN_ERR_NO_DEVICE = 4,    /* no CUDA device is visible */
    DCN_ERR_OOM = 5,          /* workspace allocation failed */
    DCN_ERR_TIMEOUT = 6,      /* a device-side bounded wait ran out (reported by dcn_sync_status) */
    DCN_ERR_BOUNDS = 7        /* a bounds-checked build (compiled with DCN_CHECK_BOUNDS) skipped a
                                 forward read or write outside the caller's tensors (reported by
                                 dcn_sync_status); the ordinary build never reports it */
} dcn_status_t;

/* Kernel selection for bf16 and fp16.  AUTO takes the tcgen05 path when
 * C % 16 == 0, O % 16 == 0, 16 <= O <= 256, x is 32-byte aligned and out is
 * 16-byte aligned, and the CUDA-core path otherwise.  The tensor-core kernel
 * contracts 64 channels at a time; when C % 64 != 0 it completes each
 * tap's last block with zeros.  fp32 always takes the
 * CUDA-core path.  (dcn_forward_ex states its own conditions.) */
typedef enum {
    DCN_PATH_AUTO = 0,
    DCN_PATH_SIMT = 1,   /* CUDA-core fused sample + FFMA contraction */
    DCN_PATH_TC = 2      /* tcgen05 fused implicit GEMM (bf16 or fp16) */
} dcn_path_t;

/* Create a handle on the current CUDA device.  Returns DCN_ERR_NO_DEVICE
 * without a device and DCN_ERR_UNSUPPORTED on a device other than compute
 * capability 10.3.  *out_handle is NULL on failure. */
DCN_API dcn_status_t dcn_create(dcn_handle_t *out_handle);

/* Release the handle and its workspace.  Synchronises the device first.
 * NULL is accepted and ignored. */
DCN_API dcn_status_t dcn_destroy(dcn_handle_t h);

/* Full forward pass on `stream` (a cudaStream_t; NULL = legacy default
 * stream): packs the weight into the handle's workspace, then runs the
 * fused sampling + contraction + epilogue kernel.  Asynchronous.
 * x, weight and out must be aligned to their element size, offset, mask
 * and bias to 4 bytes.  Sizes: every dimension > 0, pad >= 0, Ho > 0,
 * Wo > 0, and each of B*H*W*C, B*2*kh*kw*Ho*Wo, B*Ho*Wo*O, O*C*kh*kw
 * below 2^31. */
DCN_API dcn_status_t dcn_forward(dcn_handle_t h,
                         const void *x, const float *offset, const float *mask,
                         const void *weight, const float *bias, void *out,
                         int B, int C, int H, int W, int O,
                         int kh, int kw, int pad, int dtype, void *stream);

/* The two halves of dcn_forward, for callers that reuse one weight.
 * dcn_pack_weight reorders weight [O,C,kh,kw] into the handle's workspace
 * as [O][(i*kw + j)*C + c] (tap-major, channel-minor).  For bf16 and fp16
 * shapes with C % 16 == 0, the channels inside each 64-channel block are in
 * the tensor-core kernel's operand order instead and each tap is padded
 * with zeros to a whole number of blocks; the workspace is
 * private to the handle and either kernel reads it correctly.
 * dcn_forward_packed then runs the fused kernel with that packed weight;
 * it returns DCN_ERR_INVALID_ARG if (O, C, kh, kw, dtype) differ from the
 * last dcn_pack_weight on this handle.  Both are asynchronous on `stream`. */
DCN_API dcn_status_t dcn_pack_weight(dcn_handle_t h, const void *weight,
                             int O, int C, int kh, int kw, int dtype, void *stream);
DCN_API dcn_status_t dcn_forward_packed(dcn_handle_t h,
                                const void *x, const float *offset, const float *mask,
                                const float *bias, void *out,
                                int B, int C, int H, int W, int O,
                                int kh, int kw, int pad, int dtype, void *stream);

/* dcn_forward with HOST buffers (same layouts): copies every input to
 * device staging buffers owned by the handle, runs the forward pass,
 * copies out back and synchronises `stream`.  It runs as a pipeline over
 * bands of output rows: uploads on `stream`, each band's kernel on a
 * handle-owned stream, downloads on another, so later uploads overlap
 * earlier bands' work; the call returns when all of it is done.  Pinned host memory gives
 * asynchronous copies; pageable memory works but is slower.  Returns the
 * device status as dcn_sync_status would. */
DCN_API dcn_status_t dcn_forward_host(dcn_handle_t h,
                              const void *x, const float *offset, const float *mask,
                              const void *weight, const float *bias, void *out,
                              int B, int C, int H, int W, int O,
                              int kh, int kw, int pad, int dtype, void *stream);

/* Precision of the bilinear combine on the 16-bit tensor-core path. */
typedef enum {
    DCN_SAMPLE_INPUT_DTYPE = 0,  /* default: weights and fused multiply-adds in the operand type */
    DCN_SAMPLE_F32 = 1           /* fp32 weights and fp32 sums, then one rounding to the operand type */
} dcn_sample_t;

/* Choose the combine precision (dcn_sample_t) for later calls on this
 * handle.  The fp32 operand path always combines in fp32. */
DCN_API dcn_status_t dcn_set_sample_precision(dcn_handle_t h, int mode);

/* Choose the kernel path for later calls on this handle (dcn_path_t).
 * A forced path that cannot run a given shape makes that call return
 * DCN_ERR_UNSUPPORTED. */
DCN_API dcn_status_t dcn_set_path(dcn_handle_t h, int path);

/* The path (dcn_path_t, never AUTO) taken by the last successful forward
 * call on this handle, or -1 before the first. */
DCN_API int dcn_last_path(dcn_handle_t h);

/* Synchronise `stream` and report the handle's device status word:
 * DCN_OK, DCN_ERR_TIMEOUT if a kernel's bounded wait ran out (the word is
 * cleared after it is read), DCN_ERR_BOUNDS if a bounds-checked build
 * skipped an access outside the caller's tensors (this takes precedence;
 * the word is cleared likewise), or DCN_ERR_CUDA if the synchronisation
 * failed. */
DCN_API dcn_status_t dcn_sync_status(dcn_handle_t h, void *stream);

/* Launch a one-thread kernel that waits on a barrier nothing arrives on,
 * with a bound of timeout_ns nanoseconds; it then sets the status word
 * exactly as a stalled forward kernel would and returns.  Lets a caller
 * check the timeout path without stalling a real kernel.  timeout_ns must
 * be in (0, 10^10]. */
DCN_API dcn_status_t dcn_selftest_timeout(dcn_handle_t h, long long timeout_ns, void *stream);

/* Largest packed weight that dcn_forward_noalloc accepts: 8 MiB.  The
 * packed weight holds O*C'*kh*kw elements of the weight's type, where C' is
 * C rounded up to a multiple of 64 for bf16/fp16 with C % 16 == 0 (the
 * tensor-core operand order) and C otherwise. */
#define DCN_NOALLOC_MAX_WEIGHT_BYTES 8388608ull

/* dcn_forward without any device allocation.  The pages have no
 * counterpart: this exists for callers that must not let a library
 * allocate device memory -- plugin hosts and inference engines that own
 * all device memory and forbid allocations behind their back, processes
 * whose device-memory budget is fixed at start-up, and latency-critical
 * loops where cudaMalloc/cudaFree can synchronise the device and stall
 * other streams.
 *
 * It takes no handle and calls no cudaMalloc, cudaFree or other allocating
 * routine.  Its scratch (the packed weight and a status word) lives in
 * fixed device arrays built into the library, which every GPU that loads
 * the library holds until the process exits.  Same arguments, layouts,
 * kernels and results as dcn_forward; asynchronous on `stream`.
 *
 * - The packed weight must fit DCN_NOALLOC_MAX_WEIGHT_BYTES; larger
 *   weights return DCN_ERR_UNSUPPORTED and launch nothing.  Other argument
 *   errors return DCN_ERR_INVALID_ARG as for dcn_forward.
 * - The first call on each device looks up the scratch arrays' device
 *   addresses (cudaGetSymbolAddress) with that device current; make that
 *   first call before any stream capture.
 * - Every call on a device shares the same scratch, which keeps the last
 *   call's contents: calls whose work overlaps on the GPU (on different
 *   streams, or from different threads) race and may corrupt each other's
 *   results.  Order them on one stream.
 * - The status word is cleared at the start of each call; a device-side
 *   wait that runs out is not reported back by this entry point. */
DCN_API dcn_status_t dcn_forward_noalloc(const void *x, const float *offset, const float *mask,
                                         const void *weight, const float *bias, void *out,
                                         int B, int C, int H, int W, int O,
                                         int kh, int kw, int pad, int dtype, void *stream);

/* Static, human-readable name of a status code. */
DCN_API const char *dcn_status_string(dcn_status_t s);

/* ------------------------------------------------------------------ general
 * The general form: stride, per-axis padding, dilation, weight groups and
 * offset (deformable) groups.  The pages fix stride 1, dilation 1, one
 * padding and one group for their routine; the "deformops 3.0.1" page
 * (section "Deformable convolution") names torchvision deform_conv2d, with
 * a (C_out, C_in / groups, kH, kW) weight, as the operator, and these are
 * the convolution reading of its parameters.  With G = offset_groups and
 * Cq = C / G, output channel o in weight group g = o / (O / groups):
 *
 *   out[b,h,w,o] = bias[o] + sum_{i,j} sum_{c in group g}
 *                  weight[o, c - g*C/groups, i, j] * m * S(b,c,py,px)
 *   q  = c / Cq (the channel's offset group),
 *   dy = offset[b, 2*kh*kw*q + 2k, h, w], dx = offset[b, 2*kh*kw*q + 2k+1, h, w],
 *   m  = mask[b, kh*kw*q + k, h, w],
 *   py = (h*stride_h - pad_h + i*dil_h) + dy,  px = (w*stride_w - pad_w + j*dil_w) + dx,
 *   Ho = (H + 2*pad_h - dil_h*(kh-1) - 1) / stride_h + 1, likewise Wo.
 *
 * Layouts: x [B,H,W,C] and out [B,Ho,Wo,O] channels-last as above; offset
 * [B, 2*G*kh*kw, Ho, Wo] and mask [B, G*kh*kw, Ho, Wo], each offset group's
 * planes laid out like the one-group planes, one group after another;
 * weight [O, C/groups, kh, kw]. */
typedef struct {
    int B, C, H, W;        /* input x [B, H, W, C] */
    int O, kh, kw;         /* weight [O, C / groups, kh, kw] */
    int stride_h, stride_w;  /* >= 1 */
    int pad_h, pad_w;        /* >= 0, zero padding on both sides of each axis */
    int dil_h, dil_w;        /* >= 1 */
    int groups;              /* weight groups: divides C and O */
    int offset_groups;       /* offset groups: divides C */
} dcn_conv_desc_t;

/* Output size of one axis: (n + 2*pad - dil*(k-1) - 1) / stride + 1, or 0
 * if the kernel does not fit. */
DCN_API int dcn_out_size(int n, int k, int stride, int pad, int dil);

/* dcn_forward for the general form.  Argument rules as dcn_forward, plus
 * the descriptor's (its fields as commented; every size product below
 * 2^31).  AUTO takes the tcgen05 path for bf16 and fp16 when, with Cg = C/groups,
 * Og = O/groups, Cq = C/offset_groups: Cg % 16 == 0, one of Cg and Cq
 * divides the other, Cq % 64 == 0 when Cq < Cg (several offset groups in
 * one weight group), Og % 16 == 0, kh*kw*max(1, Cg/Cq) <= 512,
 * x is 32-byte and out 16-byte aligned; it runs one launch per weight group
 * and per 256 output channels.  Otherwise the CUDA-core path runs.  NULL
 * desc: DCN_ERR_INVALID_ARG. */
DCN_API dcn_status_t dcn_forward_ex(dcn_handle_t h,
                            const void *x, const float *offset, const float *mask,
                            const void *weight, const float *bias, void *out,
                            const dcn_conv_desc_t *desc, int dtype, void *stream);

/* The two halves of dcn_forward_ex: the pack keys on (O, C/groups, kh, kw,
 * dtype) of desc; dcn_forward_packed_ex returns DCN_ERR_INVALID_ARG when
 * they differ from the last pack on this handle. */
DCN_API dcn_status_t dcn_pack_weight_ex(dcn_handle_t h, const void *weight,
                                const dcn_conv_desc_t *desc, int dtype, void *stream);
DCN_API dcn_status_t dcn_forward_packed_ex(dcn_handle_t h,
                                   const void *x, const float *offset, const float *mask,
                                   const float *bias, void *out,
                                   const dcn_conv_desc_t *desc, int dtype, void *stream);

/* ------------------------------------------------------------ backward
 *
 * The gradients of the forward pass with respect to x, offset, mask, weight
 * and bias, given grad_out (the cotangent of out).  They follow from the
 * forward's definition by the chain rule; the page "deformops 3.0.1"
 * (section "Deformable convolution") keeps fp32 accumulation and no TF32 in
 * them.  With gA = sum over the outputs o of channel c's weight group of
 * grad_out[p,o] * weight[o, c - c0, i, j], for each output pixel p, tap
 * (i, j) and channel c:
 *   grad_x at each inside corner    += gA * m * wy * wx
 *   grad_offset (dy, dx)            += gA * m * (dS/dpy, dS/dpx)
 *   grad_mask                       += gA * S
 *   grad_weight[o, c - c0, i, j]    += grad_out[p,o] * m * S
 *   grad_bias[o]                    += grad_out[p,o]
 * where S is the bilinear sample and wy, wx its corner weights.  The
 * corner weights are piecewise linear in the coordinate; at an integer
 * coordinate the derivative is the one of the cell floor() selects.
 *
 * Layouts (device pointers, dense):
 *   x        [B, H, W, C]          channels-last, `dtype`
 *   offset   [B, 2*G*kh*kw, Ho, Wo] fp32     (G = offset groups)
 *   mask     [B, G*kh*kw, Ho, Wo]  fp32, or NULL (all ones)
 *   weight   [O, C/groups, kh, kw] `dtype`
 *   grad_out [B, Ho, Wo, O]        channels-last, `dtype`
 *   grad_x   [B, H, W, C]          fp32, channels-last
 *   grad_offset like offset, fp32
 *   grad_mask   like mask, fp32, or NULL (not computed; with mask NULL it is
 *               the gradient at mask = 1)
 *   grad_weight [O, C/groups, kh, kw] fp32
 *   grad_bias   [O] fp32, or NULL (not computed)
 * The gradients are overwritten (zeroed, then accumulated in fp32 with
 * atomic reductions, so the order of the sums, and the last bits, vary from
 * run to run).  Asynchronous on `stream`.
 * Kernels: with bf16/fp16 operands, one weight group, C and C/offset_groups
 * multiples of 64, O a multiple of 64 up to 256, x 32-byte and grad_out and
 * grad_x 16-byte aligned, the column gradient runs on tcgen05 tensor cores
 * (fp32 accumulators in tensor memory, never written to memory) fused with
 * the scatter into grad_x and the offset/mask sums; the handle then keeps a
 * [kh*kw*C][O] copy of the weight in its workspace (grown on demand, in
 * stream order).  Otherwise, and for fp32, CUDA cores run it and nothing is
 * allocated.  dcn_set_path(DCN_PATH_SIMT) forces the CUDA-core kernels;
 * DCN_PATH_TC returns DCN_ERR_UNSUPPORTED for shapes outside the envelope.
 * In the same envelope the weight gradient runs on tcgen05 too: each
 * 128-pixel tile of the sampled operand m * S (summed in fp32, rounded once
 * to the operand type) is contracted with the grad_out tile in shared
 * memory as soon as it is sampled, fp32 accumulation in tensor memory, no
 * TF32; the sampled operand is never written to memory.  When its blocks
 * of 128 (tap, channel) rows number at most a quarter of the SMs it runs
 * beside the column-gradient kernel, on a stream the handle owns that is
 * forked from `stream` and joined back into it (the call stays ordered on
 * `stream`; a handle is not used from two threads at once).  Otherwise a
 * CUDA-core kernel computes it in fp32.  The bias gradient runs on CUDA
 * cores.  Argument rules as
 * dcn_forward / dcn_forward_ex (sizes, NULL inputs, alignment to the
 * element size, 4 bytes for fp32 arrays); DCN_ERR_INVALID_ARG for a NULL x,
 * offset, weight, grad_out, grad_x, grad_offset or grad_weight. */
DCN_API dcn_status_t dcn_backward(dcn_handle_t h,
                          const void *x, const float *offset, const float *mask,
                          const void *weight, const void *grad_out,
                          float *grad_x, float *grad_offset, float *grad_mask,
                          float *grad_weight, float *grad_bias,
                          int B, int C, int H, int W, int O,
                          int kh, int kw, int pad, int dtype, void *stream);
DCN_API dcn_status_t dcn_backward_ex(dcn_handle_t h,
                             const void *x, const float *offset, const float *mask,
                             const void *weight, const void *grad_out,
                             float *grad_x, float *grad_offset, float *grad_mask,
                             float *grad_weight, float *grad_bias,
                             const dcn_conv_desc_t *desc, int dtype, void *stream);

/* ------------------------------------------------------------ layouts
 *
 * For callers with NCHW tensors (the torchvision layout that page
 * "deformops 3.0.1", section "torchvision drop-in", keeps for its drop-in
 * function): device-side layout copies between [B, C, H, W] and
 * [B, H, W, C] (the layout of x and out above), in `dtype`'s element size.
 * src and dst must not overlap.  Asynchronous on `stream`; allocates
 * nothing.  DCN_ERR_INVALID_ARG for NULL or equal pointers, non-positive or
 * oversized dimensions (B*C*H*W < 2^31), misalignment;
 * DCN_ERR_UNSUPPORTED for B > 65535. */
DCN_API dcn_status_t dcn_nchw_to_nhwc(const void *src, void *dst, int B, int C, int H, int W,
                              int dtype, void *stream);
DCN_API dcn_status_t dcn_nhwc_to_nchw(const void *src, void *dst, int B, int C, int H, int W,
                              int dtype, void *stream);

/* ------------------------------------------------ multi-scale deformable attention
 *
 * The forward pass of the operator of page "deformops 3.0.1", section
 * "Multi-scale deformable attention" (its functional form msda(value,
 * shapes, starts, locations, weights, method)), which shares the
 * deformable convolution's bilinear sampler.  B batch, G heads, D channels
 * per head, Q queries, L levels, K points per level:
 *
 *   out[b,q,g,d] = sum_{l,k} a[b,q,g,l,k] * S_l(b, g, d, py, px),
 *   px = loc[b,q,g,l,k,0] * W_l - 0.5,  py = loc[b,q,g,l,k,1] * H_l - 0.5,
 *
 * S_l the bilinear sample of level l (corners outside it contribute 0), a
 * the weights as given or, with softmax != 0, softmax-normalized over the
 * L*K entries of each (b, q, g).  The pages fix neither the coordinate axis
 * order nor the normalization; these are the Deformable DETR convention
 * ((x, y), pixel centres at (i + 0.5) / size).
 *
 * Layouts (device pointers, dense):
 *   value     [B, S, G, D]          `dtype`; level l occupies rows
 *                                   starts[l] .. + H_l*W_l (row y*W_l + x)
 *   locations [B, Q, G, L, K, 2]    fp32, 8-byte aligned
 *   weights   [B, Q, G, L*K]        fp32
 *   out       [B, Q, G, D]          `dtype`
 *   shapes    HOST int[L][2] = (H_l, W_l);  starts  HOST int[L]
 * Arithmetic in fp32 (coordinates, weights, softmax, sums), one rounding to
 * `dtype` at the end.  1 <= L <= 8 (else DCN_ERR_UNSUPPORTED); every level
 * inside [0, S).  Asynchronous on `stream`; allocates nothing; no handle. */
DCN_API dcn_status_t dcn_msda_forward(const void *value, const int *shapes, const int *starts,
                              int L, const float *locations, const float *weights, void *out,
                              int B, int S, int G, int D, int Q, int K, int softmax,
                              int dtype, void *stream);

/* The backward of dcn_msda_forward: for the cotangent grad_out [B, Q, G, D]
 * (`dtype`, like value), the gradients with respect to value, locations and
 * weights, all fp32.  The chain rule applied to the definition above; with
 * go = grad_out[b,q,g,:], per point t = (l, k) and inside corner c of its
 * sample, bilinear weights wy, wx:
 *
 *   grad_value[c]     += a[t] wy wx go
 *   grad_a[t]          = sum_c wy wx <go, v_c>
 *   grad_locations[t]  = a[t] (W_l sum_c wy sx <go, v_c>, H_l sum_c sy wx <go, v_c>)
 *   grad_weights[t]    = grad_a[t], or with softmax
 *                        a[t] (grad_a[t] - sum_s a[s] grad_a[s])
 *
 * sx, sy = -1 for the left/top corner and +1 for the right/bottom one: at
 * an integer coordinate the derivative of the cell floor() picks; a point
 * whose corners are all outside has zero gradients.  The page's backward
 * writes the value gradient with no intermediate sampling buffer, and its
 * float32 accumulator is the exact choice (section "Backend selection");
 * this one accumulates grad_value by fp32 reductions (so its last bits
 * depend on the order of the additions).
 *
 * Layouts (device pointers, dense): value, locations, weights, shapes,
 * starts as dcn_msda_forward; grad_out [B, Q, G, D] `dtype`; grad_value
 * [B, S, G, D] fp32, overwritten (zeroed first, then accumulated);
 * grad_locations [B, Q, G, L, K, 2] fp32, 8-byte aligned, overwritten;
 * grad_weights [B, Q, G, L*K] fp32, overwritten.  Every pointer is
 * required.  Arithmetic in fp32.  Errors as dcn_msda_forward.
 * Asynchronous on `stream`; allocates nothing; no handle. */
DCN_API dcn_status_t dcn_msda_backward(const void *value, const int *shapes, const int *starts,
                               int L, const float *locations, const float *weights,
                               const void *grad_out, float *grad_value, float *grad_locations,
                               float *grad_weights, int B, int S, int G, int D, int Q, int K,
                               int softmax, int dtype, void *stream);

/* ------------------------------------------------ single-scale deformable sampling
 *
 * The forward pass of the operator of page "deformops 3.0.1", section
 * "Single-scale deformable sampling" (the layers DeformAttn2d and
 * DeformSample2d, functional form attn; the DCNv3 operator of InternImage),
 * which samples and aggregates without the spatial weight of deformable
 * convolution.  B batch, G groups of D channels, a kh x kw tap grid (K
 * taps, tap k = i*kw + j):
 *
 *   out[b,ho,wo,g,d] = sum_k a[b,ho,wo,g,k] * S(value[b,:,:,g,d], py, px),
 *   py = ho*stride_h - pad_h + i*dil_h + dy,  px = wo*stride_w - pad_w + j*dil_w + dx,
 *
 * S the bilinear sample (corners outside the map contribute 0), (dy, dx)
 * = offsets[b,ho,wo,g,k,:], a the weights as given or, with softmax != 0,
 * softmax-normalized over the K taps of each (b, ho, wo, g).  The page
 * fixes none of the coordinate details; these are the deformable
 * convolution's own (its tap grid, stride, padding and dilation, (dy, dx)
 * pixel offsets), so the operator equals a depthwise dcn_forward_ex with
 * unit weights, G offset groups and the weights as the mask.
 * Ho = (H + 2 pad_h - dil_h (kh-1) - 1) / stride_h + 1, Wo likewise.
 *
 * Layouts (device pointers, dense, channels-last):
 *   value    [B, H, W, G, D]         `dtype`
 *   offsets  [B, Ho, Wo, G, K, 2]    fp32 (dy, dx), 8-byte aligned
 *   weights  [B, Ho, Wo, G, K]       fp32
 *   out      [B, Ho, Wo, G, D]       `dtype`
 * Arithmetic in fp32 (coordinates, weights, softmax, sums), one rounding to
 * `dtype` at the end.  Every size positive (pads >= 0), Ho, Wo > 0, each
 * tensor below 2^31 elements, else DCN_ERR_INVALID_ARG.  Asynchronous on
 * `stream`; allocates nothing; no handle. */
DCN_API dcn_status_t dcn_attn_forward(const void *value, const float *offsets,
                              const float *weights, void *out, int B, int H, int W, int G,
                              int D, int kh, int kw, int stride_h, int stride_w, int pad_h,
                              int pad_w, int dil_h, int dil_w, int softmax, int dtype,
                              void *stream);

/* The backward of dcn_attn_forward: for the cotangent grad_out [B, Ho, Wo,
 * G, D] (`dtype`, like value), the gradients with respect to value,
 * offsets and weights, all fp32.  The chain rule applied to the definition
 * above; with go = grad_out[b,ho,wo,g,:], per tap k and inside corner c of
 * its sample, bilinear weights wy, wx:
 *
 *   grad_value[c]    += a[k] wy wx go
 *   grad_a[k]         = sum_c wy wx <go, v_c>
 *   grad_offsets[k]   = a[k] (sum_c sy wx <go, v_c>, sum_c wy sx <go, v_c>)   (dy, dx)
 *   grad_weights[k]   = grad_a[k], or with softmax
 *                       a[k] (grad_a[k] - sum_s a[s] grad_a[s])
 *
 * sx, sy = -1 for the left/top corner and +1 for the right/bottom one: at
 * an integer coordinate the derivative of the cell floor() picks; a tap
 * whose corners are all outside has zero gradients.  The value gradient is
 * accumulated by fp32 reductions with no intermediate buffer (the page's
 * float32-accumulator rule, which it gives single-scale sampling and MSDA
 * alike), so its last bits depend on the order of the additions.
 *
 * Layouts (device pointers, dense, channels-last): value, offsets, weights
 * as dcn_attn_forward; grad_out [B, Ho, Wo, G, D] `dtype`; grad_value
 * [B, H, W, G, D] fp32, overwritten (zeroed first, then accumulated);
 * grad_offsets [B, Ho, Wo, G, K, 2] fp32, 8-byte aligned, overwritten;
 * grad_weights [B, Ho, Wo, G, K] fp32, overwritten.  Every pointer is
 * required.  Arithmetic in fp32.  Errors as dcn_attn_forward.
 * Asynchronous on `stream`; allocates nothing; no handle. */
DCN_API dcn_status_t dcn_attn_backward(const void *value, const float *offsets,
                               const float *weights, const void *grad_out, float *grad_value,
                               float *grad_offsets, float *grad_weights, int B, int H, int W,
                               int G, int D, int kh, int kw, int stride_h, int stride_w,
                               int pad_h, int pad_w, int dil_h, int dil_w, int softmax,
                               int dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DCN_H */
