// C ABI of the deformable convolution forward pass: argument checks,
// handle/workspace management and kernel selection.  Every entry point
// validates before launching (the entry-check-then-launch pattern of the
// "StyleGAN2 upfirdn2d" tutorial page, its C++ entry section) and reports a
// status code instead of throwing.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "dcn.h"
#include "dcn_device.cuh"
#include "dcn_backward.h"
#include "dcn_kernels.h"
#include "dcn_limits.h"
#include "dcn_sampling_ops.h"

struct dcn_handle_s {
    int device = 0;
    int sm_count = 0;
    int path = DCN_PATH_AUTO;
    int last_path = -1;
    int sample = DCN_SAMPLE_INPUT_DTYPE;

    // packed weight [O][kh*kw*(C/groups)]; the key of the last pack
    void *wpack = nullptr;
    size_t wpack_cap = 0;
    int pk_O = 0, pk_Cg = 0, pk_kh = 0, pk_kw = 0, pk_dtype = -1, pk_perm = 0;

    unsigned *status = nullptr;  // device status word

    // stream-K workspace of the tensor-core kernel: one fp32 partial tile
    // and one flag word per SM, and the flag value of the next launch
    void *partial = nullptr;
    size_t partial_cap = 0;
    void *flags = nullptr;
    size_t flags_cap = 0;
    unsigned epoch = 0;

    // backward on tensor cores: the weight packed as [kh*kw*C][O]
    void *wpack_bwd = nullptr;
    size_t wpack_bwd_cap = 0;

    // dcn_forward_host's pipeline: a kernel stream, a download stream and
    // the events between them (created on first use)
    cudaStream_t s_kernel = nullptr, s_down = nullptr;
    cudaEvent_t ev_in = nullptr, ev_k = nullptr, ev_done = nullptr;

    // dcn_backward: the weight gradient's stream beside the data kernel and
    // the fork / join events (created on first use)
    cudaStream_t s_wgrad = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;

    // device staging for dcn_forward_host: x, offset, mask, weight, bias, out
    void *stage[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    unsigned *host_status = nullptr;   // pinned copy of the status word (host-buffer entry)
    size_t stage_cap[6] = {0, 0, 0, 0, 0, 0};

    PFN_cuTensorMapEncodeTiled_v12000 encode_tiled = nullptr;
};

namespace {

// Bands of output rows per dcn_forward_host call (whole images when there
// are at least this many), the last one a quarter of the image: measured on
// the 7x7 workload, three bands of 96, 96 and 64 rows took 334 us per call,
// four of 64 rows 343 us, four of 80, 80, 64 and 32 rows 346 us and five
// bands 356-359 us (earlier, with uniform bands: 2, 3, 4, 6 and 8 bands
// 371, 359, 352, 373 and 428 us).  A band's kernel takes about as long
// whatever its height (each tile runs all its taps in sequence), so more
// bands cost more than the shorter tail after the last upload saves.
constexpr int kHostBands = 3;
constexpr int kHostLastDiv = 4;

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per barrier wait
using dcn::kIndexLimit;
using dcn::within_index_limit;

inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// A handle's workspace, status word and packed weight live on the device
// that was current at dcn_create; an entry point that launches work refuses
// the handle when another device is current (its pointers would reach
// another GPU's memory).
inline bool bad_handle(dcn_handle_t h) {
    if (!h) return true;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return dev != h->device;
}

inline bool aligned(const void *p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline size_t esize(int dtype) { return dtype == DCN_F32 ? 4 : 2; }
inline bool valid_dtype(int dtype) { return dtype == DCN_F32 || dtype == DCN_BF16 || dtype == DCN_F16; }
// bf16 and fp16 run on the tensor cores where the shape allows
inline bool tc_dtype(int dtype) { return dtype == DCN_BF16 || dtype == DCN_F16; }

// A validated problem: the descriptor and its output size.
struct Conv {
    dcn_conv_desc_t d;
    int Ho, Wo;
    int taps() const { return d.kh * d.kw; }
    int Cg() const { return d.C / d.groups; }
    int Og() const { return d.O / d.groups; }
    int Cq() const { return d.C / d.offset_groups; }
};

long long out_size_ll(long long n, long long k, long long stride, long long pad, long long dil) {
    const long long span = n + 2 * pad - dil * (k - 1) - 1;
    return span < 0 ? 0 : span / stride + 1;
}

dcn_status_t make_conv(const dcn_conv_desc_t &d, int dtype, Conv *c) {
    if (!valid_dtype(dtype)) return DCN_ERR_INVALID_ARG;
    if (d.B <= 0 || d.C <= 0 || d.H <= 0 || d.W <= 0 || d.O <= 0 || d.kh <= 0 || d.kw <= 0)
        return DCN_ERR_INVALID_ARG;
    if (d.stride_h <= 0 || d.stride_w <= 0 || d.dil_h <= 0 || d.dil_w <= 0 || d.pad_h < 0 || d.pad_w < 0)
        return DCN_ERR_INVALID_ARG;
    if (d.groups <= 0 || d.C % d.groups || d.O % d.groups) return DCN_ERR_INVALID_ARG;
    if (d.offset_groups <= 0 || d.C % d.offset_groups) return DCN_ERR_INVALID_ARG;
    const long long Ho = out_size_ll(d.H, d.kh, d.stride_h, d.pad_h, d.dil_h);
    const long long Wo = out_size_ll(d.W, d.kw, d.stride_w, d.pad_w, d.dil_w);
    if (Ho <= 0 || Wo <= 0 || Ho > kIndexLimit || Wo > kIndexLimit) return DCN_ERR_INVALID_ARG;
    if (!within_index_limit({d.kh, d.kw})) return DCN_ERR_INVALID_ARG;
    const long long taps = static_cast<long long>(d.kh) * d.kw;
    if (!within_index_limit({d.B, d.H, d.W, d.C}) ||
        !within_index_limit({d.B, 2, d.offset_groups, taps, Ho, Wo}) ||
        !within_index_limit({d.B, Ho, Wo, d.O}) ||
        !within_index_limit({d.O, d.C / d.groups, taps}))
        return DCN_ERR_INVALID_ARG;
    c->d = d;
    c->Ho = static_cast<int>(Ho);
    c->Wo = static_cast<int>(Wo);
    return DCN_OK;
}

// The page form: stride 1, dilation 1, one padding, one group.
dcn_conv_desc_t page_desc(int B, int C, int H, int W, int O, int kh, int kw, int pad) {
    dcn_conv_desc_t d;
    d.B = B; d.C = C; d.H = H; d.W = W; d.O = O; d.kh = kh; d.kw = kw;
    d.stride_h = d.stride_w = 1;
    d.pad_h = d.pad_w = pad;
    d.dil_h = d.dil_w = 1;
    d.groups = d.offset_groups = 1;
    return d;
}

// Whether the tensor-core kernel runs this problem (one launch per weight
// group and per 256 output channels; offset groups as virtual taps).  A
// group's channels go in whole 64-channel blocks, the last one completed
// with zeros when Cg % 64 != 0; several offset groups inside one weight
// group need whole blocks each.
bool tc_general_ok(const Conv &c) {
    const int Cg = c.Cg(), Cq = c.Cq(), Og = c.Og();
    if (Cg % 16 != 0 || Og % 16 != 0) return false;
    if (Cg % Cq != 0 && Cq % Cg != 0) return false;
    const int og_count = Cq >= Cg ? 1 : Cg / Cq;
    if (og_count > 1 && Cq % 64 != 0) return false;
    if (static_cast<long long>(c.taps()) * og_count > dcn::tc_max_virtual_taps) return false;
    return dcn::tc_supported(Cg, Og < 256 ? Og : 256);
}

// Grow a device buffer in stream order.
dcn_status_t ensure(void **buf, size_t *cap, size_t bytes, cudaStream_t s) {
    if (*cap >= bytes && *buf) return DCN_OK;
    if (*buf) {
        if (cudaFreeAsync(*buf, s) != cudaSuccess) return DCN_ERR_CUDA;
        *buf = nullptr;
        *cap = 0;
    }
    if (cudaMallocAsync(buf, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        *buf = nullptr;
        return DCN_ERR_OOM;
    }
    *cap = bytes;
    return DCN_OK;
}

dcn_status_t pack_impl(dcn_handle_t h, const void *weight, const Conv &c, int dtype,
                       cudaStream_t s) {
    const int O = c.d.O, Cg = c.Cg(), kh = c.d.kh, kw = c.d.kw;
    const int perm = dcn::tc_pack_permuted(dtype, Cg) ? 1 : 0;
    const size_t bytes = static_cast<size_t>(O) * dcn::pack_kc(Cg, perm) * kh * kw * esize(dtype);
    dcn_status_t st = ensure(&h->wpack, &h->wpack_cap, bytes, s);
    if (st != DCN_OK) return st;
    if (dcn::launch_pack_weight(weight, h->wpack, O, Cg, kh, kw, dtype, perm, s) != cudaSuccess)
        return DCN_ERR_CUDA;
    h->pk_O = O; h->pk_Cg = Cg; h->pk_kh = kh; h->pk_kw = kw; h->pk_dtype = dtype;
    h->pk_perm = perm;
    return DCN_OK;
}

// The next flag value of the stream-K workspace (0 is never used).
dcn_status_t next_epoch(dcn_handle_t h, cudaStream_t s, unsigned *epoch) {
    if (++h->epoch == 0) {
        // flag values wrapped: clear the flags and start again at 1
        if (cudaMemsetAsync(h->flags, 0, h->flags_cap, s) != cudaSuccess) return DCN_ERR_CUDA;
        h->epoch = 1;
    }
    *epoch = h->epoch;
    return DCN_OK;
}


// A band of output rows [h0, h0 + rows) of a one-image problem; the
// offset, mask and out pointers then address the band's first row, and
// offset/mask planes stay `plane` elements apart (the whole image's).
struct Band {
    int h0, rows, plane;
};

// after_pack: this call's pack_impl launched the weight pack just before, on
// the same stream (the first tensor-core launch then overlaps it).
dcn_status_t forward_packed_impl(dcn_handle_t h, const void *x, const float *offset,
                                 const float *mask, const float *bias, void *out, const Conv &c,
                                 int dtype, cudaStream_t s, bool after_pack = false,
                                 const Band *band = nullptr) {
    const dcn_conv_desc_t &d = c.d;
    if (h->pk_O != d.O || h->pk_Cg != c.Cg() || h->pk_kh != d.kh || h->pk_kw != d.kw ||
        h->pk_dtype != dtype)
        return DCN_ERR_INVALID_ARG;
    const int taps = c.taps();

    // the whole problem (the CUDA-core kernel's view)
    dcn::Params p;
    p.x = x; p.offset = offset; p.mask = mask; p.wpack = h->wpack; p.bias = bias; p.out = out;
    p.B = d.B; p.C = d.C; p.H = d.H; p.W = d.W; p.O = d.O; p.kh = d.kh; p.kw = d.kw;
    p.sh = d.stride_h; p.sw = d.stride_w; p.ph = d.pad_h; p.pw = d.pad_w;
    p.dh = d.dil_h; p.dw = d.dil_w;
    p.groups = d.groups;
    p.ogroups = d.offset_groups;
    p.Ho = c.Ho;
    p.Wo = c.Wo;
    p.h0 = 0;
    p.plane = p.Ho * p.Wo;
    p.P = d.B * c.Ho * c.Wo;
    if (band) {   // one image (d.B == 1), rows [h0, h0 + rows)
        p.Ho = band->rows;
        p.h0 = band->h0;
        p.plane = band->plane;
        p.P = band->rows * c.Wo;
    }
    p.kc = dcn::pack_kc(c.Cg(), h->pk_perm);
    p.K = taps * p.kc;
    p.x_cstride = d.C;
    p.out_stride = d.O;
    p.og_count = d.offset_groups;
    p.off_bstride = 2 * taps * d.offset_groups;
    p.mask_bstride = taps * d.offset_groups;
    p.status = h->status;
    p.timeout_ns = kWaitLimitNs;
#ifdef DCN_CHECK_BOUNDS
    dcn::set_bounds(p, esize(dtype));
#endif
    p.sample_f32 = h->sample == DCN_SAMPLE_F32 ? 1 : 0;
    p.f16 = dtype == DCN_F16 ? 1 : 0;
    p.partial = nullptr;
    p.flags = nullptr;
    p.epoch = 0;
    p.sm_count = h->sm_count;
    p.units_per_cta = 0;
    p.wperm = h->pk_perm;

    const bool tc_ok = tc_dtype(dtype) && tc_general_ok(c) && h->pk_perm &&
                       aligned(x, 32) && aligned(out, 16) && aligned(h->wpack, 16);
    int path = h->path;
    if (path == DCN_PATH_AUTO) path = tc_ok ? DCN_PATH_TC : DCN_PATH_SIMT;
    if (path == DCN_PATH_TC && !tc_ok) return DCN_ERR_UNSUPPORTED;

    if (path == DCN_PATH_SIMT) {
        if (dcn::launch_simt(p, dtype, s) != cudaSuccess) return DCN_ERR_CUDA;
        h->last_path = path;
        return DCN_OK;
    }

    // tensor cores: one launch per weight group and per 256 of its outputs
    const int Cg = c.Cg(), Og = c.Og(), Cq = c.Cq();
    const int chunk_max = Og < 256 ? Og : 256;
    const size_t part_bytes = static_cast<size_t>(h->sm_count) * 128 * chunk_max * sizeof(float);
    const size_t flag_bytes = static_cast<size_t>(h->sm_count + 1) * sizeof(unsigned);
    // a workspace (re)allocation or clear puts stream work between the pack
    // and the first launch, which then is an ordinary one
    if (h->partial_cap < part_bytes || !h->partial) after_pack = false;
    dcn_status_t st = ensure(&h->partial, &h->partial_cap, part_bytes, s);
    if (st != DCN_OK) return st;
    if (h->flags_cap < flag_bytes || !h->flags) {
        after_pack = false;
        st = ensure(&h->flags, &h->flags_cap, flag_bytes, s);
        if (st != DCN_OK) return st;
        if (cudaMemsetAsync(h->flags, 0, h->flags_cap, s) != cudaSuccess) return DCN_ERR_CUDA;
        h->epoch = 0;
    }
    const size_t plane = static_cast<size_t>(p.plane);
    // 16-bit elements (bf16 or fp16): pointer arithmetic only
    const uint16_t *xb = static_cast<const uint16_t *>(x);
    const uint16_t *wb = static_cast<const uint16_t *>(h->wpack);
    uint16_t *ob = static_cast<uint16_t *>(out);
    for (int g = 0; g < d.groups; ++g) {
        // the offset groups of this weight group's channels
        const int og_base = g * Cg / Cq;
        const int og_count = Cq >= Cg ? 1 : Cg / Cq;
        for (int o0 = 0; o0 < Og; o0 += 256) {
            const int n = Og - o0 < 256 ? Og - o0 : 256;
            const size_t row0 = static_cast<size_t>(g) * Og + o0;
            dcn::Params q = p;
            q.x = xb + static_cast<size_t>(g) * Cg;
            q.C = Cg;
            q.O = n;
            q.groups = 1;
            q.ogroups = og_count;
            q.og_count = og_count;
            q.offset = offset + static_cast<size_t>(og_base) * 2 * taps * plane;
            q.mask = mask ? mask + static_cast<size_t>(og_base) * taps * plane : nullptr;
            q.wpack = wb + row0 * p.K;
            q.bias = bias ? bias + row0 : nullptr;
            q.out = ob + row0;
            CUtensorMap map;
            std::memset(&map, 0, sizeof(map));
            const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(n)};
            const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(p.K) * 2};
            const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(n)};
            const cuuint32_t estride[2] = {1, 1};
            CUresult r = h->encode_tiled(&map,
                                         dtype == DCN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                         const_cast<void *>(q.wpack), gdim, gstride, box, estride,
                                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return DCN_ERR_CUDA;
            q.partial = static_cast<float *>(h->partial);
            q.flags = static_cast<unsigned *>(h->flags);
            if (h->epoch + 1 == 0) after_pack = false;   // the wrap clears the flags first
            st = next_epoch(h, s, &q.epoch);
            if (st != DCN_OK) return st;
            // only the first launch directly follows the pack
            if (dcn::launch_tc(q, map, s, after_pack && g == 0 && o0 == 0) != cudaSuccess)
                return DCN_ERR_CUDA;
        }
    }
    h->last_path = path;
    return DCN_OK;
}

dcn_status_t check_forward_ptrs(const void *x, const float *offset, const float *mask,
                                const void *weight, const float *bias, void *out, int dtype,
                                bool need_weight) {
    if (!x || !offset || !out || (need_weight && !weight)) return DCN_ERR_INVALID_ARG;
    const size_t es = esize(dtype);
    if (!aligned(x, es) || !aligned(out, es) || (weight && !aligned(weight, es)))
        return DCN_ERR_INVALID_ARG;
    if (!aligned(offset, 4) || (mask && !aligned(mask, 4)) || (bias && !aligned(bias, 4)))
        return DCN_ERR_INVALID_ARG;
    return DCN_OK;
}

}  // namespace

extern "C" {

dcn_status_t dcn_create(dcn_handle_t *out_handle) {
    if (!out_handle) return DCN_ERR_INVALID_ARG;
    *out_handle = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
        cudaGetLastError();
        return DCN_ERR_NO_DEVICE;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DCN_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DCN_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return DCN_ERR_UNSUPPORTED;

    dcn_handle_t h = new (std::nothrow) dcn_handle_s();
    if (!h) return DCN_ERR_OOM;
    h->device = dev;
    h->sm_count = prop.multiProcessorCount;

    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        delete h;
        return DCN_ERR_CUDA;
    }
    h->encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);

    if (cudaMalloc(&h->status, sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return DCN_ERR_OOM;
    }
    if (cudaMemset(h->status, 0, sizeof(unsigned)) != cudaSuccess) {
        cudaFree(h->status);
        delete h;
        return DCN_ERR_CUDA;
    }
    *out_handle = h;
    return DCN_OK;
}

dcn_status_t dcn_destroy(dcn_handle_t h) {
    if (!h) return DCN_OK;
    dcn_status_t st = DCN_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) st = DCN_ERR_CUDA;
    if (h->wpack) cudaFree(h->wpack);
    if (h->partial) cudaFree(h->partial);
    if (h->flags) cudaFree(h->flags);
    if (h->wpack_bwd) cudaFree(h->wpack_bwd);
    if (h->status) cudaFree(h->status);
    for (int i = 0; i < 6; ++i)
        if (h->stage[i]) cudaFree(h->stage[i]);
    if (h->host_status) cudaFreeHost(h->host_status);
    if (h->s_kernel) cudaStreamDestroy(h->s_kernel);
    if (h->s_down) cudaStreamDestroy(h->s_down);
    if (h->s_wgrad) cudaStreamDestroy(h->s_wgrad);
    cudaEvent_t evs[5] = {h->ev_in, h->ev_k, h->ev_done, h->ev_fork, h->ev_join};
    for (cudaEvent_t e : evs)
        if (e) cudaEventDestroy(e);
    delete h;
    return st;
}

dcn_status_t dcn_pack_weight(dcn_handle_t h, const void *weight, int O, int C, int kh, int kw,
                             int dtype, void *stream) {
    if (bad_handle(h) || !weight) return DCN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return DCN_ERR_INVALID_ARG;
    if (O <= 0 || C <= 0 || kh <= 0 || kw <= 0) return DCN_ERR_INVALID_ARG;
    if (!within_index_limit({O, C, kh, kw})) return DCN_ERR_INVALID_ARG;
    if (!aligned(weight, esize(dtype))) return DCN_ERR_INVALID_ARG;
    Conv c;
    c.d = page_desc(1, C, 1, 1, O, kh, kw, 0);   // only (O, C, kh, kw) key the pack
    c.Ho = c.Wo = 1;
    return pack_impl(h, weight, c, dtype, as_stream(stream));
}

dcn_status_t dcn_pack_weight_ex(dcn_handle_t h, const void *weight, const dcn_conv_desc_t *desc,
                                int dtype, void *stream) {
    if (bad_handle(h) || !weight || !desc) return DCN_ERR_INVALID_ARG;
    Conv c;
    dcn_status_t st = make_conv(*desc, dtype, &c);
    if (st != DCN_OK) return st;
    if (!aligned(weight, esize(dtype))) return DCN_ERR_INVALID_ARG;
    return pack_impl(h, weight, c, dtype, as_stream(stream));
}

dcn_status_t dcn_forward_packed(dcn_handle_t h, const void *x, const float *offset,
                                const float *mask, const float *bias, void *out,
                                int B, int C, int H, int W, int O, int kh, int kw, int pad,
                                int dtype, void *stream) {
    if (bad_handle(h)) return DCN_ERR_INVALID_ARG;
    Conv c;
    dcn_status_t st = make_conv(page_desc(B, C, H, W, O, kh, kw, pad), dtype, &c);
    if (st != DCN_OK) return st;
    st = check_forward_ptrs(x, offset, mask, nullptr, bias, out, dtype, false);
    if (st != DCN_OK) return st;
    return forward_packed_impl(h, x, offset, mask, bias, out, c, dtype, as_stream(stream));
}

dcn_status_t dcn_forward_packed_ex(dcn_handle_t h, const void *x, const float *offset,
                                   const float *mask, const float *bias, void *out,
                                   const dcn_conv_desc_t *desc, int dtype, void *stream) {
    if (bad_handle(h) || !desc) return DCN_ERR_INVALID_ARG;
    Conv c;
    dcn_status_t st = make_conv(*desc, dtype, &c);
    if (st != DCN_OK) return st;
    st = check_forward_ptrs(x, offset, mask, nullptr, bias, out, dtype, false);
    if (st != DCN_OK) return st;
    return forward_packed_impl(h, x, offset, mask, bias, out, c, dtype, as_stream(stream));
}

static dcn_status_t forward_general(dcn_handle_t h, const void *x, const float *offset, const float *mask,
                             const void *weight, const float *bias, void *out, const Conv &c,
                             int dtype, void *stream) {
    dcn_status_t st = check_forward_ptrs(x, offset, mask, weight, bias, out, dtype, true);
    if (st != DCN_OK) return st;
    // a forced tensor-core path that cannot run this shape launches nothing
    if (h->path == DCN_PATH_TC &&
        !(tc_dtype(dtype) && tc_general_ok(c) && aligned(x, 32) && aligned(out, 16)))
        return DCN_ERR_UNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    st = pack_impl(h, weight, c, dtype, s);
    if (st != DCN_OK) return st;
    return forward_packed_impl(h, x, offset, mask, bias, out, c, dtype, s, true);
}

dcn_status_t dcn_forward(dcn_handle_t h, const void *x, const float *offset, const float *mask,
                         const void *weight, const float *bias, void *out,
                         int B, int C, int H, int W, int O, int kh, int kw, int pad,
                         int dtype, void *stream) {
    if (bad_handle(h)) return DCN_ERR_INVALID_ARG;
    Conv c;
    dcn_status_t st = make_conv(page_desc(B, C, H, W, O, kh, kw, pad), dtype, &c);
    if (st != DCN_OK) return st;
    return forward_general(h, x, offset, mask, weight, bias, out, c, dtype, stream);
}

dcn_status_t dcn_forward_ex(dcn_handle_t h, const void *x, const float *offset, const float *mask,
                            const void *weight, const float *bias, void *out,
                            const dcn_conv_desc_t *desc, int dtype, void *stream) {
    if (bad_handle(h) || !desc) return DCN_ERR_INVALID_ARG;
    Conv c;
    dcn_status_t st = make_conv(*desc, dtype, &c);
    if (st != DCN_OK) return st;
    return forward_general(h, x, offset, mask, weight, bias, out, c, dtype, stream);
}

static dcn_status_t backward_general(dcn_handle_t h, const void *x, const float *offset,
                                     const float *mask, const void *weight, const void *grad_out,
                                     float *grad_x, float *grad_offset, float *grad_mask,
                                     float *grad_weight, float *grad_bias, const Conv &c,
                                     int dtype, void *stream) {
    if (!x || !offset || !weight || !grad_out || !grad_x || !grad_offset || !grad_weight)
        return DCN_ERR_INVALID_ARG;
    const size_t es = esize(dtype);
    if (!aligned(x, es) || !aligned(weight, es) || !aligned(grad_out, es))
        return DCN_ERR_INVALID_ARG;
    const float *f32s[] = {offset, mask, grad_x, grad_offset, grad_mask, grad_weight, grad_bias};
    for (const float *f : f32s)
        if (f && !aligned(f, 4)) return DCN_ERR_INVALID_ARG;
    const dcn_conv_desc_t &d = c.d;
    const size_t taps = static_cast<size_t>(d.kh) * d.kw;
    const size_t HoWo = static_cast<size_t>(c.Ho) * c.Wo;
    // launch-grid limits of the weight-gradient kernel (taps and 64 x 64 tiles)
    const long long tiles = static_cast<long long>(d.groups) * ((c.Og() + 63) / 64) * ((c.Cg() + 63) / 64);
    if (taps > 65535 || tiles > 65535 || (d.C + 63) / 64 > 65535) return DCN_ERR_UNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    // the kernels add into the gradients: clear them first
    const size_t bytes[5] = {
        static_cast<size_t>(d.B) * d.H * d.W * d.C * 4,
        static_cast<size_t>(d.B) * 2 * d.offset_groups * taps * HoWo * 4,
        static_cast<size_t>(d.B) * d.offset_groups * taps * HoWo * 4,
        static_cast<size_t>(d.O) * c.Cg() * taps * 4,
        static_cast<size_t>(d.O) * 4,
    };
    float *bufs[5] = {grad_x, grad_offset, grad_mask, grad_weight, grad_bias};
    for (int i = 0; i < 5; ++i)
        if (bufs[i] && cudaMemsetAsync(bufs[i], 0, bytes[i], s) != cudaSuccess) return DCN_ERR_CUDA;
    dcn::BwdParams p;
    p.x = x; p.offset = offset; p.mask = mask; p.weight = weight; p.grad_out = grad_out;
    p.grad_x = grad_x; p.grad_offset = grad_offset; p.grad_mask = grad_mask;
    p.grad_weight = grad_weight; p.grad_bias = grad_bias;
    p.B = d.B; p.C = d.C; p.H = d.H; p.W = d.W; p.O = d.O; p.kh = d.kh; p.kw = d.kw;
    p.sh = d.stride_h; p.sw = d.stride_w; p.ph = d.pad_h; p.pw = d.pad_w;
    p.dh = d.dil_h; p.dw = d.dil_w;
    p.groups = d.groups;
    p.ogroups = d.offset_groups;
    p.Ho = c.Ho;
    p.Wo = c.Wo;
    p.P = d.B * c.Ho * c.Wo;
    p.sm_count = h->sm_count;
    p.gx_vec4 = (d.C % 4 == 0 && aligned(grad_x, 16)) ? 1 : 0;
    p.pix_run = 0;
    p.status = h->status;
    p.timeout_ns = kWaitLimitNs;
    p.f16 = dtype == DCN_F16 ? 1 : 0;
#ifdef DCN_CHECK_BOUNDS
    {
        auto range = [](const void *base, size_t bytes, const void *&lo, const void *&hi) {
            lo = base;
            hi = base ? static_cast<const char *>(base) + bytes : nullptr;
        };
        range(x, static_cast<size_t>(d.B) * d.H * d.W * d.C * es, p.x_lo, p.x_hi);
        range(offset, bytes[1], p.off_lo, p.off_hi);
        range(mask, bytes[2], p.mask_lo, p.mask_hi);
        range(grad_x, bytes[0], p.gx_lo, p.gx_hi);
        range(grad_offset, bytes[1], p.goff_lo, p.goff_hi);
        range(grad_mask, bytes[2], p.gmask_lo, p.gmask_hi);
        range(grad_weight, bytes[3], p.gw_lo, p.gw_hi);
    }
#endif

    // the column gradient on tensor cores where the shape allows it
    const bool tc_ok = tc_dtype(dtype) &&
                       dcn::bwd_tc_supported(d.C, d.O, d.groups, d.offset_groups) &&
                       aligned(x, 32) && aligned(grad_out, 16) && aligned(grad_x, 16);
    int path = h->path;
    if (path == DCN_PATH_AUTO) path = tc_ok ? DCN_PATH_TC : DCN_PATH_SIMT;
    if (path == DCN_PATH_TC && !tc_ok) return DCN_ERR_UNSUPPORTED;
    if (path == DCN_PATH_SIMT) {
        if (dcn::launch_backward(p, dtype, s) != cudaSuccess) return DCN_ERR_CUDA;
        h->last_path = path;
        return DCN_OK;
    }
    const size_t wt_bytes = taps * d.C * d.O * 2;
    dcn_status_t st = ensure(&h->wpack_bwd, &h->wpack_bwd_cap, wt_bytes, s);
    if (st != DCN_OK) return st;
    if (dcn::launch_pack_weight_bwd(weight, h->wpack_bwd, d.O, d.C, d.kh, d.kw, s) != cudaSuccess)
        return DCN_ERR_CUDA;
    const CUtensorMapDataType tdt = dtype == DCN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap gmap, wmap;
    std::memset(&gmap, 0, sizeof(gmap));
    std::memset(&wmap, 0, sizeof(wmap));
    {
        // grad_out [B][Ho][Wo][O]; box = 64 outputs x one 8 x 16 pixel tile
        const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(d.O), static_cast<cuuint64_t>(c.Wo),
                                    static_cast<cuuint64_t>(c.Ho), static_cast<cuuint64_t>(d.B)};
        const cuuint64_t gstride[3] = {static_cast<cuuint64_t>(d.O) * 2,
                                       static_cast<cuuint64_t>(c.Wo) * d.O * 2,
                                       static_cast<cuuint64_t>(c.Ho) * c.Wo * d.O * 2};
        const cuuint32_t box[4] = {64, 16, 8, 1};
        const cuuint32_t estride[4] = {1, 1, 1, 1};
        if (h->encode_tiled(&gmap, tdt, 4, const_cast<void *>(grad_out), gdim, gstride, box, estride,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DCN_ERR_CUDA;
    }
    {
        // packed weight [kh*kw*C][O]; box = 64 outputs x 64 channel rows
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(d.O), static_cast<cuuint64_t>(taps * d.C)};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(d.O) * 2};
        const cuuint32_t box[2] = {64, 64};
        const cuuint32_t estride[2] = {1, 1};
        if (h->encode_tiled(&wmap, tdt, 2, h->wpack_bwd, gdim, gstride, box, estride,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DCN_ERR_CUDA;
    }
    // The weight gradient on tensor cores: the sampled operand m * S of
    // each 128-pixel tile is contracted with the grad_out tile as soon as it
    // is sampled, in shared memory; fp32 accumulation in tensor memory.
    // The data kernel is bound by its reductions into grad_x in L2, not by
    // its SMs (7x7 workload: 1.08 ms on 152 SMs, about the same on 127), so
    // when the weight gradient's row blocks fit a quarter of the SMs it runs
    // beside it, on a stream of its own, one CTA per row block on SMs the
    // data kernel leaves free.  Measured: the backward call 1.21 -> 1.14 ms
    // (7x7), 0.547 -> 0.473 ms (backbone 3x3); two CTAs per row block (fewer
    // SMs for the data kernel) made the backbone slower again (0.590 ms).
    const int wg_blocks = dcn::bwd_wgrad_row_blocks(p);
    if (wg_blocks > 0 && wg_blocks * 4 <= h->sm_count) {
        auto make_stream = [](cudaStream_t *out) {
            return *out || cudaStreamCreateWithFlags(out, cudaStreamNonBlocking) == cudaSuccess;
        };
        auto make_event = [](cudaEvent_t *out) {
            return *out || cudaEventCreateWithFlags(out, cudaEventDisableTiming) == cudaSuccess;
        };
        if (!make_stream(&h->s_wgrad) || !make_event(&h->ev_fork) || !make_event(&h->ev_join))
            return DCN_ERR_CUDA;
        if (cudaEventRecord(h->ev_fork, s) != cudaSuccess ||
            cudaStreamWaitEvent(h->s_wgrad, h->ev_fork, 0) != cudaSuccess)
            return DCN_ERR_CUDA;
        dcn::BwdParams pw = p;
        pw.sm_count = wg_blocks;
        dcn::BwdParams pd = p;
        pd.sm_count = h->sm_count - wg_blocks;
        const bool wg_ok = dcn::launch_bwd_wgrad_tc(pw, gmap, h->s_wgrad) == cudaSuccess;
        const bool d_ok = dcn::launch_bwd_data_tc(pd, gmap, wmap, s) == cudaSuccess;
        // the caller's stream waits for the weight gradient, whatever failed
        const bool joined = cudaEventRecord(h->ev_join, h->s_wgrad) == cudaSuccess &&
                            cudaStreamWaitEvent(s, h->ev_join, 0) == cudaSuccess;
        if (!wg_ok || !d_ok || !joined) return DCN_ERR_CUDA;
    } else {
        if (dcn::launch_bwd_data_tc(p, gmap, wmap, s) != cudaSuccess) return DCN_ERR_CUDA;
        if (dcn::launch_bwd_wgrad_tc(p, gmap, s) != cudaSuccess) return DCN_ERR_CUDA;
    }
    if (grad_bias && dcn::launch_bwd_bias(p, dtype, s) != cudaSuccess) return DCN_ERR_CUDA;
    h->last_path = path;
    return DCN_OK;
}

dcn_status_t dcn_backward(dcn_handle_t h, const void *x, const float *offset, const float *mask,
                          const void *weight, const void *grad_out, float *grad_x,
                          float *grad_offset, float *grad_mask, float *grad_weight,
                          float *grad_bias, int B, int C, int H, int W, int O, int kh, int kw,
                          int pad, int dtype, void *stream) {
    if (bad_handle(h)) return DCN_ERR_INVALID_ARG;
    Conv c;
    dcn_status_t st = make_conv(page_desc(B, C, H, W, O, kh, kw, pad), dtype, &c);
    if (st != DCN_OK) return st;
    return backward_general(h, x, offset, mask, weight, grad_out, grad_x, grad_offset, grad_mask,
                            grad_weight, grad_bias, c, dtype, stream);
}

dcn_status_t dcn_backward_ex(dcn_handle_t h, const void *x, const float *offset,
                             const float *mask, const void *weight, const void *grad_out,
                             float *grad_x, float *grad_offset, float *grad_mask,
                             float *grad_weight, float *grad_bias, const dcn_conv_desc_t *desc,
                             int dtype, void *stream) {
    if (bad_handle(h) || !desc) return DCN_ERR_INVALID_ARG;
    Conv c;
    dcn_status_t st = make_conv(*desc, dtype, &c);
    if (st != DCN_OK) return st;
    return backward_general(h, x, offset, mask, weight, grad_out, grad_x, grad_offset, grad_mask,
                            grad_weight, grad_bias, c, dtype, stream);
}

dcn_status_t dcn_msda_forward(const void *value, const int *shapes, const int *starts, int L,
                              const float *locations, const float *weights, void *out, int B,
                              int S, int G, int D, int Q, int K, int softmax, int dtype,
                              void *stream) {
    if (!value || !shapes || !starts || !locations || !weights || !out) return DCN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return DCN_ERR_INVALID_ARG;
    if (B <= 0 || S <= 0 || G <= 0 || D <= 0 || Q <= 0 || K <= 0) return DCN_ERR_INVALID_ARG;
    if (L <= 0 || L > dcn::kMsdaMaxLevels) return DCN_ERR_UNSUPPORTED;
    if (!within_index_limit({B, S, G, D}) || !within_index_limit({B, Q, G, L, K, 2}) ||
        !within_index_limit({B, Q, G, D}))
        return DCN_ERR_INVALID_ARG;
    const size_t es = esize(dtype);
    if (!aligned(value, es) || !aligned(out, es) || !aligned(locations, 8) || !aligned(weights, 4))
        return DCN_ERR_INVALID_ARG;
    dcn::MsdaParams p;
    for (int l = 0; l < L; ++l) {
        const int H = shapes[2 * l], W = shapes[2 * l + 1];
        if (H <= 0 || W <= 0 || starts[l] < 0 ||
            static_cast<long long>(starts[l]) + static_cast<long long>(H) * W > S)
            return DCN_ERR_INVALID_ARG;
        p.H[l] = H;
        p.W[l] = W;
        p.start[l] = starts[l];
    }
    p.value = value; p.locations = locations; p.weights = weights; p.out = out;
    p.B = B; p.S = S; p.G = G; p.D = D; p.Q = Q; p.K = K; p.L = L;
    p.softmax = softmax ? 1 : 0;
#ifdef DCN_CHECK_BOUNDS
    p.v_lo = value;
    p.v_hi = static_cast<const char *>(value) + static_cast<size_t>(B) * S * G * D * es;
    p.gv_lo = p.gv_hi = nullptr;
#endif
    const bool vec = D % (dtype == DCN_F32 ? 4 : 8) == 0 && aligned(value, 16) && aligned(out, 16);
    if (dcn::launch_msda(p, dtype, vec, as_stream(stream)) != cudaSuccess) return DCN_ERR_CUDA;
    return DCN_OK;
}

dcn_status_t dcn_msda_backward(const void *value, const int *shapes, const int *starts, int L,
                               const float *locations, const float *weights, const void *grad_out,
                               float *grad_value, float *grad_locations, float *grad_weights,
                               int B, int S, int G, int D, int Q, int K, int softmax, int dtype,
                               void *stream) {
    if (!value || !shapes || !starts || !locations || !weights || !grad_out || !grad_value ||
        !grad_locations || !grad_weights)
        return DCN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return DCN_ERR_INVALID_ARG;
    if (B <= 0 || S <= 0 || G <= 0 || D <= 0 || Q <= 0 || K <= 0) return DCN_ERR_INVALID_ARG;
    if (L <= 0 || L > dcn::kMsdaMaxLevels) return DCN_ERR_UNSUPPORTED;
    if (!within_index_limit({B, S, G, D}) || !within_index_limit({B, Q, G, L, K, 2}) ||
        !within_index_limit({B, Q, G, D}))
        return DCN_ERR_INVALID_ARG;
    const size_t es = esize(dtype);
    if (!aligned(value, es) || !aligned(grad_out, es) || !aligned(locations, 8) ||
        !aligned(weights, 4) || !aligned(grad_value, 4) || !aligned(grad_locations, 8) ||
        !aligned(grad_weights, 4))
        return DCN_ERR_INVALID_ARG;
    dcn::MsdaBwdParams p;
    for (int l = 0; l < L; ++l) {
        const int H = shapes[2 * l], W = shapes[2 * l + 1];
        if (H <= 0 || W <= 0 || starts[l] < 0 ||
            static_cast<long long>(starts[l]) + static_cast<long long>(H) * W > S)
            return DCN_ERR_INVALID_ARG;
        p.H[l] = H;
        p.W[l] = W;
        p.start[l] = starts[l];
    }
    p.value = value; p.locations = locations; p.weights = weights; p.grad_out = grad_out;
    p.grad_value = grad_value; p.grad_locations = grad_locations; p.grad_weights = grad_weights;
    p.B = B; p.S = S; p.G = G; p.D = D; p.Q = Q; p.K = K; p.L = L;
    p.softmax = softmax ? 1 : 0;
#ifdef DCN_CHECK_BOUNDS
    p.v_lo = value;
    p.v_hi = static_cast<const char *>(value) + static_cast<size_t>(B) * S * G * D * es;
    p.gv_lo = grad_value;
    p.gv_hi = grad_value + static_cast<size_t>(B) * S * G * D;
#endif
    cudaStream_t s = as_stream(stream);
    // the value gradient is a sum of reductions: start it at zero
    if (cudaMemsetAsync(grad_value, 0, static_cast<size_t>(B) * S * G * D * sizeof(float), s) !=
        cudaSuccess)
        return DCN_ERR_CUDA;
    const bool vec = D % (dtype == DCN_F32 ? 4 : 8) == 0 && aligned(value, 16) &&
                     aligned(grad_out, 16) && aligned(grad_value, 16);
    if (dcn::launch_msda_backward(p, dtype, vec, s) != cudaSuccess) return DCN_ERR_CUDA;
    return DCN_OK;
}

dcn_status_t dcn_attn_forward(const void *value, const float *offsets, const float *weights,
                              void *out, int B, int H, int W, int G, int D, int kh, int kw,
                              int stride_h, int stride_w, int pad_h, int pad_w, int dil_h,
                              int dil_w, int softmax, int dtype, void *stream) {
    if (!value || !offsets || !weights || !out) return DCN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return DCN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || W <= 0 || G <= 0 || D <= 0 || kh <= 0 || kw <= 0 || stride_h <= 0 ||
        stride_w <= 0 || pad_h < 0 || pad_w < 0 || dil_h <= 0 || dil_w <= 0)
        return DCN_ERR_INVALID_ARG;
    const long long Ho = out_size_ll(H, kh, stride_h, pad_h, dil_h);
    const long long Wo = out_size_ll(W, kw, stride_w, pad_w, dil_w);
    if (Ho <= 0 || Wo <= 0) return DCN_ERR_INVALID_ARG;
    if (!within_index_limit({kh, kw}) || !within_index_limit({B, H, W, G, D}) ||
        !within_index_limit({B, Ho, Wo, G, kh, kw, 2}) || !within_index_limit({B, Ho, Wo, G, D}))
        return DCN_ERR_INVALID_ARG;
    const size_t es = esize(dtype);
    if (!aligned(value, es) || !aligned(out, es) || !aligned(offsets, 8) || !aligned(weights, 4))
        return DCN_ERR_INVALID_ARG;
    dcn::AttnParams p;
    p.value = value; p.offsets = offsets; p.weights = weights; p.out = out;
    p.B = B; p.H = H; p.W = W; p.G = G; p.D = D;
    p.Ho = static_cast<int>(Ho); p.Wo = static_cast<int>(Wo);
    p.kh = kh; p.kw = kw; p.sh = stride_h; p.sw = stride_w; p.ph = pad_h; p.pw = pad_w;
    p.dh = dil_h; p.dw = dil_w;
    p.softmax = softmax ? 1 : 0;
#ifdef DCN_CHECK_BOUNDS
    p.v_lo = value;
    p.v_hi = static_cast<const char *>(value) + static_cast<size_t>(B) * H * W * G * D * es;
    p.gv_lo = p.gv_hi = nullptr;
#endif
    const bool vec = D % (dtype == DCN_F32 ? 4 : 8) == 0 && aligned(value, 16) && aligned(out, 16);
    if (dcn::launch_attn(p, dtype, vec, as_stream(stream)) != cudaSuccess) return DCN_ERR_CUDA;
    return DCN_OK;
}

dcn_status_t dcn_attn_backward(const void *value, const float *offsets, const float *weights,
                               const void *grad_out, float *grad_value, float *grad_offsets,
                               float *grad_weights, int B, int H, int W, int G, int D, int kh,
                               int kw, int stride_h, int stride_w, int pad_h, int pad_w,
                               int dil_h, int dil_w, int softmax, int dtype, void *stream) {
    if (!value || !offsets || !weights || !grad_out || !grad_value || !grad_offsets ||
        !grad_weights)
        return DCN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return DCN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || W <= 0 || G <= 0 || D <= 0 || kh <= 0 || kw <= 0 || stride_h <= 0 ||
        stride_w <= 0 || pad_h < 0 || pad_w < 0 || dil_h <= 0 || dil_w <= 0)
        return DCN_ERR_INVALID_ARG;
    const long long Ho = out_size_ll(H, kh, stride_h, pad_h, dil_h);
    const long long Wo = out_size_ll(W, kw, stride_w, pad_w, dil_w);
    if (Ho <= 0 || Wo <= 0) return DCN_ERR_INVALID_ARG;
    if (!within_index_limit({kh, kw}) || !within_index_limit({B, H, W, G, D}) ||
        !within_index_limit({B, Ho, Wo, G, kh, kw, 2}) || !within_index_limit({B, Ho, Wo, G, D}))
        return DCN_ERR_INVALID_ARG;
    const size_t es = esize(dtype);
    if (!aligned(value, es) || !aligned(grad_out, es) || !aligned(offsets, 8) ||
        !aligned(weights, 4) || !aligned(grad_value, 4) || !aligned(grad_offsets, 8) ||
        !aligned(grad_weights, 4))
        return DCN_ERR_INVALID_ARG;
    dcn::AttnBwdParams p;
    p.value = value; p.offsets = offsets; p.weights = weights; p.grad_out = grad_out;
    p.grad_value = grad_value; p.grad_offsets = grad_offsets; p.grad_weights = grad_weights;
    p.B = B; p.H = H; p.W = W; p.G = G; p.D = D;
    p.Ho = static_cast<int>(Ho); p.Wo = static_cast<int>(Wo);
    p.kh = kh; p.kw = kw; p.sh = stride_h; p.sw = stride_w; p.ph = pad_h; p.pw = pad_w;
    p.dh = dil_h; p.dw = dil_w;
    p.softmax = softmax ? 1 : 0;
#ifdef DCN_CHECK_BOUNDS
    p.v_lo = value;
    p.v_hi = static_cast<const char *>(value) + static_cast<size_t>(B) * H * W * G * D * es;
    p.gv_lo = grad_value;
    p.gv_hi = grad_value + static_cast<size_t>(B) * H * W * G * D;
#endif
    cudaStream_t s = as_stream(stream);
    // the value gradient is a sum of reductions: start it at zero
    if (cudaMemsetAsync(grad_value, 0, static_cast<size_t>(B) * H * W * G * D * sizeof(float), s) !=
        cudaSuccess)
        return DCN_ERR_CUDA;
    // four channels per lane: 8-byte (16-bit) or 16-byte (fp32) loads,
    // 16-byte reductions
    const size_t la = dtype == DCN_F32 ? 16 : 8;
    const bool vec = D % 4 == 0 && aligned(value, la) && aligned(grad_out, la) &&
                     aligned(grad_value, 16);
    if (dcn::launch_attn_backward(p, dtype, vec, s) != cudaSuccess) return DCN_ERR_CUDA;
    return DCN_OK;
}

static dcn_status_t layout_copy(const void *src, void *dst, int B, int R, int S, int dtype,
                                void *stream) {
    if (!src || !dst || src == dst) return DCN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || B <= 0 || R <= 0 || S <= 0) return DCN_ERR_INVALID_ARG;
    if (!within_index_limit({B, R, S})) return DCN_ERR_INVALID_ARG;
    const size_t es = esize(dtype);
    if (!aligned(src, es) || !aligned(dst, es)) return DCN_ERR_INVALID_ARG;
    if (B > 65535 || (R + 31) / 32 > 65535) return DCN_ERR_UNSUPPORTED;
    if (dcn::launch_transpose(src, dst, B, R, S, static_cast<int>(es), as_stream(stream)) != cudaSuccess)
        return DCN_ERR_CUDA;
    return DCN_OK;
}

dcn_status_t dcn_nchw_to_nhwc(const void *src, void *dst, int B, int C, int H, int W, int dtype,
                              void *stream) {
    if (H <= 0 || W <= 0 || !within_index_limit({H, W})) return DCN_ERR_INVALID_ARG;
    return layout_copy(src, dst, B, C, H * W, dtype, stream);
}

dcn_status_t dcn_nhwc_to_nchw(const void *src, void *dst, int B, int C, int H, int W, int dtype,
                              void *stream) {
    if (H <= 0 || W <= 0 || !within_index_limit({H, W})) return DCN_ERR_INVALID_ARG;
    return layout_copy(src, dst, B, H * W, C, dtype, stream);
}

int dcn_out_size(int n, int k, int stride, int pad, int dil) {
    if (n <= 0 || k <= 0 || stride <= 0 || pad < 0 || dil <= 0) return 0;
    const long long r = out_size_ll(n, k, stride, pad, dil);
    return r > kIndexLimit ? 0 : static_cast<int>(r);
}

dcn_status_t dcn_sync_status(dcn_handle_t h, void *stream) {
    if (bad_handle(h)) return DCN_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return DCN_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, h->status, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DCN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DCN_ERR_CUDA;
    if (word != 0) {
        if (cudaMemsetAsync(h->status, 0, sizeof(unsigned), s) != cudaSuccess) return DCN_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return DCN_ERR_CUDA;
        return (word & dcn::kStatusBounds) ? DCN_ERR_BOUNDS : DCN_ERR_TIMEOUT;
    }
    return DCN_OK;
}

dcn_status_t dcn_forward_host(dcn_handle_t h, const void *x, const float *offset,
                              const float *mask, const void *weight, const float *bias, void *out,
                              int B, int C, int H, int W, int O, int kh, int kw, int pad,
                              int dtype, void *stream) {
    if (bad_handle(h)) return DCN_ERR_INVALID_ARG;
    Conv c;
    dcn_status_t st = make_conv(page_desc(B, C, H, W, O, kh, kw, pad), dtype, &c);
    if (st != DCN_OK) return st;
    st = check_forward_ptrs(x, offset, mask, weight, bias, out, dtype, true);
    if (st != DCN_OK) return st;
    const size_t es = esize(dtype);
    const size_t Ho = static_cast<size_t>(c.Ho), Wo = static_cast<size_t>(c.Wo);
    const size_t taps = static_cast<size_t>(kh) * kw;
    const size_t bytes[6] = {
        static_cast<size_t>(B) * H * W * C * es,
        static_cast<size_t>(B) * 2 * taps * Ho * Wo * 4,
        mask ? static_cast<size_t>(B) * taps * Ho * Wo * 4 : 0,
        static_cast<size_t>(O) * C * taps * es,
        bias ? static_cast<size_t>(O) * 4 : 0,
        static_cast<size_t>(B) * Ho * Wo * O * es,
    };
    cudaStream_t s = as_stream(stream);
    for (int i = 0; i < 6; ++i) {
        if (bytes[i] == 0) continue;
        // round up so every staging buffer starts 256-byte aligned and is reusable
        st = ensure(&h->stage[i], &h->stage_cap[i], (bytes[i] + 255) & ~static_cast<size_t>(255), s);
        if (st != DCN_OK) return st;
    }
    // Each pipeline resource is made on first use and stored only once made,
    // so a failure part way leaves the others in place and this one null, to
    // be retried by the next call (dcn_destroy frees whichever exist).
    auto make_stream = [](cudaStream_t *out) {
        cudaStream_t t = nullptr;
        if (*out) return true;
        if (cudaStreamCreateWithFlags(&t, cudaStreamNonBlocking) != cudaSuccess) return false;
        *out = t;
        return true;
    };
    auto make_event = [](cudaEvent_t *out) {
        cudaEvent_t t = nullptr;
        if (*out) return true;
        if (cudaEventCreateWithFlags(&t, cudaEventDisableTiming) != cudaSuccess) return false;
        *out = t;
        return true;
    };
    if (!make_stream(&h->s_kernel) || !make_stream(&h->s_down) || !make_event(&h->ev_in) ||
        !make_event(&h->ev_k) || !make_event(&h->ev_done))
        return DCN_ERR_CUDA;
    if (!h->host_status) {
        void *t = nullptr;
        if (cudaHostAlloc(&t, sizeof(unsigned), cudaHostAllocDefault) != cudaSuccess)
            return DCN_ERR_CUDA;
        h->host_status = static_cast<unsigned *>(t);
    }
    // The host link is the slow part (the copies take longer than the
    // kernel), so the call is a pipeline over bands of output rows: the
    // band's offsets and mask go up on `stream`, its kernel runs on the
    // handle's kernel stream once they (and x, the weight and its pack)
    // have landed, and its rows of out come down on the download stream --
    // so later bands' uploads overlap earlier bands' kernels and downloads.
    // Stream order: copies and the pack on `stream`; each band's kernel
    // waits for its uploads; each download waits for its kernel; `stream`
    // waits for the last download before the final synchronisation.
    if (cudaMemcpyAsync(h->stage[3], weight, bytes[3], cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DCN_ERR_CUDA;
    if (bias && cudaMemcpyAsync(h->stage[4], bias, bytes[4], cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DCN_ERR_CUDA;
    st = pack_impl(h, h->stage[3], c, dtype, s);
    if (st != DCN_OK) return st;
    const int per_image = B >= kHostBands ? 1 : (kHostBands + B - 1) / B;
    int rows = static_cast<int>((Ho + per_image - 1) / per_image);
    rows = (rows + 7) & ~7;   // whole 8-row tiles
    if (rows < 8) rows = 8;
    int last_rows = 0;        // 0: every band `rows` tall
    if (per_image > 1) {
        last_rows = ((static_cast<int>(Ho) / kHostLastDiv) + 7) & ~7;
        if (last_rows < 8) last_rows = 8;
        const int rest = static_cast<int>(Ho) - last_rows;
        rows = ((rest + per_image - 2) / (per_image - 1) + 7) & ~7;
        if (rows < 8) rows = 8;
    }
    Conv c1 = c;
    c1.d.B = 1;
    const size_t img_x = static_cast<size_t>(H) * W * C * es;
    const size_t plane = Ho * Wo;
    uint8_t *sx = static_cast<uint8_t *>(h->stage[0]);
    float *soff = static_cast<float *>(h->stage[1]);
    float *smask = static_cast<float *>(h->stage[2]);
    uint8_t *sout = static_cast<uint8_t *>(h->stage[5]);
    const uint8_t *hx = static_cast<const uint8_t *>(x);
    bool queued = false;   // work sits on the pipeline streams
    auto run_bands = [&]() -> dcn_status_t {
        for (int b = 0; b < B; ++b) {
            if (cudaMemcpyAsync(sx + b * img_x, hx + b * img_x, img_x, cudaMemcpyHostToDevice, s) != cudaSuccess)
                return DCN_ERR_CUDA;
            for (int h0 = 0; h0 < static_cast<int>(Ho);) {
                int r = static_cast<int>(Ho) - h0 < rows ? static_cast<int>(Ho) - h0 : rows;
                // the last band (at most last_rows) ends the call sooner
                if (last_rows > 0 && static_cast<int>(Ho) - h0 - r < last_rows && static_cast<int>(Ho) - h0 > last_rows)
                    r = static_cast<int>(Ho) - h0 - last_rows;
                // this band's rows of every offset and mask plane of image b
                const size_t first = static_cast<size_t>(h0) * Wo;
                const size_t off0 = static_cast<size_t>(b) * 2 * taps * plane + first;
                if (cudaMemcpy2DAsync(soff + off0, plane * 4, offset + off0, plane * 4, r * Wo * 4, 2 * taps,
                                      cudaMemcpyHostToDevice, s) != cudaSuccess)
                    return DCN_ERR_CUDA;
                const size_t m0 = static_cast<size_t>(b) * taps * plane + first;
                if (mask && cudaMemcpy2DAsync(smask + m0, plane * 4, mask + m0, plane * 4, r * Wo * 4, taps,
                                              cudaMemcpyHostToDevice, s) != cudaSuccess)
                    return DCN_ERR_CUDA;
                if (cudaEventRecord(h->ev_in, s) != cudaSuccess ||
                    cudaStreamWaitEvent(h->s_kernel, h->ev_in, 0) != cudaSuccess)
                    return DCN_ERR_CUDA;
                const Band band = {h0, r, static_cast<int>(plane)};
                const size_t out0 = (static_cast<size_t>(b) * Ho + h0) * Wo * O * es;
                queued = true;
                const dcn_status_t bs = forward_packed_impl(h, sx + b * img_x, soff + off0, mask ? smask + m0 : nullptr,
                                         bias ? static_cast<const float *>(h->stage[4]) : nullptr,
                                         sout + out0, c1, dtype, h->s_kernel, false, &band);
                if (bs != DCN_OK) return bs;
                if (cudaEventRecord(h->ev_k, h->s_kernel) != cudaSuccess ||
                    cudaStreamWaitEvent(h->s_down, h->ev_k, 0) != cudaSuccess)
                    return DCN_ERR_CUDA;
                if (cudaMemcpyAsync(static_cast<uint8_t *>(out) + out0, sout + out0, r * Wo * O * es,
                                    cudaMemcpyDeviceToHost, h->s_down) != cudaSuccess)
                    return DCN_ERR_CUDA;
                h0 += r;
            }
        }
        return DCN_OK;
    };
    st = run_bands();
    if (st != DCN_OK) {
        // An error part way: earlier bands' kernels and downloads may still
        // be queued on the pipeline streams and read the staging buffers.
        // Make `stream` wait for both, so the next call's uploads and any
        // reallocation on `stream` come after them.
        if (queued) {
            if (cudaEventRecord(h->ev_k, h->s_kernel) == cudaSuccess)
                cudaStreamWaitEvent(s, h->ev_k, 0);
            if (cudaEventRecord(h->ev_done, h->s_down) == cudaSuccess)
                cudaStreamWaitEvent(s, h->ev_done, 0);
        }
        return st;
    }
    if (cudaEventRecord(h->ev_done, h->s_down) != cudaSuccess ||
        cudaStreamWaitEvent(s, h->ev_done, 0) != cudaSuccess)
        return DCN_ERR_CUDA;
    // the status word comes back behind the last download: one
    // synchronisation for both (the word is cleared only when it is set)
    if (cudaMemcpyAsync(h->host_status, h->status, sizeof(unsigned), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return DCN_ERR_CUDA;
    if (*h->host_status != 0) return dcn_sync_status(h, stream);
    return DCN_OK;
}

dcn_status_t dcn_set_path(dcn_handle_t h, int path) {
    if (!h || path < DCN_PATH_AUTO || path > DCN_PATH_TC) return DCN_ERR_INVALID_ARG;
    h->path = path;
    return DCN_OK;
}

int dcn_last_path(dcn_handle_t h) { return h ? h->last_path : -1; }

dcn_status_t dcn_set_sample_precision(dcn_handle_t h, int mode) {
    if (!h || (mode != DCN_SAMPLE_INPUT_DTYPE && mode != DCN_SAMPLE_F32)) return DCN_ERR_INVALID_ARG;
    h->sample = mode;
    return DCN_OK;
}

dcn_status_t dcn_selftest_timeout(dcn_handle_t h, long long timeout_ns, void *stream) {
    if (bad_handle(h) || timeout_ns <= 0 || timeout_ns > 10000000000ll) return DCN_ERR_INVALID_ARG;
    if (dcn::launch_selftest_timeout(h->status, static_cast<unsigned long long>(timeout_ns),
                                     as_stream(stream)) != cudaSuccess)
        return DCN_ERR_CUDA;
    return DCN_OK;
}

const char *dcn_status_string(dcn_status_t s) {
    switch (s) {
        case DCN_OK: return "DCN_OK";
        case DCN_ERR_INVALID_ARG: return "DCN_ERR_INVALID_ARG";
        case DCN_ERR_UNSUPPORTED: return "DCN_ERR_UNSUPPORTED";
        case DCN_ERR_CUDA: return "DCN_ERR_CUDA";
        case DCN_ERR_NO_DEVICE: return "DCN_ERR_NO_DEVICE";
        case DCN_ERR_OOM: return "DCN_ERR_OOM";
        case DCN_ERR_TIMEOUT: return "DCN_ERR_TIMEOUT";
        case DCN_ERR_BOUNDS: return "DCN_ERR_BOUNDS";
    }
    return "DCN_ERR_UNKNOWN";
}

}  // extern "C"
