// dcn_forward_noalloc: the forward pass without any device allocation.
//
// Some callers cannot let a library call cudaMalloc: plugin hosts and
// inference engines that hand out all device memory themselves and forbid
// allocations behind their back, processes that fix their device-memory
// budget at start-up, and latency-critical loops where cudaMalloc/cudaFree
// may synchronise the device and stall every other stream.  For them this
// entry point keeps its only scratch -- the packed weight and a status word
// -- in file-scope __device__ arrays that exist on every GPU that loads the
// library, for the life of the process.  The caller still passes inputs and
// outputs.
//
// Host code must not hand the arrays' names to a kernel: on the host they
// are stand-ins, not device addresses.  Their device addresses are looked
// up once per device, with that device current, by cudaGetSymbolAddress.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "dcn.h"
#include "dcn_kernels.h"
#include "dcn_limits.h"

namespace {

constexpr size_t kScratchWeightBytes = DCN_NOALLOC_MAX_WEIGHT_BYTES;
constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// The packed weight [O][kh*kw*C] of the current call, shared by all calls.
static __device__ __align__(256) unsigned char g_wpack_scratch[kScratchWeightBytes];
// The status word the kernels' bounded waits report into.
static __device__ __align__(256) unsigned g_status_scratch[64];

struct DeviceScratch {
    bool ready = false;
    void *wpack = nullptr;
    unsigned *status = nullptr;
    PFN_cuTensorMapEncodeTiled_v12000 encode_tiled = nullptr;
};

DeviceScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

// Once per device, with that device current: the device addresses of the
// scratch arrays and the tensor-map encoder.  No allocation.
dcn_status_t scratch_for_current_device(DeviceScratch **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DCN_ERR_NO_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return DCN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    DeviceScratch &s = g_scratch[dev];
    if (!s.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DCN_ERR_CUDA;
        if (prop.major != 10 || prop.minor != 3) return DCN_ERR_UNSUPPORTED;
        void *w = nullptr, *st = nullptr;
        if (cudaGetSymbolAddress(&w, g_wpack_scratch) != cudaSuccess) return DCN_ERR_CUDA;
        if (cudaGetSymbolAddress(&st, g_status_scratch) != cudaSuccess) return DCN_ERR_CUDA;
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return DCN_ERR_CUDA;
        s.wpack = w;
        s.status = static_cast<unsigned *>(st);
        s.encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        s.ready = true;
    }
    *out = &s;
    return DCN_OK;
}

inline bool is_aligned(const void *p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" DCN_API dcn_status_t dcn_forward_noalloc(
    const void *x, const float *offset, const float *mask, const void *weight, const float *bias,
    void *out, int B, int C, int H, int W, int O, int kh, int kw, int pad, int dtype, void *stream) {
    // the same argument rules as dcn_forward
    if (dtype != DCN_F32 && dtype != DCN_BF16 && dtype != DCN_F16) return DCN_ERR_INVALID_ARG;
    if (B <= 0 || C <= 0 || H <= 0 || W <= 0 || O <= 0 || kh <= 0 || kw <= 0 || pad < 0)
        return DCN_ERR_INVALID_ARG;
    const long long Ho = static_cast<long long>(H) + 2ll * pad - kh + 1;
    const long long Wo = static_cast<long long>(W) + 2ll * pad - kw + 1;
    if (Ho <= 0 || Wo <= 0) return DCN_ERR_INVALID_ARG;
    if (!dcn::within_index_limit({kh, kw})) return DCN_ERR_INVALID_ARG;
    const long long taps = static_cast<long long>(kh) * kw;
    if (!dcn::within_index_limit({B, H, W, C}) || !dcn::within_index_limit({B, 2, taps, Ho, Wo}) ||
        !dcn::within_index_limit({B, Ho, Wo, O}) || !dcn::within_index_limit({O, C, taps}))
        return DCN_ERR_INVALID_ARG;
    if (!x || !offset || !weight || !out) return DCN_ERR_INVALID_ARG;
    const size_t es = dtype == DCN_F32 ? 4 : 2;
    if (!is_aligned(x, es) || !is_aligned(out, es) || !is_aligned(weight, es) ||
        !is_aligned(offset, 4) || (mask && !is_aligned(mask, 4)) || (bias && !is_aligned(bias, 4)))
        return DCN_ERR_INVALID_ARG;
    // the packed weight must fit the fixed scratch array
    const int perm = dcn::tc_pack_permuted(dtype, C) ? 1 : 0;
    const int kc = dcn::pack_kc(C, perm);
    if (static_cast<unsigned long long>(O) * kc * taps * es > kScratchWeightBytes)
        return DCN_ERR_UNSUPPORTED;

    DeviceScratch *s = nullptr;
    dcn_status_t st = scratch_for_current_device(&s);
    if (st != DCN_OK) return st;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the status word keeps the previous call's value: start this call at zero
    if (cudaMemsetAsync(s->status, 0, sizeof(unsigned), cs) != cudaSuccess) return DCN_ERR_CUDA;
    if (dcn::launch_pack_weight(weight, s->wpack, O, C, kh, kw, dtype, perm, cs) != cudaSuccess)
        return DCN_ERR_CUDA;

    dcn::Params p;
    p.x = x; p.offset = offset; p.mask = mask; p.wpack = s->wpack; p.bias = bias; p.out = out;
    p.B = B; p.C = C; p.H = H; p.W = W; p.O = O; p.kh = kh; p.kw = kw;
    p.sh = p.sw = 1;
    p.ph = p.pw = pad;
    p.dh = p.dw = 1;
    p.groups = p.ogroups = 1;
    p.Ho = static_cast<int>(Ho);
    p.Wo = static_cast<int>(Wo);
    p.h0 = 0;
    p.plane = p.Ho * p.Wo;
    p.P = B * p.Ho * p.Wo;
    p.kc = kc;
    p.K = kh * kw * kc;
    p.x_cstride = C;
    p.out_stride = O;
    p.og_count = 1;
    p.off_bstride = 2 * kh * kw;
    p.mask_bstride = kh * kw;
    p.status = s->status;
    p.timeout_ns = kWaitLimitNs;
#ifdef DCN_CHECK_BOUNDS
    dcn::set_bounds(p, es);
#endif
    p.sample_f32 = 0;
    p.f16 = dtype == DCN_F16 ? 1 : 0;
    p.partial = nullptr;   // no stream-K workspace: one tile per CTA
    p.flags = nullptr;
    p.epoch = 0;
    p.sm_count = 0;
    p.units_per_cta = 0;
    p.wperm = perm;

    const bool tc = (dtype == DCN_BF16 || dtype == DCN_F16) && perm && dcn::tc_supported(C, O) && is_aligned(x, 32) &&
                    is_aligned(out, 16) && kh * kw <= dcn::tc_max_virtual_taps;
    cudaError_t e;
    if (tc) {
        CUtensorMap map;
        std::memset(&map, 0, sizeof(map));
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(O)};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(p.K) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(O)};
        const cuuint32_t estride[2] = {1, 1};
        if (s->encode_tiled(&map,
                            dtype == DCN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s->wpack, gdim, gstride, box,
                            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DCN_ERR_CUDA;
        e = dcn::launch_tc(p, map, cs);
    } else {
        e = dcn::launch_simt(p, dtype, cs);
    }
    return e == cudaSuccess ? DCN_OK : DCN_ERR_CUDA;
}
