// Row loads and stores shared by the CUDA-core sampling kernels (MSDA and
// single-scale sampling, forward and backward): CH consecutive elements of
// a value or cotangent row as fp32, from one 16-byte load (CH = 8 for the
// 16-bit types, 4 for fp32) or one element (CH = 1); four 16-bit elements
// from one 8-byte load; and the rounding of an fp32 result to the operand
// type (round to nearest even).
#pragma once

#include <cstdint>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace dcn {

template <typename T, int CH>
__device__ __forceinline__ void row_load(const T *p, float (&v)[CH]);

template <>
__device__ __forceinline__ void row_load<float, 4>(const float *p, float (&v)[4]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
template <>
__device__ __forceinline__ void row_load<__nv_bfloat16, 8>(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 r = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        v[2 * e] = __uint_as_float(w[e] << 16);
        v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}
template <>
__device__ __forceinline__ void row_load<__half, 8>(const __half *p, float (&v)[8]) {
    const uint4 r = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __half2 h;
        memcpy(&h, &w[e], 4);
        const float2 f = __half22float2(h);
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}
template <>
__device__ __forceinline__ void row_load<float, 1>(const float *p, float (&v)[1]) { v[0] = __ldg(p); }
template <>
__device__ __forceinline__ void row_load<__nv_bfloat16, 1>(const __nv_bfloat16 *p, float (&v)[1]) {
    v[0] = __bfloat162float(*p);
}
template <>
__device__ __forceinline__ void row_load<__half, 1>(const __half *p, float (&v)[1]) {
    v[0] = __half2float(*p);
}

template <>
__device__ __forceinline__ void row_load<__nv_bfloat16, 4>(const __nv_bfloat16 *p, float (&v)[4]) {
    const uint2 r = __ldg(reinterpret_cast<const uint2 *>(p));
    v[0] = __uint_as_float(r.x << 16);
    v[1] = __uint_as_float(r.x & 0xFFFF0000u);
    v[2] = __uint_as_float(r.y << 16);
    v[3] = __uint_as_float(r.y & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ void row_load<__half, 4>(const __half *p, float (&v)[4]) {
    const uint2 r = __ldg(reinterpret_cast<const uint2 *>(p));
    __half2 a, b;
    memcpy(&a, &r.x, 4);
    memcpy(&b, &r.y, 4);
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}

// Four 16-bit elements as fp32 from an 8-byte load.
template <typename T>
__device__ __forceinline__ void row_load4(const T *p, float *v);
template <>
__device__ __forceinline__ void row_load4<__nv_bfloat16>(const __nv_bfloat16 *p, float *v) {
    const uint2 r = __ldg(reinterpret_cast<const uint2 *>(p));
    v[0] = __uint_as_float(r.x << 16);
    v[1] = __uint_as_float(r.x & 0xFFFF0000u);
    v[2] = __uint_as_float(r.y << 16);
    v[3] = __uint_as_float(r.y & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ void row_load4<__half>(const __half *p, float *v) {
    const uint2 r = __ldg(reinterpret_cast<const uint2 *>(p));
    __half2 a, b;
    memcpy(&a, &r.x, 4);
    memcpy(&b, &r.y, 4);
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}

template <typename T> __device__ __forceinline__ T round_to(float v);
template <> __device__ __forceinline__ float round_to<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 round_to<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half round_to<__half>(float v) { return __float2half_rn(v); }

#ifdef DCN_CHECK_BOUNDS
// Bounds-checked builds (compiled with DCN_CHECK_BOUNDS): the address `p`
// of `n` elements if they lie inside [lo, hi), else `lo` (a safe address)
// with `bad` set.  These kernels' entry points take no handle and so have
// no status word: a thread that met an access outside its tensor writes
// NaN into every output it owns instead, which the parity tests see.
template <typename T>
__device__ __forceinline__ T *checked_ptr(T *p, int n, const void *lo, const void *hi, bool &bad) {
    const char *c = reinterpret_cast<const char *>(p);
    if (c >= static_cast<const char *>(lo) && c + n * sizeof(T) <= static_cast<const char *>(hi))
        return p;
    bad = true;
    return static_cast<T *>(const_cast<void *>(lo));
}
// Whether the `n` fp32 elements at `p` lie inside [lo, hi); `bad` is set
// when they do not (the reduction is then skipped).
__device__ __forceinline__ bool checked_ok(const float *p, int n, const void *lo, const void *hi, bool &bad) {
    const char *c = reinterpret_cast<const char *>(p);
    const bool ok = c >= static_cast<const char *>(lo) && c + n * sizeof(float) <= static_cast<const char *>(hi);
    if (!ok) bad = true;
    return ok;
}
#define DCN_ROW(ptr, n) checked_ptr((ptr), (n), p.v_lo, p.v_hi, bad)
#define DCN_GROW_OK(ptr, n) checked_ok((ptr), (n), p.gv_lo, p.gv_hi, bad)
#define DCN_BAD_DECL bool bad = false
// every lane of the warp learns whether any lane met a bad access
#define DCN_BAD_SYNC bad = __any_sync(0xffffffffu, bad)
#define DCN_POISON(x) (bad ? __int_as_float(0x7fc00000) : (x))
#else
#define DCN_ROW(ptr, n) (ptr)
#define DCN_GROW_OK(ptr, n) true
#define DCN_BAD_DECL
#define DCN_BAD_SYNC
#define DCN_POISON(x) (x)
#endif

}  // namespace dcn
