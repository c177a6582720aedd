// Device helpers shared by the sm_103a kernels: inline PTX for mbarriers,
// TMA, tcgen05 (TMEM allocation, MMA, commit, loads) and the bounded wait
// used everywhere a thread spins on a barrier.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace dcn {

// Bits of the handle's device status word.
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBounds = 2u;   // bounds-checked builds only

#ifdef DCN_CHECK_BOUNDS
// Bounds-checked builds (compiled with DCN_CHECK_BOUNDS): whether the bytes
// [p, p + bytes) lie inside [lo, hi).  An access outside sets kStatusBounds
// in *status and the caller skips it (or reads a safe address instead);
// nothing traps.
__device__ __forceinline__ bool in_bounds(const void *p, size_t bytes, const void *lo,
                                          const void *hi, unsigned *status) {
    const char *c = static_cast<const char *>(p);
    const bool ok = c >= static_cast<const char *>(lo) && c + bytes <= static_cast<const char *>(hi);
    if (!ok) atomicOr(status, kStatusBounds);
    return ok;
}
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// As mbar_try_wait, but lets the hardware suspend the thread for up to
// `hint_ns` while the phase is incomplete instead of returning at once:
// threads that only wait (the MMA issuer, the TMA producer) then stop
// competing for issue slots with the threads doing work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}

// Bounded wait that sleeps (up to hint_ns per try) instead of spinning.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity,
                                                unsigned *status, uint64_t limit_ns,
                                                uint32_t hint_ns = 20000u) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, hint_ns)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Wait until the phase with the given parity has completed, for at most
// `limit_ns` nanoseconds of global time.  On running out it sets the
// timeout bit in *status and returns false; it never traps or spins
// forever.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned *status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0u && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 256-bit read-only global load (sm_100 family); `p` must be 32-byte aligned.
struct u32x8 { uint32_t w[8]; };
__device__ __forceinline__ u32x8 ldg_v8(const void *p) {
    u32x8 v;
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
    return v;
}

// Vector shared-memory accesses (one instruction each).
__device__ __forceinline__ int4 lds_v4_s32(uint32_t addr) {
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void lds_v2_u64(uint32_t addr, uint64_t &a, uint64_t &b) {
    asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}
__device__ __forceinline__ void sts_v4_b32(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                           uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d));
}
// (with a memory clobber: kept in order with the warp barriers around
// the per-warp tables they write and read)
__device__ __forceinline__ void sts_b32(uint32_t addr, uint32_t a) {
    asm volatile("st.shared.b32 [%0], %1;" :: "r"(addr), "r"(a) : "memory");
}
__device__ __forceinline__ void sts_v4_b32_m(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ int lds_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ int4 lds_v4_s32_m(uint32_t addr) {
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void sts_v2_b32_m(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" :: "r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ uint2 lds_v2_u32(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 lds_v4_f32(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}

// Asynchronous 4-byte global -> shared copy; with valid == false nothing
// is read and the destination is zero-filled.  The thread's copies are
// complete after cp_async_wait_all.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                 :: "r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Barrier over `count` threads (a multiple of 32) of the CTA, id 1..15.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled TMA load of box (c0, c1) into shared memory, completing bytes
// on the mbarrier.  c0 is the innermost coordinate, in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 4-D tiled TMA load of box (c0, c1, c2, c3), innermost first, into shared
// memory, completing bytes on the mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
           "r"(bar)
        : "memory");
}

// ----------------------------------------------------------------- tcgen05

// Allocate `ncols` TMEM columns (a power of two >= 32); the whole warp must
// call it.  The TMEM address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4 (unused for this layout)
//   bits 32-45 stride-dimension byte offset >> 4 (1024 bytes)
//   bits 46-47 descriptor version (1 on sm_100-family)
//   bits 49-51 base offset (0: atoms are 1024-byte aligned)
//   bits 61-63 layout (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B (both
// K-major), fp32 accumulator, shape M x N.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format
//   (1 = bf16), 15/16 A/B major (0 = K), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
// The same with fp16 A and B (format 0).
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
    return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_kind_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread.  A occupies TMEM
// lanes 0..M-1 (row m in lane m) and K/2 columns from a_tmem, two 16-bit values per
// 32-bit column, the even k in the low half.
__device__ __forceinline__ void mma_kind_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Store 16 lanes x 32 columns from a warp (shape 16x256b, four repeats of
// 8 columns).  Thread t writes, in repeat r, r[4r], r[4r+1] to lane
// taddr.lane + t/4, columns 8r + 2(t%4) + {0, 1}, and r[4r+2], r[4r+3] to
// lane taddr.lane + 8 + t/4, the same columns.
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
           "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
           "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// One repeat of the same shape: 16 lanes x 8 columns, r[0], r[1] to lane
// taddr.lane + t/4, columns 2(t%4) + {0, 1}, and r[2], r[3] to lane
// taddr.lane + 8 + t/4, the same columns.
__device__ __forceinline__ void tmem_st_16x256b_x1(uint32_t taddr, uint32_t r0, uint32_t r1, uint32_t r2,
                                                   uint32_t r3) {
    asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1,%2,%3,%4};"
                 :: "r"(taddr), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}

// Load 16 lanes x 64 columns (shape 16x256b, eight repeats of 8 columns):
// the layout of tmem_st_16x256b_x4 over twice the columns.  Thread t gets,
// in repeat r, r[4r], r[4r+1] from lane taddr.lane + t/4, columns
// 8r + 2(t%4) + {0, 1}, and r[4r+2], r[4r+3] from lane taddr.lane + 8 + t/4,
// the same columns.  Followed by tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
          "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Vector reduction (add) of four fp32 values into 16-byte aligned global memory.
__device__ __forceinline__ void red_add_v4_f32(float *p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// This thread's earlier tcgen05.st have completed.
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread has
// issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        :: "r"(bar) : "memory");
}

// Load 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ numbers


__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Packed fp32 pairs (two lanes of one 64-bit register) for the sm_100-family
// f32x2 FMA pipe: each op is exactly two independent fp32 operations.
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// Round a packed fp32 pair to a bf16x2 word (lo in the low half).
__device__ __forceinline__ uint32_t f2_to_bf16x2(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return pack_bf16x2(lo, hi);
}
// The same rounding to an fp16x2 word.
__device__ __forceinline__ uint32_t f2_to_f16x2(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// bf16x2 arithmetic on 32-bit words (low half = first element); each op
// rounds once, to nearest even.
__device__ __forceinline__ uint32_t bf16x2_splat(float v) {
    __nv_bfloat162 r = __float2bfloat162_rn(v);
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// A 32-bit word with its low (high) 16-bit half in both halves.
__device__ __forceinline__ uint32_t splat_lo(uint32_t w) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %1, 0x1010;" : "=r"(d) : "r"(w));
    return d;
}
__device__ __forceinline__ uint32_t splat_hi(uint32_t w) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %1, 0x3232;" : "=r"(d) : "r"(w));
    return d;
}

// The two bf16 halves of a 32-bit word as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp16x2 counterparts (low half = first element; one rounding per op).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t f16x2_splat(float v) {
    __half2 r = __float2half2_rn(v);
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t f16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ float f16_lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// The 16-bit operand type of the tensor-core path: bf16 or fp16.  Both
// feed tcgen05.mma kind::f16 (A and B of one type) with fp32 accumulation.
template <bool kF16> struct Elem16;
template <> struct Elem16<false> {   // bf16
    __device__ static uint32_t splat(float v) { return bf16x2_splat(v); }
    __device__ static uint32_t mul(uint32_t a, uint32_t b) { return bf16x2_mul(a, b); }
    __device__ static uint32_t fma(uint32_t a, uint32_t b, uint32_t c) { return bf16x2_fma(a, b, c); }
    __device__ static float lo(uint32_t w) { return bf16_lo(w); }
    __device__ static float hi(uint32_t w) { return bf16_hi(w); }
    __device__ static uint32_t pack(float lo, float hi) { return pack_bf16x2(lo, hi); }
    __device__ static uint32_t pack_f2(uint64_t v) { return f2_to_bf16x2(v); }
    __host__ __device__ static constexpr uint32_t idesc(uint32_t M, uint32_t N) { return idesc_bf16_f32(M, N); }
};
template <> struct Elem16<true> {    // fp16
    __device__ static uint32_t splat(float v) { return f16x2_splat(v); }
    __device__ static uint32_t mul(uint32_t a, uint32_t b) { return f16x2_mul(a, b); }
    __device__ static uint32_t fma(uint32_t a, uint32_t b, uint32_t c) { return f16x2_fma(a, b, c); }
    __device__ static float lo(uint32_t w) { return f16_lo(w); }
    __device__ static float hi(uint32_t w) { return f16_hi(w); }
    __device__ static uint32_t pack(float lo, float hi) { return pack_f16x2(lo, hi); }
    __device__ static uint32_t pack_f2(uint64_t v) { return f2_to_f16x2(v); }
    __host__ __device__ static constexpr uint32_t idesc(uint32_t M, uint32_t N) { return idesc_f16_f32(M, N); }
};

}  // namespace dcn
