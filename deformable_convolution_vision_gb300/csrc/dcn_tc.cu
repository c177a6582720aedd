// tcgen05 fused implicit-GEMM forward kernel (bf16 operands, fp32 TMEM
// accumulation) for sm_103a.
//
// The contraction out[p, o] = sum_K A[p, K] * Wp[o, K] with K = (tap, c) is
// a dense GEMM whose A operand is never materialised: the im2col column
// buffer that page "deformops 3.0.1" (section "Deformable convolution")
// avoids, and that the "birefnet-lite-1024-webgpu patch_deform.py" page
// sizes at 392 MB for the 7x7, C = 64, 256 x 256 layer, exists here only as
// one 128 x 64 tile per pipeline stage in shared memory.
//
// One CTA computes a tile of 128 consecutive output pixels (flattened
// b, h, w) x all O output channels:
//   warp 0      TMA producer: the packed-weight K-block [O x 64] of each
//               stage, 128-byte swizzle; also allocates/frees TMEM.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=O,
//               K=16) x 4 per K-block, accumulating in TMEM, and commits
//               each stage back to its "empty" barrier.
//   warps 2..9  samplers: per (pixel, tap) the corner weights and
//               addresses (S1, S2), then for 8 channels per lane the four
//               16-byte corner loads, the fp32 bilinear combine, a bf16
//               round and one 16-byte store into the swizzled A stage (S3).
//               After the last K-block they run the epilogue (S5): TMEM ->
//               registers, + bias in fp32, bf16 round, channels-last store.
// K-blocks run tap-major with 64 channels each, so a tap's corner geometry
// is computed once and reused for all of its channel blocks.
// Every barrier wait is bounded; a wait that runs out sets the status word
// and the kernel winds down without trapping.
#include <cuda_bf16.h>

#include "dcn_device.cuh"
#include "dcn_kernels.h"
#include "dcn_sampling.cuh"

namespace dcn {

namespace {

constexpr int TC_BM = 128;               // output pixels per tile (MMA M)
constexpr int TC_BK = 64;                // channels per K-block (128 bytes)
constexpr int TC_SAMPLER_WARPS = 8;
constexpr int TC_THREADS = 32 * (2 + TC_SAMPLER_WARPS);
constexpr int TC_ROWS_PER_WARP = TC_BM / TC_SAMPLER_WARPS;   // 16
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;                // 16 KB
constexpr int TC_MMA_K = 16;

struct TcLayout {
    int stages;
    int b_bytes;       // O * 128
    int stage_bytes;   // A + B
    int bar_off;       // barriers after the stages
    int table_off;     // per-warp corner tables
    int total;         // bytes used from the 1024-aligned base
};

__host__ __device__ inline TcLayout tc_layout(int O, int stages) {
    TcLayout L;
    L.stages = stages;
    L.b_bytes = O * TC_BK * 2;
    L.stage_bytes = TC_A_BYTES + L.b_bytes;
    L.bar_off = stages * L.stage_bytes;
    // full[stages], empty[stages], accum_full, tmem slot (8 bytes each)
    L.table_off = L.bar_off + (2 * stages + 2) * 8;
    L.table_off = (L.table_off + 15) & ~15;
    L.total = L.table_off + TC_SAMPLER_WARPS * TC_ROWS_PER_WARP * 32;
    return L;
}

__host__ __device__ inline int tmem_cols_for(int O) {
    int n = 32;
    while (n < O) n <<= 1;
    return n;
}

__global__ void __launch_bounds__(TC_THREADS, 2)
dcn_tc_kernel(const __grid_constant__ CUtensorMap wmap, Params p, int stages) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const TcLayout L = tc_layout(p.O, stages);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + stages);
    const uint32_t accum_bar = smem_u32(bars + 2 * stages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int tile0 = blockIdx.x * TC_BM;
    const int ncb = p.C / TC_BK;
    const int taps = p.kh * p.kw;
    const int nkb = taps * ncb;
    const int tmem_cols = tmem_cols_for(p.O);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1 + TC_SAMPLER_WARPS);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(accum_bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    }
    if (warp == 1 && lane == 0) tma_prefetch_desc(&wmap);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % stages;
                const uint32_t r = kb / stages;
                if (!mbar_wait(empty0 + 8 * s, (r & 1) ^ 1, p.status, p.timeout_ns)) break;
                const uint32_t b_dst = smem_u32(smem + s * L.stage_bytes + TC_A_BYTES);
                mbar_arrive_expect_tx(full0 + 8 * s, L.b_bytes);
                tma_load_2d(b_dst, &wmap, full0 + 8 * s, kb * TC_BK, 0);
                ++issued;
            }
            // Before the CTA can exit, every weight copy it started must
            // have landed: wait (bounded) for the last phase of each stage.
            const int first = issued > stages ? issued - stages : 0;
            for (int kb = first; kb < issued; ++kb) {
                const int s = kb % stages;
                mbar_wait(full0 + 8 * s, (kb / stages) & 1, p.status, p.timeout_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(TC_BM, p.O);
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % stages;
                const uint32_t r = kb / stages;
                if (!mbar_wait(full0 + 8 * s, r & 1, p.status, p.timeout_ns)) break;
                tc_fence_after_sync();
                const uint32_t a_addr = smem_u32(smem + s * L.stage_bytes);
                const uint32_t b_addr = a_addr + TC_A_BYTES;
                const uint64_t adesc = smem_desc_sw128(a_addr);
                const uint64_t bdesc = smem_desc_sw128(b_addr);
#pragma unroll
                for (int ks = 0; ks < TC_BK / TC_MMA_K; ++ks) {
                    // advance the start address by 32 bytes per K=16 step
                    mma_bf16_ss(tmem_base, adesc + 2 * ks, bdesc + 2 * ks, idesc,
                                (kb | ks) != 0);
                }
                mma_commit(empty0 + 8 * s);
            }
            mma_commit(accum_bar);
            // the MMAs must be complete before TMEM is released
            mbar_wait(accum_bar, 0, p.status, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------ samplers
        const int sw = warp - 2;
        const __nv_bfloat16 *__restrict__ x = static_cast<const __nv_bfloat16 *>(p.x);
        float4 *cw_tab = reinterpret_cast<float4 *>(smem + L.table_off) + sw * TC_ROWS_PER_WARP * 2;
        int4 *ci_tab = reinterpret_cast<int4 *>(cw_tab + TC_ROWS_PER_WARP);
        const int HoWo = p.Ho * p.Wo;

        // lanes 0..15 own the geometry of rows sw*16 + lane
        const int my_row = sw * TC_ROWS_PER_WARP + (lane & 15);
        const int my_pix = tile0 + my_row;
        const bool my_valid = (lane < 16) && (my_pix < p.P);
        int my_b = 0, my_h = 0, my_w = 0;
        if (my_valid) {
            my_b = my_pix / HoWo;
            const int rem = my_pix - my_b * HoWo;
            my_h = rem / p.Wo;
            my_w = rem - my_h * p.Wo;
        }
        const size_t my_hw = static_cast<size_t>(my_h) * p.Wo + my_w;
        const float *off_base = p.offset + static_cast<size_t>(my_b) * 2 * taps * HoWo + my_hw;
        const float *mask_base = p.mask ? p.mask + static_cast<size_t>(my_b) * taps * HoWo + my_hw
                                        : nullptr;

        const int chunk = lane & 7;     // 8 channels = 16 bytes
        const int rsub = lane >> 3;     // 0..3
        bool ok = true;

        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % stages;
            const uint32_t r = kb / stages;
            const int tap = kb / ncb;
            const int cb = kb - tap * ncb;
            if (cb == 0) {
                __syncwarp();
                if (lane < 16) {
                    TapCorners t;
                    if (my_valid) {
                        const int i = tap / p.kw;
                        const int j = tap - i * p.kw;
                        const float dy = __ldg(off_base + static_cast<size_t>(2 * tap) * HoWo);
                        const float dx = __ldg(off_base + static_cast<size_t>(2 * tap + 1) * HoWo);
                        const float m = mask_base ? __ldg(mask_base + static_cast<size_t>(tap) * HoWo) : 1.0f;
                        tap_corners(dy, dx, m, my_h, my_w, i, j, p.pad, my_b, p.H, p.W, p.C, t);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) { t.w[q] = 0.0f; t.idx[q] = 0; }
                    }
                    cw_tab[lane] = make_float4(t.w[0], t.w[1], t.w[2], t.w[3]);
                    ci_tab[lane] = make_int4(t.idx[0], t.idx[1], t.idx[2], t.idx[3]);
                }
                __syncwarp();
            }
            // every lane waits; the warp leaves the loop together if any lane ran out
            const bool got = mbar_wait(empty0 + 8 * s, (r & 1) ^ 1, p.status, p.timeout_ns);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }

            uint8_t *a_stage = smem + s * L.stage_bytes;
            const __nv_bfloat16 *xc = x + cb * TC_BK + chunk * 8;
#pragma unroll
            for (int it = 0; it < TC_ROWS_PER_WARP / 4; ++it) {
                const int rl = it * 4 + rsub;
                const int row = sw * TC_ROWS_PER_WARP + rl;
                const float4 cw = cw_tab[rl];
                const int4 ci = ci_tab[rl];
                uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0, v2 = v0, v3 = v0;
                if (cw.x != 0.0f) v0 = __ldg(reinterpret_cast<const uint4 *>(xc + ci.x));
                if (cw.y != 0.0f) v1 = __ldg(reinterpret_cast<const uint4 *>(xc + ci.y));
                if (cw.z != 0.0f) v2 = __ldg(reinterpret_cast<const uint4 *>(xc + ci.z));
                if (cw.w != 0.0f) v3 = __ldg(reinterpret_cast<const uint4 *>(xc + ci.w));
                const uint32_t *w0 = reinterpret_cast<const uint32_t *>(&v0);
                const uint32_t *w1 = reinterpret_cast<const uint32_t *>(&v1);
                const uint32_t *w2 = reinterpret_cast<const uint32_t *>(&v2);
                const uint32_t *w3 = reinterpret_cast<const uint32_t *>(&v3);
                uint32_t packed[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float lo = cw.x * bf16_lo(w0[q]);
                    float hi = cw.x * bf16_hi(w0[q]);
                    lo = fmaf(cw.y, bf16_lo(w1[q]), lo);
                    hi = fmaf(cw.y, bf16_hi(w1[q]), hi);
                    lo = fmaf(cw.z, bf16_lo(w2[q]), lo);
                    hi = fmaf(cw.z, bf16_hi(w2[q]), hi);
                    lo = fmaf(cw.w, bf16_lo(w3[q]), lo);
                    hi = fmaf(cw.w, bf16_hi(w3[q]), hi);
                    packed[q] = pack_bf16x2(lo, hi);
                }
                // 128-byte swizzle: 16-byte chunk c of row r lives at chunk c ^ (r % 8)
                uint8_t *dst = a_stage + row * 128 + ((chunk ^ (row & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full0 + 8 * s);
        }

        // ------------------------------------------------ epilogue (S5)
        if (ok) ok = mbar_wait(accum_bar, 0, p.status, p.timeout_ns);
        __syncwarp();
        tc_fence_after_sync();
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int half = (warp - 2) >> 2;       // two warps per quarter split the columns
        const int row = q * 32 + lane;
        const int pix = tile0 + row;
        const int nch = p.O / 16;
        const int ch_begin = half == 0 ? 0 : nch / 2;
        const int ch_end = half == 0 ? nch / 2 : nch;
        __nv_bfloat16 *__restrict__ out = static_cast<__nv_bfloat16 *>(p.out);
        for (int ch = ch_begin; ch < ch_end; ++ch) {
            float v[16];
            tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ch * 16, v);
            if (ok && pix < p.P) {
                uint32_t packed[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int o = ch * 16 + 2 * e;
                    const float b0 = p.bias ? __ldg(p.bias + o) : 0.0f;
                    const float b1 = p.bias ? __ldg(p.bias + o + 1) : 0.0f;
                    packed[e] = pack_bf16x2(v[2 * e] + b0, v[2 * e + 1] + b1);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<size_t>(pix) * p.O + ch * 16);
                dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

int g_max_smem_set = 0;

}  // namespace

bool tc_supported(int C, int O) {
    return C % TC_BK == 0 && O % 16 == 0 && O >= 16 && O <= 256;
}

cudaError_t launch_tc(const Params &p, const CUtensorMap &wmap, cudaStream_t stream) {
    // Two CTAs per SM when the stages allow it, so one CTA's epilogue
    // overlaps the other's main loop.
    const int per_cta_budget = 113 * 1024;
    int stages = (per_cta_budget - 1024 - tc_layout(p.O, 0).total) / tc_layout(p.O, 1).stage_bytes;
    stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
    const TcLayout L = tc_layout(p.O, stages);
    const int smem = L.total + 1024;  // slack for 1024-byte alignment
    if (smem > g_max_smem_set) {
        cudaError_t e = cudaFuncSetAttribute(dcn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        g_max_smem_set = smem;
    }
    const int tiles = (p.P + TC_BM - 1) / TC_BM;
    dcn_tc_kernel<<<tiles, TC_THREADS, smem, stream>>>(wmap, p, stages);
    return cudaGetLastError();
}

// ------------------------------------------------------------ self-test

namespace {
__global__ void selftest_timeout_kernel(unsigned *status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
        // nothing ever arrives: the bounded wait must run out and report it
        mbar_wait(smem_u32(&bar), 0, status, limit_ns);
    }
}
}  // namespace

cudaError_t launch_selftest_timeout(unsigned *status, unsigned long long timeout_ns,
                                    cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace dcn
