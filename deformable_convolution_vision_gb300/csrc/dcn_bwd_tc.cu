// Backward pass on tensor cores: the column gradient, fused with the
// bilinear scatter into grad_x and the offset and mask sums.
//
// The column gradient gA[p, (k, c)] = sum_o grad_out[p, o] * W[o, c, k] is a
// dense GEMM [P x O] x [O x kh*kw*C] (the chain rule of the forward's
// contraction, page "deformops 3.0.1", section "Deformable convolution":
// fp32 accumulation, no TF32).  Its [P x K] result -- as large as the
// im2col buffer the forward avoids -- is never written to memory: each
// 128 x 64 block of it lives in tensor memory only until the epilogue warps
// have turned it into grad_x, grad_offset and grad_mask contributions.
//
// A tile is 8 x 16 output pixels of one image (the forward's tile); a unit
// is one (tap, 64-channel block) of it.  One CTA per SM, persistent over
// tiles:
//   warp 0      TMA producer: the tile's grad_out block [128 x O] once per
//               tile (A operand, 128-byte swizzle, K = O), then for every
//               unit the packed weight rows [64 channels x 64 outputs] of
//               each 64-output K-block (B operand) into a ring of stages;
//               also allocates/frees TMEM.
//   warp 1      MMA issuer: M = 128, N = 64, K = 16 tcgen05.mma, both
//               operands from shared memory, into one of four fp32
//               accumulators of 64 columns.
//   warps 2-17  epilogue, two teams of eight taking alternate units.  A
//               warp owns 16 pixels of a tile row: it reads their 64
//               column-gradient values (16x256b: each lane two pixels x 16
//               channels), releases the accumulator, computes the pixels'
//               sampling geometry, loads the four corners (32-byte loads,
//               four lanes per 128-byte corner row), adds gA * m * w_corner
//               into grad_x by 16-byte vector reductions and the sums of
//               gA * m * dS/dpy, gA * m * dS/dpx and gA * S over its
//               channels into grad_offset and grad_mask.
// Every barrier wait is bounded; one that runs out sets the status word and
// the kernel winds down without trapping.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dcn_attr_cache.h"
#include "dcn_device.cuh"
#include "dcn_backward.h"
#include "dcn_kernels.h"

namespace dcn {

namespace {

// Bounds-checked builds check each global access of the kernels below
// against its tensor's byte range (recording a miss in the status word and
// skipping the access); other builds take every access as it is.
#ifdef DCN_CHECK_BOUNDS
#define BWD_IN(ptr, bytes, lo, hi) in_bounds((ptr), (bytes), (lo), (hi), p.status)
#else
#define BWD_IN(ptr, bytes, lo, hi) true
#endif

constexpr int BT_BM = 128;                  // pixels per tile (MMA M)
constexpr int BT_BN = 64;                   // channels per unit (MMA N)
constexpr int BT_BK = 64;                   // outputs per K-block
constexpr int BT_TILE_W = 16, BT_TILE_H = 8;
constexpr int BT_TEAM_WARPS = 8;
constexpr int BT_EPI_WARPS = 2 * BT_TEAM_WARPS;
constexpr int BT_THREADS = 32 * (2 + BT_EPI_WARPS);
constexpr int BT_ACC = 4;                   // fp32 accumulators of BT_BN columns
constexpr int BT_STAGES = 8;                // weight stages of BT_BN x BT_BK
constexpr int BT_A_KB_BYTES = BT_BM * BT_BK * 2;        // 16 KB
constexpr int BT_B_BYTES = BT_BN * BT_BK * 2;           // 8 KB

struct BtLayout {
    int a_off, b_off, bar_off, total;
};

__host__ __device__ inline BtLayout bt_layout(int O) {
    BtLayout L;
    L.a_off = 0;
    L.b_off = (O / BT_BK) * BT_A_KB_BYTES;
    L.bar_off = L.b_off + BT_STAGES * BT_B_BYTES;
    // b_full[S], b_empty[S], a_full, a_empty, acc_full[4], acc_free[4], tmem slot
    L.total = L.bar_off + (2 * BT_STAGES + 2 + 2 * BT_ACC + 1) * 8;
    return L;
}

template <bool kF16>
__global__ void __launch_bounds__(BT_THREADS, 1)
dcn_bwd_data_tc_kernel(const __grid_constant__ CUtensorMap gmap,
                       const __grid_constant__ CUtensorMap wmap, BwdParams p) {
    using E = Elem16<kF16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const BtLayout L = bt_layout(p.O);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    const uint32_t b_full0 = smem_u32(bars);
    const uint32_t b_empty0 = smem_u32(bars + BT_STAGES);
    const uint32_t a_full = smem_u32(bars + 2 * BT_STAGES);
    const uint32_t a_empty = smem_u32(bars + 2 * BT_STAGES + 1);
    const uint32_t acc_full0 = smem_u32(bars + 2 * BT_STAGES + 2);
    const uint32_t acc_free0 = smem_u32(bars + 2 * BT_STAGES + 2 + BT_ACC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * BT_STAGES + 2 + 2 * BT_ACC);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x / 32), 0);
    const int lane = threadIdx.x % 32;
    const int tiles_x = (p.Wo + BT_TILE_W - 1) / BT_TILE_W;
    const int tiles_y = (p.Ho + BT_TILE_H - 1) / BT_TILE_H;
    const int tiles = p.B * tiles_x * tiles_y;
    const int taps = p.kh * p.kw;
    const int ncb = p.C / BT_BN;
    const int units = taps * ncb;               // per tile
    const int nkb = p.O / BT_BK;
    const uint32_t tmem_cols = BT_ACC * BT_BN;  // 256

    if (threadIdx.x == 0) {
        for (int s = 0; s < BT_STAGES; ++s) {
            mbar_init(b_full0 + 8 * s, 1);
            mbar_init(b_empty0 + 8 * s, 1);
        }
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int b = 0; b < BT_ACC; ++b) {
            mbar_init(acc_full0 + 8 * b, 1);
            mbar_init(acc_free0 + 8 * b, BT_TEAM_WARPS);
        }
        fence_barrier_init();
    }
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    }
    if (warp == 1 && lane == 0) {
        tma_prefetch_desc(&gmap);
        tma_prefetch_desc(&wmap);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0, n_a = 0, issued = 0;
            uint32_t phase = 0;
            bool live = true;
            for (int tile = blockIdx.x; live && tile < tiles; tile += gridDim.x, ++n_a) {
                const int tb = tile / (tiles_x * tiles_y);
                const int trem = tile - tb * tiles_x * tiles_y;
                const int th0 = (trem / tiles_x) * BT_TILE_H;
                const int tw0 = (trem % tiles_x) * BT_TILE_W;
                // the previous tile's MMAs have read the A region
                if (n_a > 0 && !mbar_wait_sleep(a_empty, (n_a - 1) & 1, p.status, p.timeout_ns)) break;
                mbar_arrive_expect_tx(a_full, nkb * BT_A_KB_BYTES);
                for (int kb = 0; kb < nkb; ++kb)
                    tma_load_4d(smem_u32(smem + L.a_off + kb * BT_A_KB_BYTES), &gmap, a_full,
                                kb * BT_BK, tw0, th0, tb);
                for (int u = 0; live && u < units; ++u) {
                    const int tap = u / ncb, cb = u - (u / ncb) * ncb;
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait_sleep(b_empty0 + 8 * s, phase ^ 1, p.status, p.timeout_ns)) {
                            live = false;
                            break;
                        }
                        mbar_arrive_expect_tx(b_full0 + 8 * s, BT_B_BYTES);
                        tma_load_2d(smem_u32(smem + L.b_off + s * BT_B_BYTES), &wmap, b_full0 + 8 * s,
                                    kb * BT_BK, tap * p.C + cb * BT_BN);
                        ++issued;
                        if (++s == BT_STAGES) { s = 0; phase ^= 1; }
                    }
                }
            }
            // every copy this CTA started must land before it exits
            const int first = issued > BT_STAGES ? issued - BT_STAGES : 0;
            for (int i = first; i < issued; ++i)
                mbar_wait_sleep(b_full0 + 8 * (i % BT_STAGES), (i / BT_STAGES) & 1, p.status,
                                p.timeout_ns);
            if (n_a > 0) mbar_wait_sleep(a_full, (n_a - 1) & 1, p.status, p.timeout_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = E::idesc(BT_BM, BT_BN);
            int s = 0, n_a = 0, gu = 0;
            uint32_t phase = 0;
            bool live = true;
            for (int tile = blockIdx.x; live && tile < tiles; tile += gridDim.x, ++n_a) {
                if (!mbar_wait_sleep(a_full, n_a & 1, p.status, p.timeout_ns)) break;
                tc_fence_after_sync();
                const uint64_t a_desc0 = smem_desc_sw128(smem_u32(smem + L.a_off));
                for (int u = 0; live && u < units; ++u, ++gu) {
                    const int b = gu % BT_ACC, n = gu / BT_ACC;
                    if (n > 0 && !mbar_wait_sleep(acc_free0 + 8 * b, (n - 1) & 1, p.status, p.timeout_ns)) {
                        live = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + b * BT_BN;
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait_sleep(b_full0 + 8 * s, phase, p.status, p.timeout_ns)) {
                            live = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint64_t b_desc = smem_desc_sw128(smem_u32(smem + L.b_off + s * BT_B_BYTES));
                        const uint64_t a_desc = a_desc0 + ((kb * BT_A_KB_BYTES) >> 4);
#pragma unroll
                        for (int ks = 0; ks < BT_BK / 16; ++ks)
                            mma_kind_f16_ss(d_tmem, a_desc + 2 * ks, b_desc + 2 * ks, idesc,
                                            (kb > 0 || ks > 0) ? 1u : 0u);
                        mma_commit(b_empty0 + 8 * s);
                        if (++s == BT_STAGES) { s = 0; phase ^= 1; }
                    }
                    if (!live) break;
                    mma_commit(acc_full0 + 8 * b);
                }
                // the A region is free once this tile's MMAs are complete
                mma_commit(a_empty);
            }
            // every MMA must be complete before TMEM is released
            if (gu > 0) {
                const int last = gu - 1;
                mbar_wait_sleep(acc_full0 + 8 * (last % BT_ACC), (last / BT_ACC) & 1, p.status,
                                p.timeout_ns);
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int ew = warp - 2;                         // 0 .. 15
        const int team = ew / BT_TEAM_WARPS;             // takes units team, team + 2, ...
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const int half = (ew % BT_TEAM_WARPS) / 4;       // which 16 lanes of the quarter
        const int trow = 2 * q + half;                   // tile row = pixels 16 trow .. +15
        const int quart = lane & 3;                      // channels 16 quart .. +15 of the block
        const int rsub = lane >> 2;                      // pixels rsub and rsub + 8 of the row
        const uint32_t lane_addr = static_cast<uint32_t>(16 * trow) << 16;
        const uint16_t *__restrict__ x = static_cast<const uint16_t *>(p.x);
        const int HoWo = p.Ho * p.Wo;
        bool ok = true;
        int gu = 0;
        for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
            const int tb = tile / (tiles_x * tiles_y);
            const int trem = tile - tb * tiles_x * tiles_y;
            const int oh = (trem / tiles_x) * BT_TILE_H + trow;
            const int ow0 = (trem % tiles_x) * BT_TILE_W;
            for (int u = 0; u < units; ++u, ++gu) {
                if ((gu & 1) != team) continue;
                const int b = gu % BT_ACC;
                const bool got = mbar_wait_sleep(acc_full0 + 8 * b, (gu / BT_ACC) & 1, p.status,
                                                 p.timeout_ns, 2000u);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                tc_fence_after_sync();
                float ga[32];
                tmem_ld_16x256b_x8(tmem_base + lane_addr + b * BT_BN, ga);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_free0 + 8 * b);

                const int tap = u / ncb, cb = u - (u / ncb) * ncb;
                const int i = tap / p.kw, j = tap - (tap / p.kw) * p.kw;
                const int c0 = cb * BT_BN + 16 * quart;          // this lane's 16 channels
                const int q_off = c0 / (p.C / p.ogroups);       // offset group of the block
#pragma unroll
                for (int px = 0; px < 2; ++px) {
                    const int ow = ow0 + rsub + 8 * px;
                    const bool valid = oh < p.Ho && ow < p.Wo;
                    float gm = 0.0f, gdy = 0.0f, gdx = 0.0f, m = 0.0f;
                    size_t hw = 0, bq = 0;
                    if (valid) {
                        hw = static_cast<size_t>(oh) * p.Wo + ow;
                        bq = static_cast<size_t>(tb) * p.ogroups + q_off;
                        const float *pdy = p.offset + (bq * 2 * taps + 2 * tap) * HoWo + hw;
                        const float *pdx = pdy + HoWo;
                        const float *pm = p.mask ? p.mask + (bq * taps + tap) * HoWo + hw : nullptr;
                        const float dy = BWD_IN(pdy, 4, p.off_lo, p.off_hi) ? __ldg(pdy) : 0.0f;
                        const float dx = BWD_IN(pdx, 4, p.off_lo, p.off_hi) ? __ldg(pdx) : 0.0f;
                        m = !pm ? 1.0f : (BWD_IN(pm, 4, p.mask_lo, p.mask_hi) ? __ldg(pm) : 0.0f);
                        float py = static_cast<float>(oh * p.sh - p.ph + i * p.dh) + dy;
                        float pxf = static_cast<float>(ow * p.sw - p.pw + j * p.dw) + dx;
                        py = fminf(fmaxf(py, -2.0f), static_cast<float>(p.H + 1));
                        pxf = fminf(fmaxf(pxf, -2.0f), static_cast<float>(p.W + 1));
                        const float fy = floorf(py), fx = floorf(pxf);
                        const float ly = py - fy, lx = pxf - fx;
                        const int y0 = static_cast<int>(fy), x0 = static_cast<int>(fx);
                        const float wy[2] = {1.0f - ly, ly};
                        const float wx[2] = {1.0f - lx, lx};
                        // the four corners' 16 channels (packed pairs), zero outside
                        u32x8 raw[4];
                        bool in[4];
                        size_t cidx[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int yy = y0 + (k >> 1), xx = x0 + (k & 1);
                            in[k] = static_cast<unsigned>(yy) < static_cast<unsigned>(p.H) &&
                                    static_cast<unsigned>(xx) < static_cast<unsigned>(p.W);
                            cidx[k] = in[k] ? (static_cast<size_t>((tb * p.H + yy) * p.W + xx)) * p.C + c0 : 0;
                            if (in[k] && BWD_IN(x + cidx[k], 32, p.x_lo, p.x_hi)) {
                                raw[k] = ldg_v8(x + cidx[k]);
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) raw[k].w[e] = 0u;
                            }
                        }
                        // four channels at a time: sample, derivatives, sums, scatter
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            float sc[4][4];
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int e = 4 * e4 + t;       // channel c0 + e
                                const int wd = e >> 1;          // its packed word
                                float v[4];
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    v[k] = (e & 1) ? E::hi(raw[k].w[wd]) : E::lo(raw[k].w[wd]);
                                // register of channel e: 4 (e / 2) + (e % 2), + 2 for the second pixel
                                const float g = ga[4 * (e >> 1) + (e & 1) + 2 * px];
                                const float S = wy[0] * (wx[0] * v[0] + wx[1] * v[1]) +
                                                wy[1] * (wx[0] * v[2] + wx[1] * v[3]);
                                const float sy = wx[0] * (v[2] - v[0]) + wx[1] * (v[3] - v[1]);
                                const float sx = wy[0] * (v[1] - v[0]) + wy[1] * (v[3] - v[2]);
                                gm = fmaf(g, S, gm);
                                gdy = fmaf(g, sy, gdy);
                                gdx = fmaf(g, sx, gdx);
                                const float gmm = g * m;
                                sc[0][t] = gmm * wy[0] * wx[0];
                                sc[1][t] = gmm * wy[0] * wx[1];
                                sc[2][t] = gmm * wy[1] * wx[0];
                                sc[3][t] = gmm * wy[1] * wx[1];
                            }
                            // (a tap whose mask is exactly 0 adds nothing to grad_x:
                            // its reductions are skipped)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                if (in[k] && m != 0.0f && BWD_IN(p.grad_x + cidx[k] + 4 * e4, 16, p.gx_lo, p.gx_hi))
                                    red_add_v4_f32(p.grad_x + cidx[k] + 4 * e4, sc[k][0], sc[k][1],
                                                   sc[k][2], sc[k][3]);
                        }
                    }
                    // the four lanes of a pixel hold its 64 channels
                    gm += __shfl_xor_sync(0xffffffffu, gm, 1);
                    gdy += __shfl_xor_sync(0xffffffffu, gdy, 1);
                    gdx += __shfl_xor_sync(0xffffffffu, gdx, 1);
                    gm += __shfl_xor_sync(0xffffffffu, gm, 2);
                    gdy += __shfl_xor_sync(0xffffffffu, gdy, 2);
                    gdx += __shfl_xor_sync(0xffffffffu, gdx, 2);
                    if (valid && quart == 0) {
                        float *gdy_p = p.grad_offset + (bq * 2 * taps + 2 * tap) * HoWo + hw;
                        float *gdx_p = gdy_p + HoWo;
                        if (BWD_IN(gdy_p, 4, p.goff_lo, p.goff_hi)) atomicAdd(gdy_p, gdy * m);
                        if (BWD_IN(gdx_p, 4, p.goff_lo, p.goff_hi)) atomicAdd(gdx_p, gdx * m);
                        if (p.grad_mask) {
                            float *gm_p = p.grad_mask + (bq * taps + tap) * HoWo + hw;
                            if (BWD_IN(gm_p, 4, p.gmask_lo, p.gmask_hi)) atomicAdd(gm_p, gm);
                        }
                    }
                }
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

// S0 of the backward: weight [O, C, kh, kw] -> [kh*kw*C][O] with the
// channels of each 64-block in bwd_channel_perm order.  One thread per
// output o (coalesced writes), one block row per packed row.
__global__ void pack_weight_bwd_kernel(const uint16_t *__restrict__ w, uint16_t *__restrict__ wt,
                                       int O, int C, int kh, int kw) {
    const int row = blockIdx.x;                 // tap * C + c'
    const int taps = kh * kw;
    const int tap = row / C;
    const int c = bwd_channel_perm(row - tap * C);
    for (int o = threadIdx.x + blockIdx.y * blockDim.x; o < O; o += blockDim.x * gridDim.y)
        wt[static_cast<size_t>(row) * O + o] = w[(static_cast<size_t>(o) * C + c) * taps + tap];
}

// the dynamic shared-memory limit set on each device, per operand type
PerDeviceValue<> g_bwd_smem_set[2];

}  // namespace

bool bwd_tc_supported(int C, int O, int groups, int offset_groups) {
    if (groups != 1 || C % BT_BN != 0 || O % BT_BK != 0 || O > 256 || O < BT_BK) return false;
    if (offset_groups <= 0 || C % offset_groups != 0) return false;
    return (C / offset_groups) % BT_BN == 0;
}

cudaError_t launch_pack_weight_bwd(const void *weight, void *wpack_t, int O, int C, int kh,
                                   int kw, cudaStream_t stream) {
    if (C % 64 != 0) return cudaErrorInvalidValue;
    const long long rows = static_cast<long long>(kh) * kw * C;
    if (rows > 2147483647ll) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(rows), (O + 255) / 256 < 65535 ? (O + 255) / 256 : 65535);
    pack_weight_bwd_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t *>(weight),
                                                     static_cast<uint16_t *>(wpack_t), O, C, kh, kw);
    return cudaGetLastError();
}

cudaError_t launch_bwd_data_tc(const BwdParams &p, const CUtensorMap &gmap,
                               const CUtensorMap &wmap, cudaStream_t stream) {
    const BtLayout L = bt_layout(p.O);
    const int smem = L.total + 1024;
    auto kernel = p.f16 ? dcn_bwd_data_tc_kernel<true> : dcn_bwd_data_tc_kernel<false>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = static_cast<cudaError_t>(g_bwd_smem_set[p.f16 ? 1 : 0].ensure(dev, smem, [&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    }));
    if (e != cudaSuccess) return e;
    const int tiles = p.B * ((p.Ho + BT_TILE_H - 1) / BT_TILE_H) * ((p.Wo + BT_TILE_W - 1) / BT_TILE_W);
    const int grid = tiles < p.sm_count ? tiles : p.sm_count;
    kernel<<<grid, BT_THREADS, smem, stream>>>(gmap, wmap, p);
    return cudaGetLastError();
}

}  // namespace dcn
