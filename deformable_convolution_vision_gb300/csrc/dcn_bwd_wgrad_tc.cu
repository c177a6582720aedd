// Weight gradient of the backward pass on tensor cores.
//
// grad_weight[o, c, tap] = sum_p grad_out[p, o] * m_tap(p) * S_c(p, tap) is a
// dense GEMM over the pixels p: the chain rule of the forward's contraction
// (page "deformops 3.0.1", section "Deformable convolution": one kernel
// gathers and contracts, fp32 accumulation, no TF32).  The sampled operand
// m * S -- the forward's A operand, as large as the im2col buffer -- is never
// written to memory: each CTA samples one 128-pixel tile of it at a time
// into shared memory and contracts it at once.
//
// A CTA owns 128 rows of the (tap, channel) space -- two units of one tap
// and 64 channels -- and a contiguous run of 8 x 16 pixel tiles; its fp32
// accumulator D[128 x O] stays in tensor memory across the run and is added
// into grad_weight at the end.  Both MMA operands are pixel-contiguous
// (MN-major, K = pixels, 128-byte swizzle):
//   A  the sampled tile, [unit][pixel][64 channels]: the sampler warps write
//      each (pixel, unit) row of 64 channels as it comes from the corner
//      rows, so no transpose is needed;
//   B  the grad_out tile, [64-output block][pixel][64 outputs]: the 4-D TMA
//      box of the column-gradient kernel, channels-last as stored.
// Warp roles (18 warps, one CTA per SM):
//   warp 0      TMA producer of B, one tile per stage; allocates TMEM.
//   warp 1      MMA issuer: M = 128, N = O, K = 16 tcgen05.mma, eight per
//               tile, into one accumulator.
//   warps 2-17  samplers, two teams of eight taking alternate tiles.  A warp
//               owns one tile row (16 pixels): per unit each lane gathers
//               16 channels of two pixels (32-byte corner loads, four lanes
//               per 128-byte corner row), sums the four weighted corners in
//               fp32 with the mask folded into the weights, rounds once to
//               the operand type (as the forward's fp32 combine does) and
//               stores the two 16-byte chunks of each pixel into the
//               swizzled A stage.  After the run they read the accumulator
//               out and add it into grad_weight.
// Every barrier wait is bounded; one that runs out sets the status word and
// the kernel winds down without trapping.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dcn_attr_cache.h"
#include "dcn_device.cuh"
#include "dcn_backward.h"
#include "dcn_kernels.h"
#include "dcn_sampling.cuh"

namespace dcn {

namespace {

// Bounds-checked builds check each global access of the kernel below
// against its tensor's byte range (recording a miss in the status word and
// skipping the access, or reading a safe address instead); other builds
// take every access as it is.
#ifdef DCN_CHECK_BOUNDS
#define WG_IN(ptr, bytes, lo, hi) in_bounds((ptr), (bytes), (lo), (hi), p.status)
#else
#define WG_IN(ptr, bytes, lo, hi) true
#endif

constexpr int WG_UNIT = 64;                 // channels per unit (one 128-byte row)
constexpr int WG_BM = 2 * WG_UNIT;          // (tap, channel) rows per CTA (MMA M)
constexpr int WG_TILE_W = 16, WG_TILE_H = 8;
constexpr int WG_BK = WG_TILE_W * WG_TILE_H;   // pixels per stage (MMA K per stage)
constexpr int WG_TEAM_WARPS = 8;
constexpr int WG_SAMPLER_WARPS = 2 * WG_TEAM_WARPS;
constexpr int WG_THREADS = 32 * (2 + WG_SAMPLER_WARPS);
constexpr int WG_UNIT_BYTES = WG_BK * 128;     // one unit of A: 128 pixel rows of 128 bytes
constexpr int WG_A_BYTES = 2 * WG_UNIT_BYTES;  // 32 KB
constexpr int WG_BOX_BYTES = WG_BK * 128;      // one 64-output box of B
// per sampler warp: the table of its 16 pixels for both units, fp32 weights
// of the four slots then the slot (0,0) index (16 bytes each)
constexpr int WG_TABLE_WARP_BYTES = 2 * 2 * WG_TILE_W * 16;
constexpr int WG_RAW_WARP_BYTES = 3 * 32 * 4;  // dy, dx and m planes of 32 lanes

struct WgLayout {
    int stages, b_bytes, stage_bytes, table_off, raw_off, bar_off, total;
};

__host__ __device__ inline WgLayout wg_layout(int O, int stages) {
    WgLayout L;
    L.stages = stages;
    L.b_bytes = (O / 64) * WG_BOX_BYTES;
    L.stage_bytes = WG_A_BYTES + L.b_bytes;
    L.table_off = stages * L.stage_bytes;
    L.raw_off = L.table_off + WG_SAMPLER_WARPS * WG_TABLE_WARP_BYTES;
    L.bar_off = L.raw_off + WG_SAMPLER_WARPS * WG_RAW_WARP_BYTES;
    // full[stages], empty[stages], acc_full, tmem slot
    L.total = L.bar_off + (2 * stages + 2) * 8;
    return L;
}

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// rows of 64 elements (128 bytes) along M/N for one K index, eight K rows
// to a 1024-byte swizzle atom; lbo = bytes between atoms along M/N, sbo =
// bytes between atoms along K.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

template <bool kF16>
__global__ void __launch_bounds__(WG_THREADS, 1)
dcn_bwd_wgrad_tc_kernel(const __grid_constant__ CUtensorMap gmap, BwdParams p, int stages,
                        int m_tiles, int splits) {
    using E = Elem16<kF16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const WgLayout L = wg_layout(p.O, stages);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + stages);
    const uint32_t acc_full = smem_u32(bars + 2 * stages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 1);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x / 32), 0);
    const int lane = threadIdx.x % 32;
    const int tiles_x = (p.Wo + WG_TILE_W - 1) / WG_TILE_W;
    const int tiles_y = (p.Ho + WG_TILE_H - 1) / WG_TILE_H;
    const int tiles = p.B * tiles_x * tiles_y;
    const int taps = p.kh * p.kw;
    const int ncb = p.C / WG_UNIT;
    const int units = taps * ncb;
    // this CTA's rows (units 2 mt, 2 mt + 1) and run of tiles
    const int mt = blockIdx.x % m_tiles;
    const int split = blockIdx.x / m_tiles;
    const int t_begin = static_cast<int>(static_cast<long long>(tiles) * split / splits);
    const int t_end = static_cast<int>(static_cast<long long>(tiles) * (split + 1) / splits);
    const int n_kb = t_end - t_begin;
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>(p.O)) tmem_cols <<= 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1 + WG_TEAM_WARPS);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    }
    if (warp == 1 && lane == 0) tma_prefetch_desc(&gmap);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (B)
        if (lane == 0) {
            int s = 0, issued = 0;
            uint32_t phase = 0;
            for (int kb = 0; kb < n_kb; ++kb) {
                const int tile = t_begin + kb;
                const int tb = tile / (tiles_x * tiles_y);
                const int trem = tile - tb * tiles_x * tiles_y;
                const int th0 = (trem / tiles_x) * WG_TILE_H;
                const int tw0 = (trem % tiles_x) * WG_TILE_W;
                if (!mbar_wait_sleep(empty0 + 8 * s, phase ^ 1, p.status, p.timeout_ns)) break;
                mbar_arrive_expect_tx(full0 + 8 * s, L.b_bytes);
                const uint32_t b_dst = smem_u32(smem + s * L.stage_bytes + WG_A_BYTES);
                for (int j = 0; j < p.O / 64; ++j)
                    tma_load_4d(b_dst + j * WG_BOX_BYTES, &gmap, full0 + 8 * s, j * 64, tw0, th0, tb);
                ++issued;
                if (++s == stages) { s = 0; phase ^= 1; }
            }
            // every copy this CTA started must land before it exits
            const int first = issued > stages ? issued - stages : 0;
            for (int i = first; i < issued; ++i)
                mbar_wait_sleep(full0 + 8 * (i % stages), (i / stages) & 1, p.status, p.timeout_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            // kind::f16, fp32 accumulator, both operands MN-major (bits 15, 16)
            const uint32_t idesc = E::idesc(WG_BM, p.O) | (1u << 15) | (1u << 16);
            int s = 0;
            uint32_t phase = 0;
            int done = 0;
            for (int kb = 0; kb < n_kb; ++kb) {
                if (!mbar_wait_sleep(full0 + 8 * s, phase, p.status, p.timeout_ns)) break;
                tc_fence_after_sync();
                const uint32_t a_addr = smem_u32(smem + s * L.stage_bytes);
                const uint64_t a_desc = smem_desc_mn_sw128(a_addr, WG_UNIT_BYTES, 1024);
                const uint64_t b_desc = smem_desc_mn_sw128(a_addr + WG_A_BYTES, WG_BOX_BYTES, 1024);
#pragma unroll
                for (int ks = 0; ks < WG_BK / 16; ++ks) {
                    // K = 16 pixels = two 8-row swizzle atoms, 2048 bytes on
                    mma_kind_f16_ss(tmem_base, a_desc + ks * (2048 >> 4), b_desc + ks * (2048 >> 4), idesc,
                                    (kb > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(empty0 + 8 * s);
                ++done;
                if (++s == stages) { s = 0; phase ^= 1; }
            }
            // the accumulator is complete once the last MMAs are (also
            // before TMEM is released)
            mma_commit(acc_full);
            mbar_wait_sleep(acc_full, 0, p.status, p.timeout_ns);
            (void)done;
        }
    } else {
        // ------------------------------------------------ samplers
        const int sw = warp - 2;                         // 0 .. 15
        const int team = sw / WG_TEAM_WARPS;             // takes tiles team, team + 2, ...
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const int half = (sw % WG_TEAM_WARPS) / 4;
        const int trow = 2 * q + half;                   // tile row = pixels 16 trow .. +15
        const int quart = lane & 3;                      // channels 16 quart .. +15 of a unit
        const int rsub = lane >> 2;                      // pixels rsub and rsub + 8 of the row
        const int my_px = lane & 15;                     // geometry: pixel (tile column)
        const int my_g = lane >> 4;                      // geometry: unit
        const uint16_t *__restrict__ x = static_cast<const uint16_t *>(p.x);
        const uint32_t table_s = smem_u32(smem + L.table_off + sw * WG_TABLE_WARP_BYTES);
        const uint32_t raw_s = smem_u32(smem + L.raw_off + sw * WG_RAW_WARP_BYTES) + lane * 4;
        const int HoWo = p.Ho * p.Wo;
        const int Cq = p.C / p.ogroups;
        // the unit this geometry lane tabulates: its tap, offset group and
        // row of the image's offset / mask planes
        const int u_g = min(2 * mt + my_g, units - 1);
        const int tap_g = u_g / ncb;
        const int og_g = (u_g - tap_g * ncb) * WG_UNIT / Cq;
        const int i_g = tap_g / p.kw, j_g = tap_g - (tap_g / p.kw) * p.kw;
        const int plane_g = og_g * taps + tap_g;         // mask plane; offsets 2 plane_g, 2 plane_g + 1
        // the channel base of each unit this gather lane reads
        int cbase[2];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int u = min(2 * mt + g, units - 1);
            cbase[g] = (u - (u / ncb) * ncb) * WG_UNIT + 16 * quart;
        }
        if (p.mask == nullptr) sts_b32(raw_s + 256, __float_as_uint(1.0f));
        const int step_x = p.W > 1 ? p.C : 0;
        const int step_y = p.H > 1 ? p.W * p.C : 0;

        // the geometry lane's pixel of tile `tile`
        auto pixel_of = [&](int tile, int &tb, int &oh, int &ow) {
            tb = tile / (tiles_x * tiles_y);
            const int trem = tile - tb * tiles_x * tiles_y;
            oh = (trem / tiles_x) * WG_TILE_H + trow;
            ow = (trem % tiles_x) * WG_TILE_W + my_px;
        };
        auto load_raw = [&](int tile) {
            int tb, oh, ow;
            pixel_of(tile, tb, oh, ow);
            const bool valid = oh < p.Ho && ow < p.Wo && 2 * mt + my_g < units;
            const size_t hw = valid ? static_cast<size_t>(oh) * p.Wo + ow : 0;
            const float *o = p.offset + (static_cast<size_t>(tb) * p.ogroups * taps * 2 + 2 * plane_g) * HoWo + hw;
            // an offset or mask outside its tensor is not fetched (zero)
            const bool v_dy = valid && WG_IN(o, 4, p.off_lo, p.off_hi);
            const bool v_dx = valid && WG_IN(o + HoWo, 4, p.off_lo, p.off_hi);
            cp_async_4(raw_s, v_dy ? o : p.offset, v_dy);
            cp_async_4(raw_s + 128, v_dx ? o + HoWo : p.offset, v_dx);
            if (p.mask) {
                const float *mp = p.mask + (static_cast<size_t>(tb) * p.ogroups * taps + plane_g) * HoWo + hw;
                const bool v_m = valid && WG_IN(mp, 4, p.mask_lo, p.mask_hi);
                cp_async_4(raw_s + 256, v_m ? mp : p.mask, v_m);
            }
        };
        auto tabulate = [&](int tile) {
            int tb, oh, ow;
            pixel_of(tile, tb, oh, ow);
            cp_async_wait_all();
            const float dy = lds_f32(raw_s), dx = lds_f32(raw_s + 128), m = lds_f32(raw_s + 256);
            TapBlock t;
            tap_block(dy, dx, m, oh * p.sh - p.ph + i_g * p.dh, ow * p.sw - p.pw + j_g * p.dw, tb,
                      p.H, p.W, p.C, t);
            const uint32_t ent = table_s + my_g * 2 * WG_TILE_W * 16 + my_px * 16;
            sts_v4_b32_m(ent, __float_as_uint(t.w[0]), __float_as_uint(t.w[1]), __float_as_uint(t.w[2]),
                         __float_as_uint(t.w[3]));
            sts_b32(ent + WG_TILE_W * 16, static_cast<uint32_t>(t.idx));
        };

        bool ok = true;
        int s = team;
        uint32_t phase = 0;
        // this warp's tiles: kb = team, team + 2, ...
        if (team < n_kb) load_raw(t_begin + team);
        for (int kb = team; kb < n_kb; kb += 2) {
            tabulate(t_begin + kb);
            if (kb + 2 < n_kb) load_raw(t_begin + kb + 2);
            __syncwarp();
            const bool got = mbar_wait_sleep(empty0 + 8 * s, phase ^ 1, p.status, p.timeout_ns, 2000u);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            const uint32_t a_stage = smem_u32(smem + s * L.stage_bytes);
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                const uint32_t tg = table_s + g * 2 * WG_TILE_W * 16;
                u32x8 v[8];
                float4 wgt[2];
#pragma unroll
                for (int px = 0; px < 2; ++px) {
                    const uint32_t ent = tg + (rsub + 8 * px) * 16;
                    wgt[px] = lds_v4_f32(ent);
                    const int e0 = lds_s32(ent + WG_TILE_W * 16) + cbase[g];
                    const int e1 = e0 + step_x, e2 = e0 + step_y, e3 = e2 + step_x;
#ifdef DCN_CHECK_BOUNDS
                    // a corner row outside x is read from x's first bytes instead
                    auto chk = [&](const uint16_t *a) {
                        return WG_IN(a, 32, p.x_lo, p.x_hi) ? a : static_cast<const uint16_t *>(p.x_lo);
                    };
                    v[4 * px + 0] = ldg_v8(chk(x + e0));
                    v[4 * px + 1] = ldg_v8(chk(x + e1));
                    v[4 * px + 2] = ldg_v8(chk(x + e2));
                    v[4 * px + 3] = ldg_v8(chk(x + e3));
#else
                    v[4 * px + 0] = ldg_v8(x + e0);
                    v[4 * px + 1] = ldg_v8(x + e1);
                    v[4 * px + 2] = ldg_v8(x + e2);
                    v[4 * px + 3] = ldg_v8(x + e3);
#endif
                }
#pragma unroll
                for (int px = 0; px < 2; ++px) {
                    const u32x8 *vp = v + 4 * px;
                    const uint64_t c0 = f2_make(wgt[px].x, wgt[px].x), c1 = f2_make(wgt[px].y, wgt[px].y);
                    const uint64_t c2 = f2_make(wgt[px].z, wgt[px].z), c3 = f2_make(wgt[px].w, wgt[px].w);
                    uint32_t o[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        uint64_t acc = f2_mul(c0, f2_make(E::lo(vp[0].w[m]), E::hi(vp[0].w[m])));
                        acc = f2_fma(c1, f2_make(E::lo(vp[1].w[m]), E::hi(vp[1].w[m])), acc);
                        acc = f2_fma(c2, f2_make(E::lo(vp[2].w[m]), E::hi(vp[2].w[m])), acc);
                        acc = f2_fma(c3, f2_make(E::lo(vp[3].w[m]), E::hi(vp[3].w[m])), acc);
                        o[m] = E::pack_f2(acc);
                    }
                    // pixel row of the tile, its 128-byte row in the unit's A
                    // block and the two swizzled 16-byte chunks of channels
                    // 16 quart .. +15
                    const int pix = trow * WG_TILE_W + rsub + 8 * px;
                    const uint32_t row = a_stage + g * WG_UNIT_BYTES + pix * 128;
                    const int sw8 = pix & 7;
                    sts_v4_b32(row + (((2 * quart) ^ sw8) << 4), o[0], o[1], o[2], o[3]);
                    sts_v4_b32(row + (((2 * quart + 1) ^ sw8) << 4), o[4], o[5], o[6], o[7]);
                }
            }
            // the generic-proxy writes must be visible to the MMA (async proxy)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full0 + 8 * s);
            s += 2;
            if (s >= stages) { s -= stages; phase ^= 1; }
        }
        cp_async_wait_all();

        // ---- the accumulator, added into grad_weight[o][c][tap]
        if (ok) ok = mbar_wait_sleep(acc_full, 0, p.status, p.timeout_ns);
        __syncwarp();
        tc_fence_after_sync();
        const int part = sw >> 2;                        // column quarter
        const int row = q * 32 + lane;                   // D row = (unit, channel)
        const int u = 2 * mt + row / WG_UNIT;
        if (ok && n_kb > 0) {
            const int tap = u / ncb;
            const int c = (u - tap * ncb) * WG_UNIT + row % WG_UNIT;
            const int nch = p.O / 16;
            const int ch0 = part * nch / 4, ch1 = (part + 1) * nch / 4;
            for (int ch = ch0; ch < ch1; ++ch) {
                float vv[16];
                tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ch * 16, vv);
                if (u < units) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int o = ch * 16 + e;
                        float *gw = p.grad_weight + (static_cast<size_t>(o) * p.C + c) * taps + tap;
                        if (WG_IN(gw, 4, p.gw_lo, p.gw_hi)) atomicAdd(gw, vv[e]);
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

// the dynamic shared-memory limit set on each device, per operand type
PerDeviceValue<> g_wgrad_smem_set[2];

}  // namespace

int bwd_wgrad_row_blocks(const BwdParams &p) {
    return (p.kh * p.kw * (p.C / WG_UNIT) + 1) / 2;
}

cudaError_t launch_bwd_wgrad_tc(const BwdParams &p, const CUtensorMap &gmap, cudaStream_t stream) {
    if (p.groups != 1 || p.C % WG_UNIT != 0 || p.O % 64 != 0 || p.O > 256 || p.O < 64 ||
        (p.C / p.ogroups) % WG_UNIT != 0)
        return cudaErrorInvalidValue;
    // as many stages (two at least, one per sampler team) as fit 200 KB
    int stages = 4;
    while (stages > 2 && wg_layout(p.O, stages).total + 1024 > 200 * 1024) --stages;
    const WgLayout L = wg_layout(p.O, stages);
    const int smem = L.total + 1024;
    auto kernel = p.f16 ? dcn_bwd_wgrad_tc_kernel<true> : dcn_bwd_wgrad_tc_kernel<false>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = static_cast<cudaError_t>(g_wgrad_smem_set[p.f16 ? 1 : 0].ensure(dev, smem, [&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    }));
    if (e != cudaSuccess) return e;
    const int m_tiles = bwd_wgrad_row_blocks(p);
    const int tiles = p.B * ((p.Ho + WG_TILE_H - 1) / WG_TILE_H) * ((p.Wo + WG_TILE_W - 1) / WG_TILE_W);
    // runs of tiles per row block: about one CTA per SM in all
    int splits = p.sm_count > m_tiles ? p.sm_count / m_tiles : 1;
    if (splits > tiles) splits = tiles;
    const long long grid = static_cast<long long>(m_tiles) * splits;
    if (grid > 2147483647ll) return cudaErrorInvalidValue;
    kernel<<<static_cast<unsigned>(grid), WG_THREADS, smem, stream>>>(gmap, p, stages, m_tiles, splits);
    return cudaGetLastError();
}

}  // namespace dcn
