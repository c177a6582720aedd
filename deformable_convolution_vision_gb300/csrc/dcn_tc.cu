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
// One CTA computes a tile of 8 x 16 output pixels of one image (a compact
// 2-D tile keeps each tap's sampled footprint small, so more corner reads
// hit L1) x all O output channels:
//   warp 0      TMA producer: the packed-weight K-block [O x 64] of each
//               stage, 128-byte swizzle; also allocates/frees TMEM.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=O,
//               K=16) x 4 per K-block, accumulating in TMEM, and commits
//               each stage back to its "empty" barrier.
//   warps 2..17 samplers: per (pixel, tap) the corner weights and
//               addresses (S1, S2), then for 8 channels per lane the four
//               16-byte corner loads, the bilinear combine (by default in
//               the input dtype, bf16, as packed bf16x2 FMAs; optionally in
//               fp32 with packed f32x2 FMAs), a bf16
//               round and one 16-byte store into the swizzled A stage (S3).
//               After the last K-block they run the epilogue (S5): TMEM ->
//               registers, + bias in fp32, bf16 round, channels-last store.
// K-blocks run tap-major with 64 channels each, so a tap's corner geometry
// is computed once and reused for all of its channel blocks.  The geometry
// is computed for two taps at a time by all 32 lanes of a sampler warp into
// a ring of four per-warp tables, with its inputs fetched taps ahead.  Each
// lane issues all sixteen corner loads of a stage before it waits for the
// stage to be free.
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
constexpr int TC_MMA_K = 16;
constexpr int TC_TILE_W = 16;                                 // tile = 8 x 16 output pixels
constexpr int TC_TILE_H = TC_BM / TC_TILE_W;
constexpr int TC_SAMPLER_WARPS = 16;
constexpr int TC_ROWS_PER_WARP = TC_BM / TC_SAMPLER_WARPS;    // 8 pixels: half a tile row
constexpr int TC_THREADS = 32 * (2 + TC_SAMPLER_WARPS);
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;                 // 16 KB
constexpr int TC_TAP_GROUP = 32 / TC_ROWS_PER_WARP;           // taps tabulated together (one per 8 lanes)
constexpr int TC_TABLE_BUFS = 2 * TC_TAP_GROUP;               // ring: one group in use, one ahead
static_assert(TC_ROWS_PER_WARP * 2 == TC_TILE_W, "two sampler warps per tile row");
static_assert((TC_TABLE_BUFS & (TC_TABLE_BUFS - 1)) == 0, "ring size is a power of two");

// Per-warp corner table of one tap: arrays of 16-byte rows, one row per
// pixel of the warp (conflict-free writes and broadcast reads).  The fp32
// combine keeps the weights as duplicated fp32 pairs {w0,w0,w1,w1},
// {w2,w2,w3,w3}; the bf16 combine as four bf16x2 pairs.  Then the four
// corner indices.
constexpr int TC_TABLE_ARRAY_BYTES = TC_ROWS_PER_WARP * 16;
constexpr int TC_TABLE_W01 = 0;
constexpr int TC_TABLE_W23 = TC_TABLE_ARRAY_BYTES;            // fp32 combine only
__host__ __device__ constexpr int table_buf_bytes(bool f32) { return (f32 ? 3 : 2) * TC_TABLE_ARRAY_BYTES; }
__host__ __device__ constexpr int table_idx_off(bool f32) { return (f32 ? 2 : 1) * TC_TABLE_ARRAY_BYTES; }

struct TcLayout {
    int stages;
    int b_bytes;       // O * 128
    int stage_bytes;   // A + B
    int bar_off;       // barriers after the stages
    int table_off;     // per-warp corner tables
    int total;         // bytes used from the 1024-aligned base
};

__host__ __device__ inline TcLayout tc_layout(int O, int stages, bool f32) {
    TcLayout L;
    L.stages = stages;
    L.b_bytes = O * TC_BK * 2;
    L.stage_bytes = TC_A_BYTES + L.b_bytes;
    L.bar_off = stages * L.stage_bytes;
    // full[stages], empty[stages], accum_full, tmem slot (8 bytes each)
    L.table_off = L.bar_off + (2 * stages + 2) * 8;
    L.table_off = (L.table_off + 15) & ~15;
    L.total = L.table_off + TC_SAMPLER_WARPS * TC_TABLE_BUFS * table_buf_bytes(f32);
    return L;
}

__host__ __device__ inline int tmem_cols_for(int O) {
    int n = 32;
    while (n < O) n <<= 1;
    return n;
}

// The CTA's share of the work: K-block units [u_begin, u_end) of the walk
// tile-major, K-block-minor.  A segment is the run of those units inside
// one tile.
struct Segment {
    int tile, kb0, kb1;   // K-blocks [kb0, kb1) of `tile`
};

__device__ __forceinline__ bool next_segment(int &u, int u_end, int nkb, Segment &sg) {
    if (u >= u_end) return false;
    sg.tile = u / nkb;
    sg.kb0 = u - sg.tile * nkb;
    sg.kb1 = min(nkb, sg.kb0 + (u_end - u));
    u += sg.kb1 - sg.kb0;
    return true;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float4 ld_cg_f4(const float *p) {
    return __ldcg(reinterpret_cast<const float4 *>(p));
}

template <bool kSampleF32>
__global__ void __launch_bounds__(TC_THREADS, 1)
dcn_tc_kernel(const __grid_constant__ CUtensorMap wmap, Params p, int stages) {
    constexpr int kBuf = table_buf_bytes(kSampleF32);
    constexpr int kIdx = table_idx_off(kSampleF32);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const TcLayout L = tc_layout(p.O, stages, kSampleF32);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + stages);
    const uint32_t accum_bar = smem_u32(bars + 2 * stages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int tiles_x = (p.Wo + TC_TILE_W - 1) / TC_TILE_W;
    const int tiles_y = (p.Ho + TC_TILE_H - 1) / TC_TILE_H;
    const int ncb = p.C / TC_BK;
    const int taps = p.kh * p.kw;
    const int nkb = taps * ncb;
    const int total = p.B * tiles_x * tiles_y * nkb;
    const int u_begin = blockIdx.x * p.units_per_cta;
    const int u_end = min(u_begin + p.units_per_cta, total);
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
            int s = 0;
            uint32_t phase = 0;
            int kb = u_begin % nkb;
            for (int u = u_begin; u < u_end; ++u) {
                if (!mbar_wait_sleep(empty0 + 8 * s, phase ^ 1, p.status, p.timeout_ns)) break;
                const uint32_t b_dst = smem_u32(smem + s * L.stage_bytes + TC_A_BYTES);
                mbar_arrive_expect_tx(full0 + 8 * s, L.b_bytes);
                tma_load_2d(b_dst, &wmap, full0 + 8 * s, kb * TC_BK, 0);
                ++issued;
                if (++kb == nkb) kb = 0;
                if (++s == stages) { s = 0; phase ^= 1; }
            }
            // Before the CTA can exit, every weight copy it started must
            // have landed: wait (bounded) for the last phase of each stage.
            const int first = issued > stages ? issued - stages : 0;
            for (int i = first; i < issued; ++i)
                mbar_wait_sleep(full0 + 8 * (i % stages), (i / stages) & 1, p.status, p.timeout_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(TC_BM, p.O);
            int s = 0;
            uint32_t phase = 0;
            int segs = 0;
            Segment sg;
            int u = u_begin;
            bool live = true;
            while (live && next_segment(u, u_end, nkb, sg)) {
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!mbar_wait_sleep(full0 + 8 * s, phase, p.status, p.timeout_ns)) { live = false; break; }
                    tc_fence_after_sync();
                    const uint32_t a_addr = smem_u32(smem + s * L.stage_bytes);
                    const uint32_t b_addr = a_addr + TC_A_BYTES;
                    const uint64_t adesc = smem_desc_sw128(a_addr);
                    const uint64_t bdesc = smem_desc_sw128(b_addr);
#pragma unroll
                    for (int ks = 0; ks < TC_BK / TC_MMA_K; ++ks) {
                        // advance the start address by 32 bytes per K=16 step; the
                        // segment's first MMA overwrites the accumulator
                        mma_bf16_ss(tmem_base, adesc + 2 * ks, bdesc + 2 * ks, idesc,
                                    (kb > sg.kb0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(empty0 + 8 * s);
                    if (++s == stages) { s = 0; phase ^= 1; }
                }
                // the segment's accumulator is complete once its MMAs are
                mma_commit(accum_bar);
                ++segs;
            }
            // the MMAs must be complete before TMEM is released
            if (segs > 0) mbar_wait_sleep(accum_bar, (segs - 1) & 1, p.status, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------ samplers
        const int sw = warp - 2;                         // sampler warp 0..15
        const int trow = sw >> 1;                        // its tile row
        const int tcol0 = (sw & 1) * TC_ROWS_PER_WARP;   // its first tile column
        const int row_base = trow * TC_TILE_W + tcol0;   // its first A row
        const __nv_bfloat16 *__restrict__ x = static_cast<const __nv_bfloat16 *>(p.x);
        uint8_t *table = smem + L.table_off + sw * TC_TABLE_BUFS * kBuf;
        const uint32_t table_s = smem_u32(table);
        const uint32_t stage0_s = smem_u32(smem);
        const int HoWo = p.Ho * p.Wo;
        const int my_g = lane >> 3;     // geometry: tap offset within a group of four
        const int my_px = lane & 7;     // geometry: pixel of the warp
        const int quart = lane & 3;     // gather: 16 channels of the 64-channel K-block
        const int rsub = lane >> 2;     // gather: warp row 0..7
        const int arow = row_base + rsub;
        const uint32_t r_off = rsub * 16;
        // the lane's two 16-byte chunks in an A stage (128-byte swizzle: chunk
        // c of row r lives at chunk c ^ (r % 8))
        const uint32_t sts0 = arow * 128 + (((2 * quart) ^ (arow & 7)) << 4);
        const uint32_t sts1 = arow * 128 + (((2 * quart + 1) ^ (arow & 7)) << 4);
        // epilogue: TMEM lane quarter, column part, A row of this thread
        const int q = warp & 3;
        const int part = sw >> 2;
        const int erow = q * 32 + lane;
        const int nch = p.O / 16;
        const int ch_begin = part * nch / 4;
        const int ch_end = (part + 1) * nch / 4;
        const size_t part_floats = static_cast<size_t>(nch) * TC_BM * 16;   // one partial tile
        bool ok = true;
        int s = 0;
        uint32_t phase = 0;
        uint32_t a_stage = stage0_s;
        int segs = 0;

        Segment sg;
        int u = u_begin;
        while (next_segment(u, u_end, nkb, sg)) {
            // ---- this segment's tile
            const int tb = sg.tile / (tiles_x * tiles_y);
            const int trem = sg.tile - tb * tiles_x * tiles_y;
            const int th0 = (trem / tiles_x) * TC_TILE_H;
            const int tw0 = (trem % tiles_x) * TC_TILE_W;
            const int my_h = th0 + trow;
            const int my_w = tw0 + tcol0 + my_px;
            const bool my_valid = (my_h < p.Ho) && (my_w < p.Wo);
            const int my_hw = my_valid ? my_h * p.Wo + my_w : 0;
            const int t0 = sg.kb0 / ncb;                 // first tap of the segment
            const int g0 = t0 & ~(TC_TAP_GROUP - 1);     // its group of four taps

            // raw inputs (dy, dx, mask) of this lane's next tap, fetched a whole
            // tap group ahead of their use so their latency hides behind gathers
            float n_dy = 0.0f, n_dx = 0.0f, n_m = 0.0f;
            auto load_raw = [&](int group_tap) {
                const int tap = group_tap + my_g;
                if (my_valid && tap < taps) {
                    const float *o = p.offset + (static_cast<size_t>(tb) * 2 * taps + 2 * tap) * HoWo + my_hw;
                    n_dy = __ldg(o);
                    n_dx = __ldg(o + HoWo);
                    n_m = p.mask ? __ldg(p.mask + (static_cast<size_t>(tb) * taps + tap) * HoWo + my_hw)
                                 : 1.0f;
                }
            };
            // kernel row and column (ti, tj) of this lane's tap, advanced by
            // four taps per tabulation instead of divided out each time
            int ti = (g0 + my_g) / p.kw;
            int tj = (g0 + my_g) - ti * p.kw;
            // corner tables of taps group_tap .. group_tap + 3 (ring slot tap % 8)
            auto tabulate = [&](int group_tap) {
                const int tap = group_tap + my_g;
                TapCorners t;
                if (my_valid && tap < taps) {
                    tap_corners(n_dy, n_dx, n_m, my_h, my_w, ti, tj, p.pad, tb, p.H, p.W, p.C, t);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) { t.w[k] = 0.0f; t.idx[k] = 0; }
                }
                uint8_t *slot = table + (tap & (TC_TABLE_BUFS - 1)) * kBuf;
                const int rowb = my_px * 16;
                if constexpr (kSampleF32) {
                    *reinterpret_cast<float4 *>(slot + TC_TABLE_W01 + rowb) = make_float4(t.w[0], t.w[0], t.w[1], t.w[1]);
                    *reinterpret_cast<float4 *>(slot + TC_TABLE_W23 + rowb) = make_float4(t.w[2], t.w[2], t.w[3], t.w[3]);
                } else {
                    // the weights rounded to bf16, each duplicated into a bf16x2 pair
                    *reinterpret_cast<uint4 *>(slot + TC_TABLE_W01 + rowb) =
                        make_uint4(bf16x2_splat(t.w[0]), bf16x2_splat(t.w[1]), bf16x2_splat(t.w[2]),
                                   bf16x2_splat(t.w[3]));
                }
                *reinterpret_cast<int4 *>(slot + kIdx + rowb) = make_int4(t.idx[0], t.idx[1], t.idx[2], t.idx[3]);
                tj += TC_TAP_GROUP;
                while (tj >= p.kw) { tj -= p.kw; ++ti; }
            };
            // the four 32-byte corner loads of this lane's item from a table
            // slot; corners outside the image read a clamped in-image address
            // and carry weight 0
            auto issue = [&](uint32_t slot, const __nv_bfloat16 *xc, u32x8 (&v)[4]) {
                const int4 ci = lds_v4_s32(slot + kIdx + r_off);
                v[0] = ldg_v8(xc + ci.x);
                v[1] = ldg_v8(xc + ci.y);
                v[2] = ldg_v8(xc + ci.z);
                v[3] = ldg_v8(xc + ci.w);
            };

            // Tables of the first two tap groups.  (The group after a group
            // that starts inside the segment is tabulated when that group's
            // first tap ends; a segment that starts mid-group never sees that
            // tap end, so its second group is tabulated here.)  Slots of the
            // previous segment are free: this warp finished reading them.
            load_raw(g0);
            tabulate(g0);
            if (g0 + TC_TAP_GROUP < taps) load_raw(g0 + TC_TAP_GROUP);
            if (t0 != g0 && g0 + TC_TAP_GROUP < taps) {
                tabulate(g0 + TC_TAP_GROUP);
                if (g0 + 2 * TC_TAP_GROUP < taps) load_raw(g0 + 2 * TC_TAP_GROUP);
            }
            __syncwarp();

            // Rolling pipeline: the corner loads of K-block kb + 1 go out as
            // K-block kb is combined, so each lane always has loads in flight.
            u32x8 v[4];
            int tap = t0, cb = sg.kb0 - t0 * ncb;
            int n_tap = tap, n_cb = cb;
            if (++n_cb == ncb) { n_cb = 0; ++n_tap; }
            issue(table_s + (tap & (TC_TABLE_BUFS - 1)) * kBuf, x + cb * TC_BK + quart * 16, v);

            for (int kb = sg.kb0; ok && kb < sg.kb1; ++kb) {
                const bool has_next = kb + 1 < sg.kb1;
                const uint32_t cur_slot = table_s + (tap & (TC_TABLE_BUFS - 1)) * kBuf;

                // every lane waits; the warp leaves the loop together if any lane ran out
                const bool got = mbar_wait_sleep(empty0 + 8 * s, phase ^ 1, p.status, p.timeout_ns, 2000u);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }

                uint32_t packed[8];
                if constexpr (kSampleF32) {
                    uint64_t c0, c1, c2, c3;   // {w_q, w_q} fp32 pairs
                    lds_v2_u64(cur_slot + TC_TABLE_W01 + r_off, c0, c1);
                    lds_v2_u64(cur_slot + TC_TABLE_W23 + r_off, c2, c3);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        // channels 2k, 2k+1: w0*x00 + w1*x01 + w2*x10 + w3*x11 in fp32
                        uint64_t acc = f2_mul(c0, f2_make(bf16_lo(v[0].w[k]), bf16_hi(v[0].w[k])));
                        acc = f2_fma(c1, f2_make(bf16_lo(v[1].w[k]), bf16_hi(v[1].w[k])), acc);
                        acc = f2_fma(c2, f2_make(bf16_lo(v[2].w[k]), bf16_hi(v[2].w[k])), acc);
                        acc = f2_fma(c3, f2_make(bf16_lo(v[3].w[k]), bf16_hi(v[3].w[k])), acc);
                        packed[k] = f2_to_bf16x2(acc);
                    }
                } else {
                    // the same sum in the input dtype: bf16 weights, one bf16
                    // rounding per fused multiply-add, two channels per op
                    const int4 cw = lds_v4_s32(cur_slot + TC_TABLE_W01 + r_off);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint32_t acc = bf16x2_mul(cw.x, v[0].w[k]);
                        acc = bf16x2_fma(cw.y, v[1].w[k], acc);
                        acc = bf16x2_fma(cw.z, v[2].w[k], acc);
                        acc = bf16x2_fma(cw.w, v[3].w[k], acc);
                        packed[k] = acc;
                    }
                }
                if (has_next)
                    issue(table_s + (n_tap & (TC_TABLE_BUFS - 1)) * kBuf, x + n_cb * TC_BK + quart * 16, v);
                sts_v4_b32(a_stage + sts0, packed[0], packed[1], packed[2], packed[3]);
                sts_v4_b32(a_stage + sts1, packed[4], packed[5], packed[6], packed[7]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full0 + 8 * s);

                if (cb == ncb - 1 && (tap & (TC_TAP_GROUP - 1)) == 0 && tap + TC_TAP_GROUP < taps) {
                    // the ring slots of taps tap - 4 .. tap - 1 are no longer read:
                    // fill them for taps tap + 4 .. tap + 7 and fetch the group after
                    tabulate(tap + TC_TAP_GROUP);
                    if (tap + 2 * TC_TAP_GROUP < taps) load_raw(tap + 2 * TC_TAP_GROUP);
                    __syncwarp();
                }
                tap = n_tap;
                cb = n_cb;
                if (++n_cb == ncb) { n_cb = 0; ++n_tap; }
                a_stage += L.stage_bytes;
                if (++s == stages) { s = 0; phase ^= 1; a_stage = stage0_s; }
            }

            // ---- epilogue (S5) of the segment
            if (ok) ok = mbar_wait_sleep(accum_bar, segs & 1, p.status, p.timeout_ns);
            ++segs;
            __syncwarp();
            tc_fence_after_sync();
            const int oh = th0 + erow / TC_TILE_W;
            const int ow = tw0 + erow % TC_TILE_W;
            const bool pix_valid = oh < p.Ho && ow < p.Wo;
            const size_t pix = (static_cast<size_t>(tb) * p.Ho + oh) * p.Wo + ow;
            if (sg.kb0 > 0) {
                // The tile's other K-blocks belong to the CTA before this one:
                // leave the fp32 partial for it and raise this CTA's flag.
                float *dst = p.partial + static_cast<size_t>(blockIdx.x) * part_floats;
                for (int ch = ch_begin; ch < ch_end; ++ch) {
                    float vv[16];
                    tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ch * 16, vv);
                    float4 *d4 = reinterpret_cast<float4 *>(dst + (static_cast<size_t>(ch) * TC_BM + erow) * 16);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        d4[e] = make_float4(vv[4 * e], vv[4 * e + 1], vv[4 * e + 2], vv[4 * e + 3]);
                }
                __threadfence();
                named_barrier_sync(1, 32 * TC_SAMPLER_WARPS);
                if (sw == 0 && lane == 0) st_release_u32(p.flags + blockIdx.x, p.epoch);
            } else {
                // The tile's last K-blocks may belong to the next CTA: wait
                // (bounded) for its partial and add it.
                const bool merge = sg.kb1 < nkb;
                const float *src = p.partial + static_cast<size_t>(blockIdx.x + 1) * part_floats;
                if (merge && ok) {
                    const uint64_t t0ns = global_timer_ns();
                    while (ld_acquire_u32(p.flags + blockIdx.x + 1) != p.epoch) {
                        if (global_timer_ns() - t0ns > p.timeout_ns) {
                            atomicOr(p.status, kStatusTimeout);
                            ok = false;
                            break;
                        }
                    }
                }
                __nv_bfloat16 *__restrict__ out = static_cast<__nv_bfloat16 *>(p.out);
                for (int ch = ch_begin; ch < ch_end; ++ch) {
                    float vv[16];
                    tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ch * 16, vv);
                    if (merge && ok) {
                        const float *sp = src + (static_cast<size_t>(ch) * TC_BM + erow) * 16;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float4 a = ld_cg_f4(sp + 4 * e);
                            vv[4 * e] += a.x; vv[4 * e + 1] += a.y; vv[4 * e + 2] += a.z; vv[4 * e + 3] += a.w;
                        }
                    }
                    if (ok && pix_valid) {
                        uint32_t pk[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int o = ch * 16 + 2 * e;
                            const float b0 = p.bias ? __ldg(p.bias + o) : 0.0f;
                            const float b1 = p.bias ? __ldg(p.bias + o + 1) : 0.0f;
                            pk[e] = pack_bf16x2(vv[2 * e] + b0, vv[2 * e + 1] + b1);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(out + pix * p.O + ch * 16);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            }
            // TMEM reads of this segment finish before the next one's stages
            // are handed to the MMA warp
            tc_fence_before_sync();
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
int g_max_smem_set_f32 = 0;

// Carveout preference (percent of the 228 KB maximum) that selects the
// smallest supported shared-memory size holding `needed` bytes; the driver
// rounds a percentage up to the next supported size.
int carveout_percent(int needed) {
    static const int kSizesKb[] = {0, 8, 16, 32, 64, 100, 132, 164, 196, 228};
    for (int kb : kSizesKb) {
        if (kb * 1024 >= needed) return kb == 0 ? 0 : (kb * 100) / 228;
    }
    return 100;
}

// Shared memory the CTA may use (stages + tables + alignment).  The SM's
// L1/shared array is 256 KB; at 131 KB the 132 KB carveout leaves 124 KB of
// L1 for the corner gathers.
#ifndef DCN_TC_SMEM_BUDGET
#define DCN_TC_SMEM_BUDGET (131 * 1024)
#endif

}  // namespace

bool tc_supported(int C, int O) {
    return C % TC_BK == 0 && O % 16 == 0 && O >= 16 && O <= 256;
}

cudaError_t launch_tc(const Params &p_in, const CUtensorMap &wmap, cudaStream_t stream) {
    // One CTA per SM.  Its shared memory is kept small so that most of the
    // SM's L1/shared array stays L1 cache, which holds a good part of the
    // tile's corner footprint across taps.
    Params p = p_in;
    const bool f32 = p.sample_f32 != 0;
    const int fixed = tc_layout(p.O, 0, f32).total + 1024;
    int stages = (DCN_TC_SMEM_BUDGET - fixed) / tc_layout(p.O, 1, f32).stage_bytes;
    stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
    const TcLayout L = tc_layout(p.O, stages, f32);
    const int smem = L.total + 1024;  // slack for 1024-byte alignment
    auto kernel = f32 ? dcn_tc_kernel<true> : dcn_tc_kernel<false>;
    int &smem_set = f32 ? g_max_smem_set_f32 : g_max_smem_set;
    if (smem != smem_set) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        // ask for just enough shared memory for the one resident CTA (plus
        // the 1 KB the system reserves per CTA); the rest stays L1
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 carveout_percent(smem + 1024));
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    const int tiles = p.B * ((p.Ho + TC_TILE_H - 1) / TC_TILE_H) * ((p.Wo + TC_TILE_W - 1) / TC_TILE_W);
    const int nkb = p.kh * p.kw * (p.C / TC_BK);
    const long long total = static_cast<long long>(tiles) * nkb;
    if (p.partial && p.flags && tiles > p.sm_count && p.sm_count > 0) {
        // Stream-K: every CTA (one per SM, all resident) takes an equal run
        // of (tile, K-block) units, so no SM idles through a last partial
        // wave; a tile split between two CTAs is merged by the first.
        const int units = static_cast<int>((total + p.sm_count - 1) / p.sm_count);
        p.units_per_cta = units;
        const int grid = static_cast<int>((total + units - 1) / units);
        void *args[] = {const_cast<CUtensorMap *>(&wmap), &p, &stages};
        const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kernel),
                                                          dim3(grid), dim3(TC_THREADS), args, smem,
                                                          stream);
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        cudaGetLastError();   // not all CTAs could be resident: one tile per CTA instead
    }
    // one tile per CTA
    p.units_per_cta = nkb;
    kernel<<<tiles, TC_THREADS, smem, stream>>>(wmap, p, stages);
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
