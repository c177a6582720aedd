// tcgen05 fused implicit-GEMM forward kernel (bf16 or fp16 operands, fp32
// TMEM accumulation) for sm_103a.
//
// The contraction out[p, o] = sum_K A[p, K] * Wp[o, K] with K = (tap, c) is
// a dense GEMM whose A operand is never materialised in memory: the im2col
// column buffer that page "deformops 3.0.1" (section "Deformable
// convolution") avoids, and that the "birefnet-lite-1024-webgpu
// patch_deform.py" page sizes at 392 MB for the 7x7, C = 64, 256 x 256
// layer, exists here only as one 128 x 64 tile per pipeline stage, in
// tensor memory.
//
// A tile is 8 x 16 output pixels of one image (a compact 2-D tile keeps each
// tap's sampled footprint small, so more corner reads hit L1) x all O
// output channels.  One CTA per SM:
//   warp 0      TMA producer: the packed-weight K-block [O x 64] of each
//               stage into shared memory, 128-byte swizzle; also
//               allocates/frees TMEM.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=O,
//               K=16, A from TMEM, B from shared memory) x 4 per K-block,
//               accumulating in TMEM, and commits each stage back to its
//               "empty" barrier.
//   warps 2..9  samplers, eight warps that each take every K-block.
//               A sampler warp owns one tile row (16 pixels, TMEM lanes
//               32q + 16h .. +15 of its lane quarter q).  Per (pixel, tap)
//               it computes the corner weights and addresses (S1, S2); per
//               K-block each lane gathers 16 channels of two pixels: eight
//               32-byte corner loads, the bilinear combine (by default in
//               the input dtype, as packed bf16x2 / fp16x2 FMAs; optionally
//               in fp32 with packed f32x2 FMAs) and one 16x256b store of both
//               pixels' rows into the stage's TMEM columns (S3).  After a
//               tile's last K-block all sixteen run the epilogue (S5): TMEM
//               -> registers, + bias in fp32, rounding to the operand type,
//               channels-last store.
// K-blocks of 64 channels run block-major: every tap of the first channel
// block, then every tap of the next, so that the corner lines a tile
// re-reads from tap to tap are one block's and stay in L1.  The geometry of
// a warp's next two K-blocks is computed by all 32 lanes (one K-block per
// half-warp) into a ring of four per-warp tables, with its inputs fetched a
// pair ahead.  Each lane issues the corner loads of its next K-block before
// it stores the current one.
//
// With more tiles than SMs the launch is persistent and stream-K: every
// CTA takes an equal run of (tile, K-block) units; a tile split between two
// CTAs is finished by the first, which adds the second's fp32 partial.
//
// Every barrier wait is bounded; a wait that runs out sets the status word
// and the kernel winds down without trapping.
#include <cuda_bf16.h>

#include "dcn_attr_cache.h"
#include "dcn_device.cuh"
#include "dcn_kernels.h"
#include "dcn_sampling.cuh"

namespace dcn {

namespace {

constexpr int TC_BM = 128;               // output pixels per tile (MMA M)
constexpr int TC_BK = 64;                // channels per K-block
constexpr int TC_MMA_K = 16;
constexpr int TC_TILE_W = 16;                                 // tile = 8 x 16 output pixels
constexpr int TC_TILE_H = TC_BM / TC_TILE_W;
// Sampler teams: a team of eight warps covers the 128 rows of a K-block,
// each warp one tile row of 16 pixels.  Two register budgets are built:
//  - two teams (18 warps, at most 96 registers a thread) that take
//    alternate K-blocks, each warp with the corner loads of its next
//    K-block in flight while it waits for its stage;
//  - one team (10 warps, 168 registers: three warps share a scheduler's
//    16 K registers) whose warps take every K-block with the loads of the
//    next two in flight, so every load has a whole K-block of the warp's
//    own work to land in.
#ifndef DCN_TC_TEAMS
#define DCN_TC_TEAMS 2
#endif
constexpr int TC_TEAMS = DCN_TC_TEAMS;
static_assert(TC_TEAMS == 1 || TC_TEAMS == 2, "one or two sampler teams");
constexpr int TC_TEAM_WARPS = 8;
constexpr int TC_SAMPLER_WARPS = TC_TEAM_WARPS * TC_TEAMS;
constexpr int TC_DEPTH = TC_TEAMS == 1 ? 2 : 1;               // K-blocks of loads in flight per warp
constexpr int TC_EPI_PARTS = TC_SAMPLER_WARPS / 4;            // epilogue column parts per lane quarter
constexpr int TC_CTRL_WARPS = 2;                              // TMA producer, MMA issuer
constexpr int TC_THREADS = 32 * (TC_CTRL_WARPS + TC_SAMPLER_WARPS);
constexpr int TC_MAX_REGS = TC_TEAMS == 1 ? 168 : 96;
constexpr int TC_A_COLS = TC_BK / 2;                          // TMEM columns of one A stage
constexpr int TC_TAP_GROUP = 32 / TC_TILE_W;                  // taps tabulated together (one per 16 lanes)
constexpr int TC_TABLE_SLOTS = 2 * TC_TAP_GROUP;              // ring: one group in use, one ahead
static_assert(TC_TEAM_WARPS * TC_TILE_W == TC_BM, "a team covers the tile");
static_assert(TC_TABLE_SLOTS == 4 && TC_TAP_GROUP == 2, "ring index arithmetic assumes four slots");

// Per-warp sampling table of one K-block: one 16-byte entry per pixel of
// the warp's tile row (conflict-free writes, broadcast reads).  A sample is
// read as the clamped 2 x 2 block of tap_block.  An entry holds its four
// slot weights (mask folded in), the element index of its slot (0,0) at
// the K-block's first channel, and the limit of a lane's channel offset
// within the K-block.  For the 16-bit combine the weights are rounded to
// the operand type, two to a word, and all four fields share the entry;
// for the fp32 combine the weights are fp32 and fill the entry, and the
// index and limit sit in a second array.
constexpr int TC_ENTRY_ARRAY_BYTES = TC_TILE_W * 16;
__host__ __device__ constexpr int table_buf_bytes(bool f32) { return (f32 ? 2 : 1) * TC_ENTRY_ARRAY_BYTES; }

struct TcLayout {
    int stages;
    int b_bytes;       // O * 128: one weight K-block
    int bar_off;       // barriers after the stages
    int table_off;     // per-warp corner tables
    int vt_off;        // virtual-tap table, int4 per (tap, offset group)
    int bias_off;      // the bias, fp32 per output channel (zero without one)
    int total;         // bytes used from the 1024-aligned base
};

__host__ __device__ inline TcLayout tc_layout(int O, int stages, bool f32, int vtaps) {
    TcLayout L;
    L.stages = stages;
    L.b_bytes = O * TC_BK * 2;
    L.bar_off = stages * L.b_bytes;
    // full[stages], empty[stages], acc_full[2], acc_free[2], tmem slot (8 bytes each)
    L.table_off = L.bar_off + (2 * stages + 5) * 8;
    L.table_off = (L.table_off + 15) & ~15;
    L.vt_off = L.table_off + TC_SAMPLER_WARPS * TC_TABLE_SLOTS * table_buf_bytes(f32);
    L.bias_off = L.vt_off + vtaps * 16;
    L.total = L.bias_off + O * 4;
    return L;
}

// TMEM columns: the fp32 accumulator [128 x O] from column 0, twice when
// both copies and the A stages fit the 512 columns (a tile's epilogue then
// overlaps the next tile's K-blocks), then the A stages, TC_A_COLS columns
// each.
__host__ __device__ inline int tmem_acc_cols(int O) { return (O + 31) & ~31; }
__host__ __device__ inline int tmem_acc_bufs(int O, int stages) {
    return 2 * tmem_acc_cols(O) + stages * TC_A_COLS <= 512 ? 2 : 1;
}
__host__ __device__ inline int tmem_cols_for(int O, int stages) {
    const int need = tmem_acc_bufs(O, stages) * tmem_acc_cols(O) + stages * TC_A_COLS;
    int n = 32;
    while (n < need) n <<= 1;
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

// Walk position j of a tile's K-blocks -> (channel block, virtual tap):
// returns j / vtaps and sets vt = j % vtaps.  rcp is 1.0f / vtaps; for j
// below 2^22 the float quotient is off by at most one, which the two
// corrections take back.
__device__ __forceinline__ int walk_split(int j, int vtaps, float rcp, int &vt) {
    int q = __float2int_rz(__int2float_rn(j) * rcp);
    int r = j - q * vtaps;
    if (r < 0) { --q; r += vtaps; }
    if (r >= vtaps) { ++q; r -= vtaps; }
    vt = r;
    return q;
}

template <bool kSampleF32, bool kF16>
__global__ void __maxnreg__(TC_MAX_REGS)
dcn_tc_kernel(const __grid_constant__ CUtensorMap wmap, Params p, int stages) {
    using E = Elem16<kF16>;   // the 16-bit operand type: its packed arithmetic and MMA format
    constexpr int kBuf = table_buf_bytes(kSampleF32);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const TcLayout L = tc_layout(p.O, stages, kSampleF32, p.kh * p.kw * p.og_count);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + stages);
    // acc_full[b]: the MMAs of a segment using accumulator b are complete;
    // acc_free[b]: all sampler warps have read accumulator b out
    const uint32_t acc_full0 = smem_u32(bars + 2 * stages);
    const uint32_t acc_free0 = smem_u32(bars + 2 * stages + 2);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * stages + 4);

    // the warp index, broadcast so that the compiler treats everything
    // derived from it as warp-uniform (uniform registers)
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x / 32), 0);
    const int lane = threadIdx.x % 32;
    const int tiles_x = (p.Wo + TC_TILE_W - 1) / TC_TILE_W;
    const int tiles_y = (p.Ho + TC_TILE_H - 1) / TC_TILE_H;
    // channel blocks of the launch; with C % 64 != 0 the last block of each
    // tap is completed with zeros (the packed weight is zero there too)
    const int ncb = (p.C + TC_BK - 1) / TC_BK;
    const int taps = p.kh * p.kw;
    const int nkb = taps * ncb;
    // Virtual taps: (tap, offset group) pairs, each with its own offsets and
    // mask, of vncb channel blocks each; packed-weight K-block vt * vncb + cb.
    // A tile walks its K-blocks block-major: position j = cb * vtaps + vt,
    // every virtual tap of channel block 0, then of block 1, ...  Between
    // two taps that read a corner pixel the L1 then holds one 128-byte line
    // of it (its 64 channels of the block), not the vncb lines of all its
    // channels.
    const int vtaps = taps * p.og_count;
    const int vncb = ncb / p.og_count;
    const float vt_rcp = 1.0f / static_cast<float>(vtaps);
    const int total = p.B * tiles_x * tiles_y * nkb;
    const int u_begin = blockIdx.x * p.units_per_cta;
    const int u_end = min(u_begin + p.units_per_cta, total);
    const int tmem_cols = tmem_cols_for(p.O, stages);
    const int acc_bufs = tmem_acc_bufs(p.O, stages);
    const uint32_t acc_cols = tmem_acc_cols(p.O);
    const uint32_t a_col0 = acc_bufs * acc_cols;

    // virtual-tap table: {i*dil_h - pad_h, j*dil_w - pad_w, mask plane
    // og*taps + tap of the launch's offset groups, channel offset of the
    // offset group's first block}
    int4 *vt_tab = reinterpret_cast<int4 *>(smem + L.vt_off);
    for (int vt = threadIdx.x; vt < vtaps; vt += blockDim.x) {
        const int tap = vt / p.og_count;
        const int og = vt - tap * p.og_count;
        const int i = tap / p.kw;
        const int j = tap - i * p.kw;
        vt_tab[vt] = make_int4(i * p.dh - p.ph, j * p.dw - p.pw, og * taps + tap, og * vncb * TC_BK);
    }
    float *bias_tab = reinterpret_cast<float *>(smem + L.bias_off);
    for (int o = threadIdx.x; o < p.O; o += blockDim.x) bias_tab[o] = p.bias ? __ldg(p.bias + o) : 0.0f;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1 + TC_TEAM_WARPS);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full0 + 8 * b, 1);
            mbar_init(acc_free0 + 8 * b, TC_SAMPLER_WARPS);
        }
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
            // walk position u_begin % nkb as (virtual tap, channel block)
            int vt, cb = walk_split(u_begin % nkb, vtaps, vt_rcp, vt);
            // The packed weight may still be in the making when this grid
            // was launched as the pack's programmatic dependent: wait for
            // that grid to complete (a no-op for an ordinary launch).
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int u = u_begin; u < u_end; ++u) {
                if (!mbar_wait_sleep(empty0 + 8 * s, phase ^ 1, p.status, p.timeout_ns)) break;
                const uint32_t b_dst = smem_u32(smem + s * L.b_bytes);
                mbar_arrive_expect_tx(full0 + 8 * s, L.b_bytes);
                tma_load_2d(b_dst, &wmap, full0 + 8 * s, (vt * vncb + cb) * TC_BK, 0);
                ++issued;
                if (++vt == vtaps) {
                    vt = 0;
                    if (++cb == vncb) cb = 0;
                }
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
            const uint32_t idesc = E::idesc(TC_BM, p.O);
            int s = 0;
            uint32_t phase = 0;
            int segs = 0;
            Segment sg;
            int u = u_begin;
            bool live = true;
            while (live && next_segment(u, u_end, nkb, sg)) {
                // segment segs accumulates in buffer b, its use n of that buffer;
                // use n >= 1 waits until the samplers have read use n - 1 out
                const int b = segs % acc_bufs, n = segs / acc_bufs;
                if (n > 0 && !mbar_wait_sleep(acc_free0 + 8 * b, (n - 1) & 1, p.status, p.timeout_ns)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * acc_cols;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!mbar_wait_sleep(full0 + 8 * s, phase, p.status, p.timeout_ns)) { live = false; break; }
                    tc_fence_after_sync();
                    const uint32_t a_tmem = tmem_base + a_col0 + s * TC_A_COLS;
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(smem + s * L.b_bytes));
#pragma unroll
                    for (int ks = 0; ks < TC_BK / TC_MMA_K; ++ks) {
                        // K=16 steps: 8 TMEM columns of A, 32 bytes of the
                        // swizzled B rows; the segment's first MMA
                        // overwrites the accumulator
                        mma_kind_f16_ts(d_tmem, a_tmem + ks * (TC_MMA_K / 2), bdesc + 2 * ks, idesc,
                                    (kb > sg.kb0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(empty0 + 8 * s);
                    if (++s == stages) { s = 0; phase ^= 1; }
                }
                // the segment's accumulator is complete once its MMAs are
                mma_commit(acc_full0 + 8 * b);
                ++segs;
            }
            // the MMAs must be complete before TMEM is released
            if (segs > 0) {
                const int last = segs - 1;
                mbar_wait_sleep(acc_full0 + 8 * (last % acc_bufs), (last / acc_bufs) & 1, p.status,
                                p.timeout_ns);
            }
        }
    } else {
        // ------------------------------------------------ samplers
        const int sw = warp - TC_CTRL_WARPS;             // sampler warp 0 .. TC_SAMPLER_WARPS - 1
        const int q = warp & 3;                          // TMEM lane quarter this warp may access
        const int team = sw / TC_TEAM_WARPS;             // takes units u_begin + team + TC_TEAMS * i
        const int half = (sw % TC_TEAM_WARPS) / 4;       // which 16 lanes of the quarter
        const int trow = 2 * q + half;                   // its tile row = A rows 16 trow .. +15
        const uint16_t *__restrict__ x = static_cast<const uint16_t *>(p.x);   // 16-bit elements
        const uint32_t table_s = smem_u32(smem + L.table_off + sw * TC_TABLE_SLOTS * kBuf);
        const uint32_t vt_s = smem_u32(smem + L.vt_off);
        const uint32_t a_lane = static_cast<uint32_t>(16 * trow) << 16;
        const int plane = p.plane;                       // offset / mask plane stride
        const int my_g = lane >> 4;     // geometry: tap of the group
        const int my_px = lane & 15;    // geometry: pixel (tile column)
        const int quart16 = (lane & 3) * 16;   // gather: the lane's 16 channels of the K-block
        // A lane whose 16 channels lie past the last one (C % 64 != 0, last
        // block) reads the last 16 real channels instead: finite data in
        // bounds, which the packed weight's zero rows cancel in the MMA.
        const int chan_last = p.C - 16;
        const int rsub = lane >> 2;     // gather: pixels rsub and rsub + 8 of the row
        const uint32_t r_off0 = rsub * 16;
        constexpr uint32_t r_off1_rel = 8 * 16;                 // pixel rsub + 8's entry, after rsub's
        // element steps from a sample block's slot (0,0) to slots (0,1) and (1,0)
        const int step_x = p.W > 1 ? p.x_cstride : 0;
        const int step_y = p.H > 1 ? p.W * p.x_cstride : 0;
        bool ok = true;
        int s = team;                   // this warp's stages: team, team + TC_TEAMS, ...
        uint32_t phase = 0;

        // Epilogue (S5) of segment e, the idx-th of this CTA: wait for its
        // accumulator, read it out, then tell the MMA warp it is free.
        auto epilogue = [&](const Segment &e, int idx) {
            // TMEM lane quarter, column part, A row of this thread
            const int part = sw >> 2;                        // 0 .. TC_EPI_PARTS - 1
            const int erow = q * 32 + lane;
            const int nch = p.O / 16;
            const int ch_begin = part * nch / TC_EPI_PARTS;
            const int ch_end = (part + 1) * nch / TC_EPI_PARTS;
            const size_t part_floats = static_cast<size_t>(nch) * TC_BM * 16;   // one partial tile
            const int etb = e.tile / (tiles_x * tiles_y);
            const int erem = e.tile - etb * tiles_x * tiles_y;
            const int eth0 = (erem / tiles_x) * TC_TILE_H;
            const int etw0 = (erem % tiles_x) * TC_TILE_W;
            const uint32_t b = idx % acc_bufs;
            if (ok) ok = mbar_wait_sleep(acc_full0 + 8 * b, (idx / acc_bufs) & 1, p.status, p.timeout_ns);
            __syncwarp();
            tc_fence_after_sync();
                const int oh = eth0 + erow / TC_TILE_W;
                const int ow = etw0 + erow % TC_TILE_W;
                const bool pix_valid = oh < p.Ho && ow < p.Wo;
                const size_t pix = (static_cast<size_t>(etb) * p.Ho + oh) * p.Wo + ow;
                const uint32_t acc_lane = (static_cast<uint32_t>(q * 32) << 16) + b * acc_cols;
                if (e.kb0 > 0) {
                    // The tile's other K-blocks belong to the CTA before this one:
                    // leave the fp32 partial for it and raise this CTA's flag.
                    float *dst = p.partial + static_cast<size_t>(blockIdx.x) * part_floats;
                    for (int ch = ch_begin; ch < ch_end; ++ch) {
                        float vv[16];
                        tmem_ld16(tmem_base + acc_lane + ch * 16, vv);
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
                    const bool merge = e.kb1 < nkb;
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
                    uint16_t *__restrict__ out = static_cast<uint16_t *>(p.out);
                    for (int ch = ch_begin; ch < ch_end; ++ch) {
                        float vv[16];
                        tmem_ld16(tmem_base + acc_lane + ch * 16, vv);
                        if (merge && ok) {
                            const float *sp = src + (static_cast<size_t>(ch) * TC_BM + erow) * 16;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float4 a = ld_cg_f4(sp + 4 * e);
                                vv[4 * e] += a.x; vv[4 * e + 1] += a.y; vv[4 * e + 2] += a.z; vv[4 * e + 3] += a.w;
                            }
                        }
                        if (ok && pix_valid) {
                            // + bias in fp32 (from its shared-memory copy), rounded
                            // once to the operand type
                            const uint32_t bs = smem_u32(smem + L.bias_off) + ch * 64;
                            uint32_t pk[8];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float4 bb = lds_v4_f32(bs + 16 * e);
                                pk[2 * e] = E::pack(vv[4 * e] + bb.x, vv[4 * e + 1] + bb.y);
                                pk[2 * e + 1] = E::pack(vv[4 * e + 2] + bb.z, vv[4 * e + 3] + bb.w);
                            }
                            uint4 *dst = reinterpret_cast<uint4 *>(out + pix * p.out_stride + ch * 16);
#ifdef DCN_CHECK_BOUNDS
                            if (in_bounds(dst, 32, p.out_lo, p.out_hi, p.status))
#endif
                            {
                                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                            }
                        }
                    }
                }
            // this warp's TMEM reads are complete: accumulator b is free
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free0 + 8 * b);
        };

        // One pass per segment, plus one to finish: the pass for segment i
        // samples it and then runs the epilogue of segment i (one
        // accumulator) or of segment i - 1 (two: the MMA drain and the
        // read-out then overlap with sampling).
        const bool deferred = acc_bufs == 2;
        Segment sg, prev;
        int u = u_begin;
        for (int seg_idx = 0;; ++seg_idx) {
          const bool got = next_segment(u, u_end, nkb, sg);
          if (got) {
            // ---- this segment's tile
            const int tb = sg.tile / (tiles_x * tiles_y);
            const int trem = sg.tile - tb * tiles_x * tiles_y;
            const int th0 = (trem / tiles_x) * TC_TILE_H;
            const int tw0 = (trem % tiles_x) * TC_TILE_W;
            // this warp's K-blocks: every TC_TEAMS-th from the first of its team
            const int seg_u0 = sg.tile * nkb + sg.kb0;
            const int kb_first = sg.kb0 + (team - (seg_u0 - u_begin) % TC_TEAMS + TC_TEAMS) % TC_TEAMS;
            if (kb_first < sg.kb1) {
                const int my_h = th0 + trow;
                const int my_w = tw0 + my_px;
                const bool my_valid = (my_h < p.Ho) && (my_w < p.Wo);
                const int my_hw = my_valid ? my_h * p.Wo + my_w : 0;
                // the image's first offset and mask planes
                const float *off_img = p.offset + static_cast<size_t>(tb) * p.off_bstride * plane;
                const float *mask_img = p.mask ? p.mask + static_cast<size_t>(tb) * p.mask_bstride * plane
                                               : p.offset;
                const int y_base = (p.h0 + my_h) * p.sh;
                const int x_base = my_w * p.sw;
                const int n = (sg.kb1 - kb_first + TC_TEAMS - 1) / TC_TEAMS;   // this warp's K-blocks
                const uint32_t tl = table_s + r_off0;           // this lane's first entry in slot 0

                // Walk position of the raw inputs this lane loaded last, as
                // (virtual tap, channel block): the lane's loads are walk
                // positions kb_first + TC_TEAMS * (2g + my_g), g = 0, 1, ...,
                // each one 2 * TC_TEAMS after the one before.  A load and the
                // tabulation of what it loaded alternate, so the table entry
                // is always made from the most recent load.
                int r_vt;
                int r_cb = walk_split(kb_first + TC_TEAMS * my_g, vtaps, vt_rcp, r_vt);
                // Raw inputs (dy, dx, mask) of the lane's next walk position
                // (its first when `first`) for its pixel, loaded into
                // registers a pair ahead of their use.
                float r_dy = 0.0f, r_dx = 0.0f, r_m = 0.0f;
                int4 r_e = make_int4(0, 0, 0, 0);   // the position's virtual-tap entry
                auto load_raw = [&](bool first) {
                    if (!first) {
                        r_vt += 2 * TC_TEAMS;
                        while (r_vt >= vtaps) { r_vt -= vtaps; ++r_cb; }
                    }
                    const bool valid = my_valid && r_cb < vncb;                  // j < nkb
                    r_e = lds_v4_s32_m(vt_s + r_vt * 16);
                    const int mc = r_e.z;                            // mask plane; offsets 2mc, 2mc + 1
                    const float *o = off_img + (2 * mc * plane + my_hw);
                    const float *mp = mask_img + (mc * plane + my_hw);
#ifdef DCN_CHECK_BOUNDS
                    // an offset or mask outside its tensor is not read (zero)
                    r_dy = valid && in_bounds(o, 4, p.off_lo, p.off_hi, p.status) ? __ldg(o) : 0.0f;
                    r_dx = valid && in_bounds(o + plane, 4, p.off_lo, p.off_hi, p.status) ? __ldg(o + plane) : 0.0f;
                    r_m = !p.mask ? 1.0f
                          : (valid && in_bounds(mp, 4, p.mask_lo, p.mask_hi, p.status) ? __ldg(mp) : 0.0f);
#else
                    r_dy = valid ? __ldg(o) : 0.0f;
                    r_dx = valid ? __ldg(o + plane) : 0.0f;
                    r_m = !p.mask ? 1.0f : (valid ? __ldg(mp) : 0.0f);
#endif
                };
                // The table entry of the last loaded walk position for this
                // lane's pixel, in ring slot `slot`: the sample block's slot
                // weights, the element index of its slot (0,0) at the
                // K-block's first channel, and the limit of a lane's channel
                // offset in the K-block (a lane past the last channel reads
                // the last 16 instead).  A position past the last one gets an
                // entry that is never read.
                auto tabulate = [&](int slot) {
                    const float dy = r_dy, dx = r_dx, m = r_m;
                    const int4 e = r_e;
                    TapBlock t;
                    tap_block(dy, dx, m, y_base + e.x, x_base + e.y, tb, p.H, p.W, p.x_cstride, t);
                    const int c0 = e.w + r_cb * TC_BK;
                    const uint32_t ent = table_s + slot * kBuf + my_px * 16;
                    if constexpr (kSampleF32) {
                        sts_v4_b32_m(ent, __float_as_uint(t.w[0]), __float_as_uint(t.w[1]),
                                     __float_as_uint(t.w[2]), __float_as_uint(t.w[3]));
                        sts_v2_b32_m(ent + TC_ENTRY_ARRAY_BYTES, static_cast<uint32_t>(t.idx + c0),
                                     static_cast<uint32_t>(chan_last - c0));
                    } else {
                        sts_v4_b32_m(ent, E::pack(t.w[0], t.w[1]), E::pack(t.w[2], t.w[3]),
                                     static_cast<uint32_t>(t.idx + c0), static_cast<uint32_t>(chan_last - c0));
                    }
                };
                // The corner-row loads of both of this lane's pixels from the
                // entries in ring slot `slot`: each sample block's four slots
                // from the index of its slot (0,0), every one inside the image,
                // advanced by the lane's channel offset.
                auto issue = [&](int slot, u32x8 (&v)[8]) {
                    const uint32_t ent = tl + slot * kBuf + (kSampleF32 ? TC_ENTRY_ARRAY_BYTES : 8);
#pragma unroll
                    for (int px = 0; px < 2; ++px) {
                        const uint2 ei = lds_v2_u32(ent + (px ? r_off1_rel : 0u));
                        const int e0 = static_cast<int>(ei.x) + min(quart16, static_cast<int>(ei.y));
                        const int e1 = e0 + step_x;
                        const int e2 = e0 + step_y;
                        const int e3 = e2 + step_x;
#ifdef DCN_CHECK_BOUNDS
                        // a corner row outside x is read from x's first bytes instead
                        auto chk = [&](const uint16_t *a) {
                            return in_bounds(a, 32, p.x_lo, p.x_hi, p.status)
                                       ? a : static_cast<const uint16_t *>(p.x_lo);
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
                };
                // Wait for the current stage, combine the loaded corners with
                // the weights in ring slot `slot` and store the stage row of
                // both pixels (S3), 16 words in the order of one 16x256b.x4
                // store: w[4k], w[4k+1] are words 2k, 2k+1 (channels 4k .. 4k+3
                // of the lane's 16) of the first pixel, w[4k+2], w[4k+3] those
                // of the second.
                auto combine_store = [&](int slot, const u32x8 (&v)[8], uint2 p0, uint2 p1) -> bool {
                    // every lane waits; the warp leaves together if any lane ran out
                    const bool got = mbar_wait_sleep(empty0 + 8 * s, phase ^ 1, p.status, p.timeout_ns, 2000u);
                    if (!__all_sync(0xffffffffu, got)) return false;
                    // TMEM writes after the MMAs that read this stage
                    tc_fence_after_sync();
                    // the weights of both pixels
                    const uint32_t taddr = tmem_base + a_lane + a_col0 + s * TC_A_COLS;
                    if constexpr (kSampleF32) {
                        uint64_t c[2][4];
#pragma unroll
                        for (int px = 0; px < 2; ++px) {
                            const float4 cw = lds_v4_f32(tl + slot * kBuf + (px ? r_off1_rel : 0u));
                            c[px][0] = f2_make(cw.x, cw.x); c[px][1] = f2_make(cw.y, cw.y);
                            c[px][2] = f2_make(cw.z, cw.z); c[px][3] = f2_make(cw.w, cw.w);
                        }
                        // repeat k of the 16x256b store: words 2k, 2k+1 of both pixels
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t r[4];
#pragma unroll
                            for (int px = 0; px < 2; ++px) {
                                const u32x8 *vp = v + 4 * px;
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int m = 2 * k + h;
                                    // channels 2m, 2m+1: the four slots' weighted sum in fp32
                                    uint64_t acc = f2_mul(c[px][0], f2_make(E::lo(vp[0].w[m]), E::hi(vp[0].w[m])));
                                    acc = f2_fma(c[px][1], f2_make(E::lo(vp[1].w[m]), E::hi(vp[1].w[m])), acc);
                                    acc = f2_fma(c[px][2], f2_make(E::lo(vp[2].w[m]), E::hi(vp[2].w[m])), acc);
                                    acc = f2_fma(c[px][3], f2_make(E::lo(vp[3].w[m]), E::hi(vp[3].w[m])), acc);
                                    r[2 * px + h] = E::pack_f2(acc);
                                }
                            }
                            tmem_st_16x256b_x1(taddr + 8 * k, r[0], r[1], r[2], r[3]);
                        }
                    } else {
                        const int4 cw0 = make_int4(splat_lo(p0.x), splat_hi(p0.x), splat_lo(p0.y), splat_hi(p0.y));
                        const int4 cw1 = make_int4(splat_lo(p1.x), splat_hi(p1.x), splat_lo(p1.y), splat_hi(p1.y));
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t r[4];
#pragma unroll
                            for (int px = 0; px < 2; ++px) {
                                const u32x8 *vp = v + 4 * px;
                                const int4 cw = px ? cw1 : cw0;
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    // the same sum in the input dtype: 16-bit weights, one
                                    // rounding per fused multiply-add, two channels per op
                                    const int m = 2 * k + h;
                                    uint32_t acc = E::mul(cw.x, vp[0].w[m]);
                                    acc = E::fma(cw.y, vp[1].w[m], acc);
                                    acc = E::fma(cw.z, vp[2].w[m], acc);
                                    acc = E::fma(cw.w, vp[3].w[m], acc);
                                    r[2 * px + h] = acc;
                                }
                            }
                            tmem_st_16x256b_x1(taddr + 8 * k, r[0], r[1], r[2], r[3]);
                        }
                    }
                    return true;
                };
                // This stage's row is written: release it to the MMA warp.
                auto finish_stage = [&]() {
                    tmem_wait_st();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full0 + 8 * s);
                    s += TC_TEAMS;
                    if (s >= stages) { s -= stages; phase ^= 1; }
                };
                // The loads of this warp's next TC_DEPTH K-blocks are in flight
                // while one is combined; with two in flight va and vb alternate.
                u32x8 va[8], vb[8];   // (vb unused with one K-block in flight)
                u32x8 (&v_odd)[8] = TC_DEPTH == 2 ? vb : va;

                // This warp's K-block jj of the segment is walk position
                // j = kb_first + TC_TEAMS * jj, its table in ring slot jj % 4.
                // Tables are made in pairs of the warp's sequence {2g, 2g + 1}
                // (slots 2g % 4 and 2g % 4 + 1, one per half-warp), so in a
                // body unrolled by four K-blocks every slot is a constant.
                auto load_pair = [&](int g) { load_raw(g == 0); };
                auto tab_pair = [&](int g) { tabulate((2 * g + my_g) & (TC_TABLE_SLOTS - 1)); };
                load_pair(0);
                tab_pair(0);
                if (2 < n) { load_pair(1); tab_pair(1); }
                if (4 < n) load_pair(2);
                __syncwarp();
                issue(0, va);
                if constexpr (TC_DEPTH == 2) {
                    if (n > 1) issue(1, vb);
                }
                // K-block jj = base + k in ring slot k; at an even k (past the
                // segment's first K-block) the pair after next is tabulated
                // into the slots the last pair used; then the loads of
                // K-block jj + TC_DEPTH.  (Issuing those loads before the
                // tabulation was measured slower: the tabulation's shared
                // reads then queue behind them.)
                auto step = [&](int jj, int k, u32x8 (&v)[8]) -> bool {
                    // this K-block's weights, read before the stage wait
                    const uint2 p0 = lds_v2_u32(tl + k * kBuf);
                    const uint2 p1 = lds_v2_u32(tl + k * kBuf + r_off1_rel);
                    if (!combine_store(k, v, p0, p1)) return false;
                    if ((k & 1) == 0 && jj > 0 && jj + 2 < n) {
                        const int g = jj / 2 + 1;
                        tab_pair(g);
                        if (2 * g + 2 < n) load_pair(g + 1);
                        __syncwarp();
                    }
                    if (jj + TC_DEPTH < n) issue((k + TC_DEPTH) & (TC_TABLE_SLOTS - 1), v);
                    finish_stage();
                    return true;
                };
                for (int jj = 0; jj < n; jj += 4) {
                    if (!step(jj, 0, va)) { ok = false; break; }
                    if (jj + 1 >= n) break;
                    if (!step(jj + 1, 1, v_odd)) { ok = false; break; }
                    if (jj + 2 >= n) break;
                    if (!step(jj + 2, 2, va)) { ok = false; break; }
                    if (jj + 3 >= n) break;
                    if (!step(jj + 3, 3, v_odd)) { ok = false; break; }
                }
            }

          }
          if (deferred ? seg_idx > 0 : got)
              epilogue(deferred ? prev : sg, deferred ? seg_idx - 1 : seg_idx);
          if (!got) break;
          prev = sg;
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

// The dynamic shared-memory size last set on each device for each
// instantiation [fp32 combine][fp16 operands].
PerDeviceValue<> g_max_smem_set[2][2];

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

// Shared memory the CTA may use (weight stages + tables + alignment + the
// 1 KB the system reserves).  The SM's L1/shared array is 256 KB.  With
// O = 64 a 140 KB budget gives eight stages (107 KB; the carveout then
// leaves 124 KB of L1 for the corner gathers): measured against six stages
// in 100 KB (156 KB of L1), the 7x7 workload 114.7 -> 112.6 us and the
// boundary 5x5 157.7 -> 151.6 us; ten stages in the same L1 and twelve
// with 92 KB of L1 were no better.  Wide weights (large O) may take up to
// the second budget to keep four stages.
#ifndef DCN_TC_SMEM_BUDGET
#define DCN_TC_SMEM_BUDGET (140 * 1024)
#endif
#ifndef DCN_TC_SMEM_WIDE_BUDGET
#define DCN_TC_SMEM_WIDE_BUDGET (164 * 1024)
#endif

// Launch with the cooperative attribute (all CTAs co-resident, for the
// stream-K flags) and/or as a programmatic dependent of the previous kernel.
template <typename Kernel>
cudaError_t launch_ex(Kernel kernel, int grid, int smem, cudaStream_t stream, bool cooperative,
                      bool dependent, const CUtensorMap &wmap, const Params &p, int stages) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    if (dependent) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, wmap, p, stages);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e;
}

}  // namespace

bool tc_supported(int C, int O) {
    return C % 16 == 0 && C > 0 && O % 16 == 0 && O >= 16 && O <= 256;
}

cudaError_t launch_tc(const Params &p_in, const CUtensorMap &wmap, cudaStream_t stream,
                      bool after_pack) {
    // One CTA per SM.  Its shared memory is kept small so that most of the
    // SM's L1/shared array stays L1 cache, which holds a good part of the
    // tile's corner footprint across taps.
    Params p = p_in;
    const bool f32 = p.sample_f32 != 0;
    // A multiple of TC_TEAMS stages (with two teams each owns every other
    // one), as many as fit the budget and TMEM, at most 8.
    // A channel count that is not a multiple of 64 (zero-completed last
    // block) only with one offset group per launch.
    const int vtaps = p.kh * p.kw * p.og_count;
    const int ncb = (p.C + TC_BK - 1) / TC_BK;
    if (vtaps > tc_max_virtual_taps || p.og_count <= 0 || !tc_supported(p.C, p.O) ||
        (p.og_count > 1 && (p.C % TC_BK != 0 || ncb % p.og_count != 0)) || p.K != p.kh * p.kw * ncb * TC_BK)
        return cudaErrorInvalidValue;
    auto smem_for = [&](int st) { return tc_layout(p.O, st, f32, vtaps).total + 1024 + 1024; };
    auto tmem_fits = [&](int st) { return tmem_acc_cols(p.O) + st * TC_A_COLS <= 512; };
    int stages = 2;
    for (int st = 8; st > 2; st -= TC_TEAMS) {
        if (tmem_fits(st) && smem_for(st) <= DCN_TC_SMEM_BUDGET) { stages = st; break; }
    }
    if (stages < 4 && tmem_fits(4) && smem_for(4) <= DCN_TC_SMEM_WIDE_BUDGET) stages = 4;
    const TcLayout L = tc_layout(p.O, stages, f32, vtaps);
    const int smem = L.total + 1024;  // slack for 1024-byte alignment
    const bool f16 = p.f16 != 0;
    using KernelFn = void (*)(const CUtensorMap, Params, int);
    static const KernelFn kKernels[2][2] = {
        {dcn_tc_kernel<false, false>, dcn_tc_kernel<false, true>},
        {dcn_tc_kernel<true, false>, dcn_tc_kernel<true, true>}};
    const KernelFn kernel = kKernels[f32 ? 1 : 0][f16 ? 1 : 0];
    int dev = 0;
    cudaError_t ae = cudaGetDevice(&dev);
    if (ae != cudaSuccess) return ae;
    ae = static_cast<cudaError_t>(g_max_smem_set[f32 ? 1 : 0][f16 ? 1 : 0].ensure(dev, smem, [&] {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        // ask for just enough shared memory for the one resident CTA (plus
        // the 1 KB the system reserves per CTA); the rest stays L1
        return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    carveout_percent(smem + 1024));
    }));
    if (ae != cudaSuccess) return ae;
    const int tiles = p.B * ((p.Ho + TC_TILE_H - 1) / TC_TILE_H) * ((p.Wo + TC_TILE_W - 1) / TC_TILE_W);
    const int nkb = p.kh * p.kw * ncb;
    const long long total = static_cast<long long>(tiles) * nkb;
    if (p.partial && p.flags && tiles > p.sm_count && p.sm_count > 0) {
        // Stream-K: every CTA (one per SM, all resident) takes an equal run
        // of (tile, K-block) units, so no SM idles through a last partial
        // wave; a tile split between two CTAs is merged by the first.
        const int units = static_cast<int>((total + p.sm_count - 1) / p.sm_count);
        p.units_per_cta = units;
        const int grid = static_cast<int>((total + units - 1) / units);
        const cudaError_t e = launch_ex(kernel, grid, smem, stream, true, after_pack, wmap, p, stages);
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        cudaGetLastError();   // not all CTAs could be resident: one tile per CTA instead
    }
    // one tile per CTA
    p.units_per_cta = nkb;
    return launch_ex(kernel, tiles, smem, stream, false, after_pack, wmap, p, stages);
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
