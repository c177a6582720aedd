// Layout copies for callers with NCHW tensors (the torchvision argument
// layout that page "deformops 3.0.1", section "torchvision drop-in", keeps
// for its drop-in function): NCHW <-> NHWC, as a batched 2-D transpose
// [B][R][S] -> [B][S][R] (R = C, S = H*W one way; R = H*W, S = C the
// other).  32 x 32 tiles through shared memory (one padding column against
// bank conflicts), so that both the reads and the writes are coalesced.
// Pure data movement, bound by HBM: 2 x bytes per call.
#include <cstdint>

#include "dcn_kernels.h"

namespace dcn {

namespace {

constexpr int TR_TILE = 32;
constexpr int TR_ROWS = 8;

template <typename T>
__global__ void __launch_bounds__(TR_TILE * TR_ROWS)
transpose_kernel(const T *__restrict__ src, T *__restrict__ dst, int R, int S) {
    __shared__ T tile[TR_TILE][TR_TILE + 1];
    const size_t plane = static_cast<size_t>(R) * S;
    const T *in = src + blockIdx.z * plane;
    T *out = dst + blockIdx.z * plane;
    const int s0 = blockIdx.x * TR_TILE, r0 = blockIdx.y * TR_TILE;
    // read rows r0.. of the [R][S] matrix, S contiguous
    for (int dr = threadIdx.y; dr < TR_TILE; dr += TR_ROWS) {
        const int r = r0 + dr, s = s0 + threadIdx.x;
        if (r < R && s < S) tile[dr][threadIdx.x] = in[static_cast<size_t>(r) * S + s];
    }
    __syncthreads();
    // write rows s0.. of the [S][R] matrix, R contiguous
    for (int ds = threadIdx.y; ds < TR_TILE; ds += TR_ROWS) {
        const int s = s0 + ds, r = r0 + threadIdx.x;
        if (s < S && r < R) out[static_cast<size_t>(s) * R + r] = tile[threadIdx.x][ds];
    }
}

}  // namespace

cudaError_t launch_transpose(const void *src, void *dst, int B, int R, int S, int esize,
                             cudaStream_t stream) {
    const dim3 grid((S + TR_TILE - 1) / TR_TILE, (R + TR_TILE - 1) / TR_TILE, B);
    const dim3 block(TR_TILE, TR_ROWS);
    if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidValue;
    if (esize == 4)
        transpose_kernel<uint32_t><<<grid, block, 0, stream>>>(static_cast<const uint32_t *>(src),
                                                               static_cast<uint32_t *>(dst), R, S);
    else if (esize == 2)
        transpose_kernel<uint16_t><<<grid, block, 0, stream>>>(static_cast<const uint16_t *>(src),
                                                               static_cast<uint16_t *>(dst), R, S);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace dcn
