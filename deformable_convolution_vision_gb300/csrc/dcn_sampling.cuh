// Per-(pixel, tap) sampling geometry shared by the forward kernels.
//
// The rule (page "litert-community/Idol ... deform_conv.py", module
// docstring and the four-corner loop of deform_conv2d_gather): output pixel
// (h, w), tap (i, j) samples the input at
//   py = (h - pad + i) + dy,  px = (w - pad + j) + dx       (fp32)
// bilinearly from corners (y0 + a, x0 + e), y0 = floor(py), x0 = floor(px),
// with weights (1-ly)(1-lx), (1-ly)lx, ly(1-lx), ly*lx, and every corner
// outside the image contributes 0.  With stride, per-axis padding and
// dilation (the convolution reading of torchvision deform_conv2d, which the
// "deformops 3.0.1" page names) the integer part of the coordinate is
// h*stride_h - pad_h + i*dil_h, likewise for w.  The mask scales the whole
// sample, so it is folded into the four corner weights here.
#pragma once

#include <cstdint>

namespace dcn {

struct TapCorners {
    float w[4];    // corner weights, mask folded in, 0 for outside corners
    int idx[4];    // element offset of the corner's channel row in x (NHWC),
                   // clamped inside the image so every load is in bounds
};

// y_base = h*stride_h - pad_h + i*dil_h, x_base likewise; cstride = the
// element distance between neighbouring pixels of x.
__device__ __forceinline__ void tap_corners(float dy, float dx, float m, int y_base, int x_base,
                                            int b, int H, int W, int cstride, TapCorners &t) {
    float py = static_cast<float>(y_base) + dy;
    float px = static_cast<float>(x_base) + dx;
    // Coordinates below -1 or above H (W) leave every corner outside, so
    // clamping to [-2, H+1] changes no result; it keeps the integer
    // conversion in range for huge or non-finite offsets (NaN -> -2).
    py = fminf(fmaxf(py, -2.0f), static_cast<float>(H + 1));
    px = fminf(fmaxf(px, -2.0f), static_cast<float>(W + 1));
    const float fy = floorf(py);
    const float fx = floorf(px);
    const float ly = py - fy;
    const float lx = px - fx;
    const int y0 = static_cast<int>(fy);
    const int x0 = static_cast<int>(fx);
    // a corner row / column is inside when 0 <= index < H (W)
    const bool vy0 = static_cast<unsigned>(y0) < static_cast<unsigned>(H);
    const bool vy1 = static_cast<unsigned>(y0 + 1) < static_cast<unsigned>(H);
    const bool vx0 = static_cast<unsigned>(x0) < static_cast<unsigned>(W);
    const bool vx1 = static_cast<unsigned>(x0 + 1) < static_cast<unsigned>(W);
    // row weights carry the mask; a corner outside gets weight 0
    const float wy0 = vy0 ? (1.0f - ly) * m : 0.0f;
    const float wy1 = vy1 ? ly * m : 0.0f;
    const float wx0 = vx0 ? 1.0f - lx : 0.0f;
    const float wx1 = vx1 ? lx : 0.0f;
    t.w[0] = wy0 * wx0;
    t.w[1] = wy0 * wx1;
    t.w[2] = wy1 * wx0;
    t.w[3] = wy1 * wx1;
    // clamped corner addresses: the top-left one, then steps of one column
    // and one row that are 0 where the clamp folds both corners together
    const int yc0 = min(max(y0, 0), H - 1);
    const int xc0 = min(max(x0, 0), W - 1);
    const int dxc = (x0 + 1 >= 1 && x0 + 1 <= W - 1) ? cstride : 0;      // xc1 - xc0, in elements
    const int dyc = (y0 + 1 >= 1 && y0 + 1 <= H - 1) ? W * cstride : 0;  // yc1 - yc0, in elements
    t.idx[0] = ((b * H + yc0) * W + xc0) * cstride;
    t.idx[1] = t.idx[0] + dxc;
    t.idx[2] = t.idx[0] + dyc;
    t.idx[3] = t.idx[2] + dxc;
}

// The same sample read as a 2 x 2 block of pixels that always lies inside
// the image: rows yb, yb + sy and columns xb, xb + sx with sy = (H > 1),
// sx = (W > 1).  Each corner inside the image falls on one of the block's
// four slots and carries its weight there; a slot that no inside corner
// falls on has weight 0.  No slot receives two corners, so the slot weights
// are the corner weights of tap_corners, each moved to the slot of its
// pixel, and a weighted sum over the slots equals the one over the corners.
// The block's fixed shape lets a reader form the four addresses from one
// index and two per-launch steps.
struct TapBlock {
    float w[4];    // slots (0,0), (0,sx), (sy,0), (sy,sx); mask folded in
    int idx;       // element offset of slot (0,0)'s channel row in x
};

// One axis: coordinate q in [-2, n+1] -> block start b in [0, max(n-2, 0)]
// and the weights of slots b and b + 1 (slot b + 1 only when n > 1).
__device__ __forceinline__ void axis_block(float q, int n, int &b, float &w0, float &w1) {
    const float f = floorf(q);
    const float l = q - f;
    const int i0 = static_cast<int>(f);          // corners i0 (weight 1 - l) and i0 + 1 (weight l)
    b = min(max(i0, 0), max(n - 2, 0));
    // corner i0 lies on slot d = i0 - b: d == 0 puts both corners inside, on
    // slots 0 and 1; d == -1 (i0 = -1) leaves corner i0 + 1 on slot 0;
    // d == 1 (i0 = n - 1) leaves corner i0 on slot 1; otherwise both are outside
    const int d = i0 - b;
    const float u = 1.0f - l;
    w0 = d == 0 ? u : (d == -1 ? l : 0.0f);
    w1 = d == 0 ? l : (d == 1 ? u : 0.0f);
    if (n == 1) w1 = 0.0f;                       // no second slot: corner i0 + 1 is outside
}

__device__ __forceinline__ void tap_block(float dy, float dx, float m, int y_base, int x_base,
                                          int b, int H, int W, int cstride, TapBlock &t) {
    float py = static_cast<float>(y_base) + dy;
    float px = static_cast<float>(x_base) + dx;
    // as in tap_corners: the clamp changes no result and keeps the integer
    // conversion in range for huge or non-finite offsets
    py = fminf(fmaxf(py, -2.0f), static_cast<float>(H + 1));
    px = fminf(fmaxf(px, -2.0f), static_cast<float>(W + 1));
    int yb, xb;
    float wy0, wy1, wx0, wx1;
    axis_block(py, H, yb, wy0, wy1);
    axis_block(px, W, xb, wx0, wx1);
    wy0 *= m;
    wy1 *= m;
    t.w[0] = wy0 * wx0;
    t.w[1] = wy0 * wx1;
    t.w[2] = wy1 * wx0;
    t.w[3] = wy1 * wx1;
    t.idx = ((b * H + yb) * W + xb) * cstride;
}

}  // namespace dcn
