// Per-(pixel, tap) sampling geometry shared by the forward kernels.
//
// The rule (page "litert-community/Idol ... deform_conv.py", module
// docstring and the four-corner loop of deform_conv2d_gather): output pixel
// (h, w), tap (i, j) samples the input at
//   py = (h - pad + i) + dy,  px = (w - pad + j) + dx       (fp32)
// bilinearly from corners (y0 + a, x0 + e), y0 = floor(py), x0 = floor(px),
// with weights (1-ly)(1-lx), (1-ly)lx, ly(1-lx), ly*lx, and every corner
// outside the image contributes 0.  The mask scales the whole sample, so it
// is folded into the four corner weights here.
#pragma once

#include <cstdint>

namespace dcn {

struct TapCorners {
    float w[4];    // corner weights, mask folded in, 0 for outside corners
    int idx[4];    // element offset of the corner's channel row in x (NHWC),
                   // clamped inside the image so every load is in bounds
};

__device__ __forceinline__ void tap_corners(float dy, float dx, float m,
                                            int h, int w, int i, int j, int pad,
                                            int b, int H, int W, int C, TapCorners &t) {
    float py = static_cast<float>(h - pad + i) + dy;
    float px = static_cast<float>(w - pad + j) + dx;
    // Coordinates below -1 or above H (W) leave every corner outside, so
    // clamping to [-2, H+1] changes no result; it keeps the integer
    // conversion in range for huge or non-finite offsets (NaN -> -2).
    py = fminf(fmaxf(py, -2.0f), static_cast<float>(H + 1));
    px = fminf(fmaxf(px, -2.0f), static_cast<float>(W + 1));
    const float fy = floorf(py);
    const float fx = floorf(px);
    const float ly = py - fy;
    const float lx = px - fx;
    const float hy = 1.0f - ly;
    const float hx = 1.0f - lx;
    const int y0 = static_cast<int>(fy);
    const int x0 = static_cast<int>(fx);
    const int y1 = y0 + 1;
    const int x1 = x0 + 1;
    const bool vy0 = (y0 >= 0) && (y0 <= H - 1);
    const bool vy1 = (y1 >= 0) && (y1 <= H - 1);
    const bool vx0 = (x0 >= 0) && (x0 <= W - 1);
    const bool vx1 = (x1 >= 0) && (x1 <= W - 1);
    t.w[0] = (vy0 && vx0) ? hy * hx * m : 0.0f;
    t.w[1] = (vy0 && vx1) ? hy * lx * m : 0.0f;
    t.w[2] = (vy1 && vx0) ? ly * hx * m : 0.0f;
    t.w[3] = (vy1 && vx1) ? ly * lx * m : 0.0f;
    const int yc0 = min(max(y0, 0), H - 1);
    const int yc1 = min(max(y1, 0), H - 1);
    const int xc0 = min(max(x0, 0), W - 1);
    const int xc1 = min(max(x1, 0), W - 1);
    const int row0 = (b * H + yc0) * W;
    const int row1 = (b * H + yc1) * W;
    t.idx[0] = (row0 + xc0) * C;
    t.idx[1] = (row0 + xc1) * C;
    t.idx[2] = (row1 + xc0) * C;
    t.idx[3] = (row1 + xc1) * C;
}

}  // namespace dcn
