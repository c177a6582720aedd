"""Pins of the MSDA oracle: checks against what the mathematics and a
library routine fix, independently of the oracle's own code.

- the library bilinear resampler (torch.nn.functional.grid_sample, zero
  padding, align_corners=False, fp64) per head and level, then the weighted
  sum (softmax by torch in fp64);
- locations at pixel centres: every sample is one value row, exactly;
- locations whose corners are all outside: output exactly 0;
- a constant value map sampled inside every level with softmax weights:
  the constant (the weights sum to one);
- one-hot weights on one level of a map whose levels hold different
  constants: that level's constant (catches level offsets and shapes);
- hand-derived samples and weighted sums on a two-level map of two heads
  (tests/golden/msda_samples.txt), exact in binary.
"""

import os

import numpy as np
import torch
import torch.nn.functional as F

LEVELS = [
    ([[8, 8], [4, 4]], 2, 3),                     # (shapes, K points, heads)
    ([[6, 10], [3, 5], [2, 2]], 4, 2),
    ([[16, 12], [8, 6], [4, 3], [2, 2]], 4, 1),
]


def _starts(shapes):
    s, out = 0, []
    for h, w in shapes:
        out.append(s)
        s += h * w
    return out, s


def _problem(seed, shapes, K, G, B=2, Q=7, D=5):
    g = torch.Generator().manual_seed(seed)
    starts, S = _starts(shapes)
    L = len(shapes)
    value = torch.randn(B, S, G, D, generator=g)
    # locations slightly beyond [0, 1] too, so some corners fall outside
    loc = torch.rand(B, Q, G, L, K, 2, generator=g) * 1.2 - 0.1
    w = torch.randn(B, Q, G, L * K, generator=g)
    return value, starts, loc, w


def _reference(value, shapes, starts, loc, w, softmax):
    B, S, G, D = value.shape
    _, Q, _, L, K, _ = loc.shape
    a = torch.softmax(w.double(), dim=-1) if softmax else w.double()
    out = torch.zeros(B, Q, G, D, dtype=torch.float64)
    for l, (H, W) in enumerate(shapes):
        lvl = value[:, starts[l]:starts[l] + H * W].double().view(B, H, W, G, D)
        for g in range(G):
            inp = lvl[:, :, :, g, :].permute(0, 3, 1, 2)                   # [B, D, H, W]
            # the oracle's fp32 pixel coordinates, mapped so that grid_sample
            # (align_corners=False) lands on them
            px = loc[:, :, g, l, :, 0] * float(W) - 0.5
            py = loc[:, :, g, l, :, 1] * float(H) - 0.5
            gx = (2.0 * px.double() + 1.0) / W - 1.0
            gy = (2.0 * py.double() + 1.0) / H - 1.0
            grid = torch.stack([gx, gy], dim=-1)                          # [B, Q, K, 2]
            samp = F.grid_sample(inp, grid, mode="bilinear", padding_mode="zeros",
                                 align_corners=False)                     # [B, D, Q, K]
            aw = a[:, :, g, l * K:(l + 1) * K]                            # [B, Q, K]
            out[:, :, g, :] += torch.einsum("bdqk,bqk->bqd", samp, aw)
    return out.numpy()


def _rel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))


def pin_msda_grid_sample(orc):
    for n, (shapes, K, G) in enumerate(LEVELS):
        for softmax in (False, True):
            value, starts, loc, w = _problem(500 + n, shapes, K, G)
            got = orc.msda_forward(value, shapes, starts, loc, w, softmax)
            ref = _reference(value, shapes, starts, loc, w, softmax)
            err = _rel(got, ref)
            assert err <= 1e-10, f"msda grid_sample {shapes} softmax={softmax}: {err:.3e}"


def pin_msda_pixel_centres(orc):
    shapes, K, G = [[8, 8], [4, 4], [2, 2]], 3, 2
    value, starts, loc, w = _problem(520, shapes, K, G)
    g = torch.Generator().manual_seed(521)
    B, Q = loc.shape[0], loc.shape[1]
    idx = torch.zeros(B, Q, G, len(shapes), K, 2, dtype=torch.long)
    for l, (H, W) in enumerate(shapes):
        ix = torch.randint(0, W, (B, Q, G, K), generator=g)
        iy = torch.randint(0, H, (B, Q, G, K), generator=g)
        idx[:, :, :, l, :, 0], idx[:, :, :, l, :, 1] = ix, iy
        loc[:, :, :, l, :, 0] = (ix.float() + 0.5) / W
        loc[:, :, :, l, :, 1] = (iy.float() + 0.5) / H
    got = orc.msda_forward(value, shapes, starts, loc, w, False)
    exp = np.zeros_like(got)
    for b in range(B):
        for q in range(Q):
            for gg in range(G):
                for l, (H, W) in enumerate(shapes):
                    for k in range(K):
                        x, y = idx[b, q, gg, l, k].tolist()
                        exp[b, q, gg] += float(w[b, q, gg, l * K + k]) * \
                            value[b, starts[l] + y * W + x, gg].double().numpy()
    assert _rel(got, exp) <= 1e-13


def pin_msda_outside(orc):
    shapes, K, G = [[6, 10], [3, 5]], 4, 2
    value, starts, loc, w = _problem(530, shapes, K, G)
    loc[..., 0] = torch.where(torch.rand(loc[..., 0].shape) < 0.5, -0.6, 1.7)
    got = orc.msda_forward(value, shapes, starts, loc, w, True)
    assert not np.any(got)


def pin_msda_constant(orc):
    shapes, K, G = [[16, 12], [8, 6], [4, 4]], 4, 2
    value, starts, loc, w = _problem(540, shapes, K, G)
    const = torch.randn(G, value.shape[3])
    value = const.view(1, 1, G, -1).expand_as(value).contiguous()
    # every sample at least half a pixel inside, so all four corners count
    for l, (H, W) in enumerate(shapes):
        loc[:, :, :, l, :, 0] = (1.0 + torch.rand(loc[:, :, :, l, :, 0].shape) * (W - 2)) / W
        loc[:, :, :, l, :, 1] = (1.0 + torch.rand(loc[:, :, :, l, :, 1].shape) * (H - 2)) / H
    got = orc.msda_forward(value, shapes, starts, loc, w, True)
    exp = const.double().numpy()[None, None].repeat(got.shape[0], 0).repeat(got.shape[1], 1)
    assert np.abs(got - exp).max() <= 1e-12 * np.abs(exp).max()


def pin_msda_levels(orc):
    shapes, K, G = [[6, 10], [3, 5], [2, 2]], 2, 1
    value, starts, loc, w = _problem(550, shapes, K, G)
    lv = torch.tensor([3.0, -5.0, 7.0])
    for l, (H, W) in enumerate(shapes):
        value[:, starts[l]:starts[l] + H * W] = lv[l]
        loc[:, :, :, l, :, 0] = (1.0 + torch.rand(loc[:, :, :, l, :, 0].shape) * (W - 2)) / W
        loc[:, :, :, l, :, 1] = (1.0 + torch.rand(loc[:, :, :, l, :, 1].shape) * (H - 2)) / H
    for l in range(len(shapes)):
        w1 = torch.zeros_like(w)
        w1[..., l * K] = 1.0
        got = orc.msda_forward(value, shapes, starts, loc, w1, False)
        assert np.allclose(got, float(lv[l]), rtol=0, atol=1e-13), f"level {l}"


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "msda_samples.txt")


def _golden():
    levels, points, queries = [], [], []
    with open(GOLDEN) as fh:
        for line in fh:
            f = line.split("#", 1)[0].split()
            if not f:
                continue
            if f[0] == "level":
                H, W = int(f[1]), int(f[2])
                levels.append((H, W, [float(v) for v in f[3:]]))
                assert len(levels[-1][2]) == H * W
            elif f[0] == "point":
                points.append((int(f[1]), int(f[2]), float(f[3]), float(f[4]), float(f[5])))
            elif f[0] == "query":
                queries.append(([float(v) for v in f[1:5]], f[5] == "softmax", float(f[6])))
    return levels, points, queries


def pin_msda_golden(orc):
    """Hand-derived samples and weighted sums (tests/golden/msda_samples.txt),
    exact in binary: each point alone (a one-hot weight) gives its sample,
    and each query its weighted sum; head 1 holds ten times head 0's values
    and gives ten times its results."""
    levels, points, queries = _golden()
    shapes = [[H, W] for H, W, _ in levels]
    starts, S = _starts(shapes)
    L, K, G = len(levels), 2, 2
    head0 = torch.tensor([v for _, _, vals in levels for v in vals], dtype=torch.float32)
    value = torch.stack([head0, 10.0 * head0], dim=-1).view(1, S, G, 1)
    loc = torch.zeros(1, 1, G, L, K, 2)
    for l, k, x, y, _ in points:
        loc[0, 0, :, l, k, 0], loc[0, 0, :, l, k, 1] = x, y
    for l, k, x, y, sample in points:
        w = torch.zeros(1, 1, G, L * K)
        w[..., l * K + k] = 1.0
        got = orc.msda_forward(value, shapes, starts, loc, w, False)[0, 0, :, 0]
        for g in range(G):
            want = sample * 10.0 ** g
            assert float(got[g]) == want, \
                f"point (level {l}, k {k}) at ({x}, {y}) head {g}: {float(got[g])} != {want}"
    for weights, softmax, expected in queries:
        w = torch.tensor(weights, dtype=torch.float32).view(1, 1, 1, L * K).repeat(1, 1, G, 1)
        got = orc.msda_forward(value, shapes, starts, loc, w, softmax)[0, 0, :, 0]
        for g in range(G):
            want = expected * 10.0 ** g
            assert abs(float(got[g]) - want) <= 1e-12 * max(1.0, abs(want)), \
                f"query {weights} softmax={softmax} head {g}: {float(got[g])} != {want}"


ALL_MSDA_PINS = [pin_msda_grid_sample, pin_msda_pixel_centres, pin_msda_outside,
                 pin_msda_constant, pin_msda_levels, pin_msda_golden]
