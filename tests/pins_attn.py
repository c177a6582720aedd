"""Pins of the single-scale deformable sampling oracle: checks against what
the mathematics, a library routine and the separately pinned convolution
oracle fix, independently of this oracle's own code.

- the operator is a depthwise deformable convolution with unit weights, G
  offset groups and the aggregation weights as the mask: the convolution
  oracle (pinned on its own) on those inputs;
- the library bilinear resampler (torch grid_sample, zero padding, fp64)
  per group and tap, then the weighted sum (softmax by torch in fp64);
- integer offsets: every sample is one pixel of the map, exactly;
- every corner outside: exactly 0;
- a constant map sampled inside with softmax weights: the constant;
- hand-derived samples and weighted sums on a 2x3 map, and on a
  two-group 5x5 map with stride 2 and dilation 2
  (tests/golden/attn_samples.txt), exact in binary.
"""

import os

import numpy as np
import torch
import torch.nn.functional as F

# (B, H, W, G, D, kernel, stride, padding, dilation)
CASES = [
    (2, 9, 11, 2, 3, (3, 3), (1, 1), (1, 1), (1, 1)),
    (1, 12, 10, 3, 2, (3, 2), (2, 1), (1, 0), (1, 2)),
    (1, 7, 8, 1, 4, (1, 1), (1, 1), (0, 0), (1, 1)),
    (2, 10, 9, 4, 1, (5, 3), (2, 2), (2, 1), (2, 1)),
]


def _out_size(n, k, s, p, d):
    return (n + 2 * p - d * (k - 1) - 1) // s + 1


def _problem(seed, B, H, W, G, D, kernel, stride, padding, dilation, offset_std=1.5):
    g = torch.Generator().manual_seed(seed)
    kh, kw = kernel
    Ho = _out_size(H, kh, stride[0], padding[0], dilation[0])
    Wo = _out_size(W, kw, stride[1], padding[1], dilation[1])
    K = kh * kw
    value = torch.randn(B, H, W, G, D, generator=g)
    off = torch.randn(B, Ho, Wo, G, K, 2, generator=g) * offset_std
    w = torch.randn(B, Ho, Wo, G, K, generator=g)
    return value, off, w, Ho, Wo


def _rel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))


def pin_attn_depthwise_convolution(orc):
    from oracle import ConvDesc
    for n, (B, H, W, G, D, kernel, stride, padding, dilation) in enumerate(CASES):
        value, off, w, Ho, Wo = _problem(700 + n, B, H, W, G, D, kernel, stride, padding, dilation)
        kh, kw = kernel
        K, C = kh * kw, G * D
        x = value.reshape(B, H, W, C).permute(0, 3, 1, 2).contiguous()
        # offset group q's planes: 2 (q K + k) = dy, 2 (q K + k) + 1 = dx
        offset = off.permute(0, 3, 4, 5, 1, 2).reshape(B, 2 * G * K, Ho, Wo).contiguous()
        weight = torch.ones(C, 1, kh, kw)
        conv = ConvDesc(stride=stride, padding=padding, dilation=dilation, groups=C, offset_groups=G)
        for softmax in (False, True):
            a = torch.softmax(w.double(), dim=-1).float() if softmax else w
            mask = a.permute(0, 3, 4, 1, 2).reshape(B, G * K, Ho, Wo).contiguous()
            ref = orc.forward_ex(x, offset, mask, weight, None, conv)        # [B, C, Ho, Wo]
            ref = ref.transpose(0, 2, 3, 1).reshape(B, Ho, Wo, G, D)
            got = orc.attn_forward(value, off, a if softmax else w, kernel, stride, padding,
                                   dilation, softmax=False)
            err = _rel(got, ref)
            assert err <= 1e-12, f"attn vs depthwise convolution, case {n}: {err:.3e}"
            if softmax:
                # the operator's own softmax against torch's, rounded to fp32
                got_sm = orc.attn_forward(value, off, w, kernel, stride, padding, dilation,
                                          softmax=True)
                assert _rel(got_sm, ref) <= 1e-6, f"attn softmax, case {n}"


def _grid_sample_reference(value, off, w, kernel, stride, padding, dilation, softmax):
    B, H, W, G, D = value.shape
    _, Ho, Wo, _, K, _ = off.shape
    kh, kw = kernel
    a = torch.softmax(w.double(), dim=-1) if softmax else w.double()
    out = torch.zeros(B, Ho, Wo, G, D, dtype=torch.float64)
    hs = torch.arange(Ho).view(Ho, 1) * stride[0] - padding[0]
    ws = torch.arange(Wo).view(1, Wo) * stride[1] - padding[1]
    for g in range(G):
        inp = value[:, :, :, g, :].double().permute(0, 3, 1, 2)          # [B, D, H, W]
        for k in range(K):
            i, j = k // kw, k % kw
            # the oracle's fp32 coordinates
            py = ((hs + i * dilation[0]).float() + off[:, :, :, g, k, 0]).double()
            px = ((ws + j * dilation[1]).float() + off[:, :, :, g, k, 1]).double()
            grid = torch.stack([(2.0 * px + 1.0) / W - 1.0, (2.0 * py + 1.0) / H - 1.0], dim=-1)
            samp = F.grid_sample(inp, grid, mode="bilinear", padding_mode="zeros",
                                 align_corners=False)                     # [B, D, Ho, Wo]
            out[:, :, :, g, :] += samp.permute(0, 2, 3, 1) * a[:, :, :, g, k].unsqueeze(-1)
    return out.numpy()


def pin_attn_grid_sample(orc):
    for n, (B, H, W, G, D, kernel, stride, padding, dilation) in enumerate(CASES):
        value, off, w, _, _ = _problem(720 + n, B, H, W, G, D, kernel, stride, padding, dilation)
        for softmax in (False, True):
            got = orc.attn_forward(value, off, w, kernel, stride, padding, dilation, softmax)
            ref = _grid_sample_reference(value, off, w, kernel, stride, padding, dilation, softmax)
            err = _rel(got, ref)
            assert err <= 1e-10, f"attn grid_sample case {n} softmax={softmax}: {err:.3e}"


def pin_attn_integer_offsets(orc):
    B, H, W, G, D, kernel, stride, padding, dilation = CASES[1]
    value, off, w, Ho, Wo = _problem(740, B, H, W, G, D, kernel, stride, padding, dilation)
    off = torch.round(off * 2.0)
    got = orc.attn_forward(value, off, w, kernel, stride, padding, dilation, False)
    kh, kw = kernel
    v = value.double().numpy()
    exp = np.zeros_like(got)
    for b in range(B):
        for ho in range(Ho):
            for wo in range(Wo):
                for g in range(G):
                    for k in range(kh * kw):
                        i, j = k // kw, k % kw
                        y = ho * stride[0] - padding[0] + i * dilation[0] + int(off[b, ho, wo, g, k, 0])
                        x = wo * stride[1] - padding[1] + j * dilation[1] + int(off[b, ho, wo, g, k, 1])
                        if 0 <= y < H and 0 <= x < W:
                            exp[b, ho, wo, g] += float(w[b, ho, wo, g, k]) * v[b, y, x, g]
    assert _rel(got, exp) <= 1e-13


def pin_attn_outside(orc):
    B, H, W, G, D, kernel, stride, padding, dilation = CASES[0]
    value, off, w, _, _ = _problem(750, B, H, W, G, D, kernel, stride, padding, dilation)
    off[..., 1] = torch.where(torch.rand(off[..., 1].shape) < 0.5, -float(W + 3), float(2 * W + 3))
    for softmax in (False, True):
        got = orc.attn_forward(value, off, w, kernel, stride, padding, dilation, softmax)
        assert not np.any(got)


def pin_attn_constant(orc):
    B, H, W, G, D, kernel, stride, padding, dilation = (1, 12, 14, 3, 4, (3, 3), (1, 1), (1, 1), (1, 1))
    value, off, w, Ho, Wo = _problem(760, B, H, W, G, D, kernel, stride, padding, dilation)
    const = torch.randn(G, D)
    value = const.view(1, 1, 1, G, D).expand_as(value).contiguous()
    # positions within half a pixel of the tap, clamped into [0, H-1] x [0, W-1]:
    # every corner with a nonzero weight is inside, so the softmax-weighted
    # sum is the constant
    kh, kw = kernel
    for k in range(kh * kw):
        i, j = k // kw, k % kw
        by = (torch.arange(Ho) * stride[0] - padding[0] + i * dilation[0]).view(1, Ho, 1, 1).float()
        bx = (torch.arange(Wo) * stride[1] - padding[1] + j * dilation[1]).view(1, 1, Wo, 1).float()
        r = torch.rand(B, Ho, Wo, G, 2) - 0.5
        off[..., k, 0] = (by + r[..., 0]).clamp(0.0, H - 1.0) - by
        off[..., k, 1] = (bx + r[..., 1]).clamp(0.0, W - 1.0) - bx
    got = orc.attn_forward(value, off, w, kernel, stride, padding, dilation, True)
    exp = const.double().numpy()[None, None, None].repeat(Ho, 1).repeat(Wo, 2)
    assert np.abs(got - exp).max() <= 1e-12 * np.abs(exp).max()


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "attn_samples.txt")


def _golden():
    """The cases of the fixture: each a dict of the problem, the groups'
    maps, the taps (k, dy, dx, samples per group) and the weight vectors
    (weights, softmax, expected per group)."""
    cases = []
    with open(GOLDEN) as fh:
        for line in fh:
            f = line.split("#", 1)[0].split()
            if not f:
                continue
            if f[0] == "case":
                H, W, G, sh, sw, ph, pw, dh, dw, h, w = (int(v) for v in f[1:12])
                cases.append({"H": H, "W": W, "G": G, "stride": (sh, sw), "padding": (ph, pw),
                              "dilation": (dh, dw), "pixel": (h, w), "maps": {}, "taps": [],
                              "weights": []})
            elif f[0] == "map":
                c = cases[-1]
                c["maps"][int(f[1])] = [float(v) for v in f[2:]]
                assert len(c["maps"][int(f[1])]) == c["H"] * c["W"]
            elif f[0] == "tap":
                cases[-1]["taps"].append((int(f[1]), float(f[2]), float(f[3]),
                                          [float(v) for v in f[4:]]))
            elif f[0] == "weights":
                cases[-1]["weights"].append(([float(v) for v in f[1:10]], f[10] == "softmax",
                                             [float(v) for v in f[11:]]))
    return cases


def pin_attn_golden(orc):
    """Hand-derived samples and weighted sums at one output pixel per case
    (tests/golden/attn_samples.txt): each tap alone (a one-hot weight) gives
    its sample in every group, exactly, and each weight vector its sum."""
    for n, c in enumerate(_golden()):
        H, W, G, K = c["H"], c["W"], c["G"], 9
        kernel, stride, padding, dilation = (3, 3), c["stride"], c["padding"], c["dilation"]
        Ho = _out_size(H, 3, stride[0], padding[0], dilation[0])
        Wo = _out_size(W, 3, stride[1], padding[1], dilation[1])
        h, w = c["pixel"]
        value = torch.stack([torch.tensor(c["maps"][g], dtype=torch.float32).view(H, W)
                             for g in range(G)], dim=-1).view(1, H, W, G, 1)
        off = torch.zeros(1, Ho, Wo, G, K, 2)
        for k, dy, dx, _ in c["taps"]:
            off[0, h, w, :, k, 0], off[0, h, w, :, k, 1] = dy, dx
        for k, dy, dx, samples in c["taps"]:
            a = torch.zeros(1, Ho, Wo, G, K)
            a[0, h, w, :, k] = 1.0
            got = orc.attn_forward(value, off, a, kernel, stride, padding, dilation, False)
            for g in range(G):
                v = float(got[0, h, w, g, 0])
                assert v == samples[g], f"case {n + 1} tap {k} group {g}: {v} != {samples[g]}"
        for weights, softmax, expected in c["weights"]:
            a = torch.zeros(1, Ho, Wo, G, K)
            a[0, h, w, :] = torch.tensor(weights)
            got = orc.attn_forward(value, off, a, kernel, stride, padding, dilation, softmax)
            for g in range(G):
                v = float(got[0, h, w, g, 0])
                assert abs(v - expected[g]) <= 1e-12 * max(1.0, abs(expected[g])), \
                    f"case {n + 1} weights {weights} softmax={softmax} group {g}: {v} != {expected[g]}"


ALL_ATTN_PINS = [pin_attn_depthwise_convolution, pin_attn_grid_sample, pin_attn_integer_offsets,
                 pin_attn_outside, pin_attn_constant, pin_attn_golden]
