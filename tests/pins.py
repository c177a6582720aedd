"""Pins for the oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function takes an oracle object (``oracle.Oracle``) and
raises AssertionError when the oracle disagrees with an independent fact:

* zero offsets, mask 1: a library direct cross-correlation
  (torch.nn.functional.conv2d in fp64) -- the deformable sampling reduces to
  the regular 3x3 / 7x7 / kh x kw grid;
* per-tap integer offsets: a shifted convolution built from padding and
  slicing (bilinear weights collapse to 1 on the integer point and 0 on the
  other corners);
* hand-derived bilinear samples on tiny maps (tests/golden);
* fractional offsets in general: a library bilinear resampler with zero
  padding (torch.nn.functional.grid_sample, align_corners=True, fp64), one
  resample per tap, then the tap/channel contraction with einsum;
* samples pushed out of the image: exactly the bias;
* the mask: linearity, and mask 0 gives exactly the bias;
* an affine input map: bilinear interpolation reproduces it exactly;
* with stride, per-axis padding, dilation, weight groups and offset groups:
  zero offsets against the library convolution with those parameters,
  integer offsets against sliced shifted copies per offset group, fractional
  offsets against the library resampler per offset group, and identical
  offsets in every offset group against the one-group result.

The rule being pinned is the one on the page "litert-community/Idol ...
deform_conv.py" (module docstring and four-corner loop) and the page
"deformops 3.0.1", section "Deformable convolution" (torchvision
deform_conv2d, offsets (dy, dx) per kernel point, mask optional).
"""

import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand_problem(seed, B, C, H, W, O, kh, kw, pad, off_std, mask=True, bias=True):
    g = torch.Generator().manual_seed(seed)
    Ho, Wo = H + 2 * pad - kh + 1, W + 2 * pad - kw + 1
    k = kh * kw
    x = torch.randn(B, C, H, W, generator=g)
    off = torch.randn(B, 2 * k, Ho, Wo, generator=g) * off_std
    m = torch.rand(B, k, Ho, Wo, generator=g) * 2 if mask else None
    w = torch.randn(O, C, kh, kw, generator=g) * 0.3
    b = torch.randn(O, generator=g) if bias else None
    return x, off, m, w, b


def _rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = max(np.abs(ref).max(), 1e-300)
    return float(np.abs(got - ref).max() / scale)


# Shapes used by several pins: square and non-square kernels, 1x1, the 7x7
# ASPP kernel, ragged maps, pad 0 and pad > kernel radius.
SHAPES = [
    dict(B=2, C=3, H=7, W=9, O=4, kh=3, kw=3, pad=1),
    dict(B=1, C=2, H=6, W=5, O=3, kh=3, kw=5, pad=2),
    dict(B=1, C=4, H=8, W=8, O=2, kh=1, kw=1, pad=0),
    dict(B=1, C=2, H=9, W=10, O=2, kh=7, kw=7, pad=3),
    dict(B=1, C=2, H=5, W=6, O=3, kh=2, kw=3, pad=0),
]


def pin_direct_conv(orc):
    """Zero offsets with mask 1 (or no mask) equal a direct convolution."""
    for n, s in enumerate(SHAPES):
        x, off, m, w, b = _rand_problem(10 + n, off_std=0.0, **s)
        off.zero_()
        ref = F.conv2d(x.double(), w.double(), b.double(), padding=s["pad"])
        for mask in (None, torch.ones_like(m)):
            got = orc.forward(x, off, mask, w, b, s["pad"])
            err = _rel_err(got, ref.numpy())
            assert err <= 1e-13, f"direct conv {s} mask={mask is not None}: rel err {err:.3e}"


def _shift(xp, P, dy, dx, H_out, W_out, y_base, x_base):
    """x sampled at (y_base + h + dy, x_base + w + dx), zero outside; xp is x
    zero-padded by P on each side."""
    y0 = y_base + dy + P
    x0 = x_base + dx + P
    return xp[:, :, y0:y0 + H_out, x0:x0 + W_out]


def pin_shifted_conv(orc):
    """Per-tap integer offsets equal a convolution of shifted copies of x."""
    for n, s in enumerate(SHAPES):
        x, off, m, w, b = _rand_problem(20 + n, off_std=0.0, **s)
        kh, kw, pad = s["kh"], s["kw"], s["pad"]
        Ho, Wo = off.shape[2], off.shape[3]
        g = torch.Generator().manual_seed(200 + n)
        shifts = torch.randint(-3, 4, (kh * kw, 2), generator=g)
        for k in range(kh * kw):
            off[:, 2 * k] = float(shifts[k, 0])
            off[:, 2 * k + 1] = float(shifts[k, 1])
        P = 16
        xp = F.pad(x.double(), (P, P, P, P))
        ref = b.double().view(1, -1, 1, 1).expand(x.shape[0], -1, Ho, Wo).clone()
        for i in range(kh):
            for j in range(kw):
                k = i * kw + j
                xs = _shift(xp, P, int(shifts[k, 0]), int(shifts[k, 1]), Ho, Wo, i - pad, j - pad)
                ref += torch.einsum("oc,bchw->bohw", w[:, :, i, j].double(), xs) * m[:, k:k + 1].double()
        got = orc.forward(x, off, m, w, b, pad)
        err = _rel_err(got, ref.numpy())
        assert err <= 1e-13, f"shifted conv {s}: rel err {err:.3e}"


def pin_integer_gather(orc):
    """Per-pixel integer offsets equal a direct gather from the zero-padded map."""
    for n, s in enumerate(SHAPES):
        x, off, m, w, b = _rand_problem(30 + n, off_std=0.0, **s)
        kh, kw, pad = s["kh"], s["kw"], s["pad"]
        B, C, H, W = x.shape
        Ho, Wo = off.shape[2], off.shape[3]
        g = torch.Generator().manual_seed(300 + n)
        ioff = torch.randint(-4, 5, off.shape, generator=g)
        off = ioff.float()
        P = 32
        xp = F.pad(x.double(), (P, P, P, P))
        hh = torch.arange(Ho).view(Ho, 1)
        ww = torch.arange(Wo).view(1, Wo)
        ref = b.double().view(1, -1, 1, 1).expand(B, -1, Ho, Wo).clone()
        for bi in range(B):
            for i in range(kh):
                for j in range(kw):
                    k = i * kw + j
                    yy = hh - pad + i + ioff[bi, 2 * k] + P
                    xx = ww - pad + j + ioff[bi, 2 * k + 1] + P
                    samp = xp[bi][:, yy, xx]  # [C, Ho, Wo]
                    ref[bi] += torch.einsum("oc,chw->ohw", w[:, :, i, j].double(), samp) * m[bi, k].double()
        got = orc.forward(x, off, m, w, b, pad)
        err = _rel_err(got, ref.numpy())
        assert err <= 1e-13, f"integer gather {s}: rel err {err:.3e}"


def load_golden(path=None):
    """Parse tests/golden/bilinear_samples.txt into [(x_map, [(h, w, dy, dx, expected)])]."""
    path = path or os.path.join(GOLDEN, "bilinear_samples.txt")
    maps = []
    with open(path) as fh:
        for line in fh:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            if line[0] == "map":
                H, W = int(line[1]), int(line[2])
                vals = [float(v) for v in line[3:]]
                assert len(vals) == H * W
                maps.append((np.array(vals, dtype=np.float32).reshape(H, W), []))
            elif line[0] == "sample":
                h, w = int(line[1]), int(line[2])
                dy, dx, exp = float(line[3]), float(line[4]), float(line[5])
                maps[-1][1].append((h, w, dy, dx, exp))
    return maps


def pin_bilinear_golden(orc):
    """Hand-derived bilinear samples on tiny maps, exact."""
    maps = load_golden()
    assert maps and all(s for _, s in maps)
    for xmap, samples in maps:
        H, W = xmap.shape
        x = xmap.reshape(1, 1, H, W)
        w = np.ones((1, 1, 1, 1), dtype=np.float32)
        for h, ww, dy, dx, exp in samples:
            off = np.zeros((1, 2, H, W), dtype=np.float32)
            off[0, 0, h, ww] = dy
            off[0, 1, h, ww] = dx
            got = orc.forward(x, off, None, w, None, 0)[0, 0, h, ww]
            assert got == exp, f"golden ({h},{ww}) offset ({dy},{dx}): got {got}, expected {exp}"


def _sample_coords(off, kh, kw, pad, Ho, Wo):
    """fp32 sampling coordinates py, px [B, k, Ho, Wo] (the page builds its
    grid in the input dtype, fp32 here)."""
    B = off.shape[0]
    k = kh * kw
    o = off.view(B, k, 2, Ho, Wo)
    ki = torch.arange(kh).repeat_interleave(kw).view(1, k, 1, 1).float()
    kj = torch.arange(kw).repeat(kh).view(1, k, 1, 1).float()
    gy = torch.arange(Ho).view(1, 1, Ho, 1).float() - pad
    gx = torch.arange(Wo).view(1, 1, 1, Wo).float() - pad
    py = (gy + ki) + o[:, :, 0]
    px = (gx + kj) + o[:, :, 1]
    return py, px


def pin_grid_sample(orc):
    """General fractional offsets (many corners outside the image) equal
    torch's bilinear resampler with zero padding, then the contraction."""
    cases = [dict(s, off_std=2.5) for s in SHAPES if s["H"] > 1 and s["W"] > 1]
    cases.append(dict(B=2, C=3, H=6, W=11, O=5, kh=5, kw=5, pad=2, off_std=6.0))
    for n, s in enumerate(cases):
        s = dict(s)
        off_std = s.pop("off_std")
        x, off, m, w, b = _rand_problem(40 + n, off_std=off_std, **s)
        kh, kw, pad = s["kh"], s["kw"], s["pad"]
        B, C, H, W = x.shape
        Ho, Wo = off.shape[2], off.shape[3]
        py, px = _sample_coords(off, kh, kw, pad, Ho, Wo)
        ref = b.double().view(1, -1, 1, 1).expand(B, -1, Ho, Wo).clone()
        for i in range(kh):
            for j in range(kw):
                k = i * kw + j
                gx = px[:, k].double() * (2.0 / (W - 1)) - 1.0
                gy = py[:, k].double() * (2.0 / (H - 1)) - 1.0
                grid = torch.stack([gx, gy], dim=-1)  # [B, Ho, Wo, 2], (x, y)
                samp = F.grid_sample(x.double(), grid, mode="bilinear",
                                     padding_mode="zeros", align_corners=True)
                ref += torch.einsum("oc,bchw->bohw", w[:, :, i, j].double(),
                                    samp * m[:, k:k + 1].double())
        got = orc.forward(x, off, m, w, b, pad)
        err = _rel_err(got, ref.numpy())
        assert err <= 1e-10, f"grid_sample {s}: rel err {err:.3e}"


def pin_outside_is_bias(orc):
    """Offsets that push every corner out of the image contribute exactly 0;
    so do non-finite offsets."""
    for n, s in enumerate(SHAPES):
        x, off, m, w, b = _rand_problem(50 + n, off_std=0.0, **s)
        H, W, kh, kw = s["H"], s["W"], s["kh"], s["kw"]
        far = [(-(H + kh + 3), 0.3), (H + kh + 3, -0.7), (0.25, -(W + kw + 3)),
               (0.5, W + kw + 3.5), (float("inf"), 0.0), (0.0, float("-inf")),
               (float("nan"), 0.5), (1e30, -1e30)]
        for dy, dx in far:
            off[:, 0::2] = dy
            off[:, 1::2] = dx
            got = orc.forward(x, off, m, w, b, s["pad"])
            exp = np.broadcast_to(b.double().numpy().reshape(1, -1, 1, 1), got.shape)
            assert np.array_equal(got, exp), f"outside ({dy},{dx}) {s}: not exactly the bias"
            got0 = orc.forward(x, off, m, w, None, s["pad"])
            assert np.array_equal(got0, np.zeros_like(got0))


def pin_mask(orc):
    """The mask scales each tap linearly; mask 0 gives exactly the bias."""
    for n, s in enumerate(SHAPES):
        x, off, m, w, b = _rand_problem(60 + n, off_std=2.0, **s)
        base = orc.forward(x, off, m, w, b, s["pad"])
        # scaling by a power of two keeps the fp32 mask values exact
        scaled = orc.forward(x, off, m * 4.0, w, b, s["pad"])
        bb = b.double().numpy().reshape(1, -1, 1, 1)
        err = _rel_err(scaled - bb, 4.0 * (base - bb))
        assert err <= 1e-13, f"mask linearity {s}: {err:.3e}"
        zero = orc.forward(x, off, torch.zeros_like(m), w, b, s["pad"])
        assert np.array_equal(zero, np.broadcast_to(bb, zero.shape)), f"mask 0 {s}"
        # one tap's mask scaled by 4 moves the output by 3x that tap's share
        k = (s["kh"] * s["kw"]) // 2
        m1 = m.clone()
        m1[:, k] *= 4.0
        only = torch.zeros_like(m)
        only[:, k] = m[:, k]
        share = orc.forward(x, off, only, w, None, s["pad"])
        got = orc.forward(x, off, m1, w, b, s["pad"])
        err = _rel_err(got, base + 3.0 * share)
        assert err <= 1e-13, f"per-tap mask {s}: {err:.3e}"


def pin_affine_map(orc):
    """Bilinear interpolation reproduces an affine map exactly: with
    x[c, y, x] = a_c*y + b_c*x + c_c, a 1x1 kernel and an identity weight,
    every sample inside [0,H-1]x[0,W-1] equals a_c*py + b_c*px + c_c."""
    g = torch.Generator().manual_seed(70)
    C, H, W = 3, 9, 7
    a = torch.tensor([1.0, -2.0, 0.5])
    bx = torch.tensor([3.0, 0.25, -1.0])
    cc = torch.tensor([0.5, 1.0, -4.0])
    yy = torch.arange(H).view(1, H, 1).float()
    xx = torch.arange(W).view(1, 1, W).float()
    x = (a.view(C, 1, 1) * yy + bx.view(C, 1, 1) * xx + cc.view(C, 1, 1)).unsqueeze(0)
    off = (torch.rand(1, 2, H, W, generator=g) - 0.5) * 3.0
    w = torch.eye(C).view(C, C, 1, 1)
    got = orc.forward(x, off, None, w, None, 0)
    py, px = _sample_coords(off, 1, 1, 0, H, W)
    py, px = py[0, 0].double(), px[0, 0].double()
    inside = (py >= 0) & (py <= H - 1) & (px >= 0) & (px <= W - 1)
    assert inside.sum() > H * W // 3
    for c in range(C):
        exp = a[c].double() * py + bx[c].double() * px + cc[c].double()
        diff = (torch.from_numpy(got[0, c]) - exp).abs()[inside]
        assert float(diff.max()) <= 1e-12, f"affine map channel {c}: {float(diff.max()):.3e}"


# ------------------------------------------------------------------ general
# Stride, per-axis padding, dilation, weight groups and offset groups: the
# convolution reading of torchvision deform_conv2d's parameters, which the
# "deformops 3.0.1" page (section "Deformable convolution") names as the
# operator, with a (C_out, C_in / groups, kH, kW) weight.

GEN_SHAPES = [
    dict(B=2, C=4, H=9, W=11, O=6, kh=3, kw=3, stride=(2, 1), padding=(1, 2), dilation=(1, 2),
         groups=2, offset_groups=2),
    dict(B=1, C=6, H=10, W=8, O=3, kh=3, kw=2, stride=(1, 3), padding=(2, 0), dilation=(2, 1),
         groups=3, offset_groups=3),
    dict(B=1, C=4, H=12, W=12, O=4, kh=3, kw=3, stride=2, padding=1, dilation=2,
         groups=1, offset_groups=4),
    # offset groups that straddle weight groups (C/groups = 3, C/offset_groups = 2)
    dict(B=1, C=6, H=7, W=9, O=4, kh=2, kw=3, stride=1, padding=(0, 1), dilation=1,
         groups=2, offset_groups=3),
    dict(B=2, C=2, H=5, W=6, O=2, kh=1, kw=1, stride=2, padding=0, dilation=3,
         groups=1, offset_groups=2),
]


def _conv_desc(s):
    import oracle
    return oracle.ConvDesc(stride=s["stride"], padding=s["padding"], dilation=s["dilation"],
                           groups=s["groups"], offset_groups=s["offset_groups"])


def _pair(v):
    return (v, v) if isinstance(v, int) else tuple(v)


def _rand_problem_ex(seed, s, off_std, mask=True, bias=True):
    g = torch.Generator().manual_seed(seed)
    B, C, H, W, O, kh, kw = (s[k] for k in ("B", "C", "H", "W", "O", "kh", "kw"))
    Ho, Wo = _conv_desc(s).out_size(H, W, kh, kw)
    k, G = kh * kw, s["offset_groups"]
    x = torch.randn(B, C, H, W, generator=g)
    off = torch.randn(B, 2 * G * k, Ho, Wo, generator=g) * off_std
    m = torch.rand(B, G * k, Ho, Wo, generator=g) * 2 if mask else None
    w = torch.randn(O, C // s["groups"], kh, kw, generator=g) * 0.3
    b = torch.randn(O, generator=g) if bias else None
    return x, off, m, w, b


def _dense_tap_weight(w, groups, C, i, j):
    """[O, C] weight of tap (i, j) with zeros outside each output's group."""
    O, Cg = w.shape[0], w.shape[1]
    Og = O // groups
    Wd = torch.zeros(O, C, dtype=torch.float64)
    for o in range(O):
        g = o // Og
        Wd[o, g * Cg:(g + 1) * Cg] = w[o, :, i, j].double()
    return Wd


def pin_general_direct_conv(orc):
    """Zero offsets with mask 1 (or no mask) equal a library convolution with
    the same stride, padding, dilation and groups."""
    for n, s in enumerate(GEN_SHAPES):
        x, off, m, w, b = _rand_problem_ex(110 + n, s, off_std=0.0)
        off.zero_()
        ref = F.conv2d(x.double(), w.double(), b.double(), stride=_pair(s["stride"]),
                       padding=_pair(s["padding"]), dilation=_pair(s["dilation"]),
                       groups=s["groups"])
        for mask in (None, torch.ones_like(m)):
            got = orc.forward_ex(x, off, mask, w, b, _conv_desc(s))
            assert got.shape == tuple(ref.shape), f"{s}: shape {got.shape} != {tuple(ref.shape)}"
            err = _rel_err(got, ref.numpy())
            assert err <= 1e-13, f"general direct conv {s} mask={mask is not None}: {err:.3e}"


def _strided_samples(x, s, i, j, dy, dx, Ho, Wo):
    """x at (h*sh - ph + i*dh + dy, w*sw - pw + j*dw + dx) for integer dy,
    dx, zero outside: padding and strided slicing."""
    sh, sw = _pair(s["stride"])
    ph, pw = _pair(s["padding"])
    dh, dw = _pair(s["dilation"])
    P = 40
    xp = F.pad(x.double(), (P, P, P, P))
    y0 = -ph + i * dh + dy + P
    x0 = -pw + j * dw + dx + P
    return xp[:, :, y0:y0 + sh * (Ho - 1) + 1:sh, x0:x0 + sw * (Wo - 1) + 1:sw]


def pin_general_shifted_conv(orc):
    """Integer offsets, one shift per (offset group, tap), equal a sum over
    groups and taps of library-sliced shifted copies of x, contracted with
    each group's weight."""
    for n, s in enumerate(GEN_SHAPES):
        x, off, m, w, b = _rand_problem_ex(120 + n, s, off_std=0.0)
        B, C, H, W = x.shape
        kh, kw, G = s["kh"], s["kw"], s["offset_groups"]
        k_all, Cq = kh * kw, C // G
        Ho, Wo = off.shape[2], off.shape[3]
        gen = torch.Generator().manual_seed(1200 + n)
        shifts = torch.randint(-3, 4, (G, k_all, 2), generator=gen)
        for q in range(G):
            for k in range(k_all):
                off[:, 2 * (q * k_all + k)] = float(shifts[q, k, 0])
                off[:, 2 * (q * k_all + k) + 1] = float(shifts[q, k, 1])
        ref = b.double().view(1, -1, 1, 1).expand(B, -1, Ho, Wo).clone()
        for q in range(G):
            cs = slice(q * Cq, (q + 1) * Cq)
            for i in range(kh):
                for j in range(kw):
                    k = i * kw + j
                    samp = _strided_samples(x, s, i, j, int(shifts[q, k, 0]), int(shifts[q, k, 1]), Ho, Wo)
                    Wd = _dense_tap_weight(w, s["groups"], C, i, j)
                    ref += torch.einsum("oc,bchw->bohw", Wd[:, cs], samp[:, cs]) * \
                        m[:, q * k_all + k:q * k_all + k + 1].double()
        got = orc.forward_ex(x, off, m, w, b, _conv_desc(s))
        err = _rel_err(got, ref.numpy())
        assert err <= 1e-13, f"general shifted conv {s}: {err:.3e}"


def pin_general_grid_sample(orc):
    """Fractional offsets per offset group equal the library bilinear
    resampler on that group's channels, then the grouped contraction."""
    for n, s in enumerate(GEN_SHAPES):
        x, off, m, w, b = _rand_problem_ex(130 + n, s, off_std=2.5)
        B, C, H, W = x.shape
        kh, kw, G = s["kh"], s["kw"], s["offset_groups"]
        k_all, Cq = kh * kw, C // G
        sh, sw = _pair(s["stride"])
        ph, pw = _pair(s["padding"])
        dh, dw = _pair(s["dilation"])
        Ho, Wo = off.shape[2], off.shape[3]
        hh = torch.arange(Ho, dtype=torch.float32).view(1, Ho, 1)
        ww = torch.arange(Wo, dtype=torch.float32).view(1, 1, Wo)
        ref = b.double().view(1, -1, 1, 1).expand(B, -1, Ho, Wo).clone()
        for q in range(G):
            cs = slice(q * Cq, (q + 1) * Cq)
            for i in range(kh):
                for j in range(kw):
                    k = q * k_all + i * kw + j
                    # fp32 coordinates, as the oracle forms them
                    py = (hh * sh + float(i * dh - ph)) + off[:, 2 * k]
                    px = (ww * sw + float(j * dw - pw)) + off[:, 2 * k + 1]
                    grid = torch.stack([px.double() * (2.0 / (W - 1)) - 1.0,
                                        py.double() * (2.0 / (H - 1)) - 1.0], dim=-1)
                    samp = F.grid_sample(x[:, cs].double(), grid, mode="bilinear",
                                         padding_mode="zeros", align_corners=True)
                    Wd = _dense_tap_weight(w, s["groups"], C, i, j)
                    ref += torch.einsum("oc,bchw->bohw", Wd[:, cs], samp) * m[:, k:k + 1].double()
        got = orc.forward_ex(x, off, m, w, b, _conv_desc(s))
        err = _rel_err(got, ref.numpy())
        assert err <= 1e-10, f"general grid_sample {s}: {err:.3e}"


def pin_offset_groups_collapse(orc):
    """Offset groups that all carry the same offsets and mask give exactly
    the one-group result."""
    for n, s in enumerate(GEN_SHAPES):
        if s["offset_groups"] == 1:
            continue
        x, off, m, w, b = _rand_problem_ex(140 + n, s, off_std=2.0)
        G, k_all = s["offset_groups"], s["kh"] * s["kw"]
        off1, m1 = off[:, :2 * k_all].clone(), m[:, :k_all].clone()
        offG, mG = off1.repeat(1, G, 1, 1), m1.repeat(1, G, 1, 1)
        s1 = dict(s, offset_groups=1)
        got = orc.forward_ex(x, offG, mG, w, b, _conv_desc(s))
        one = orc.forward_ex(x, off1, m1, w, b, _conv_desc(s1))
        assert np.array_equal(got, one), f"offset groups collapse {s}"


ALL_PINS = [pin_direct_conv, pin_shifted_conv, pin_integer_gather, pin_bilinear_golden,
            pin_grid_sample, pin_outside_is_bias, pin_mask, pin_affine_map,
            pin_general_direct_conv, pin_general_shifted_conv, pin_general_grid_sample,
            pin_offset_groups_collapse]
