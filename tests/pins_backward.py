"""Pins of the oracle's backward pass: checks of its gradients against what
the mathematics fixes, independently of the oracle's own code.

- autograd: the forward written with a library bilinear resampler
  (torch.nn.functional.grid_sample, zero padding, align_corners=True, fp64)
  and an einsum, differentiated by torch's autograd, gives every gradient;
- adjoints: the forward is linear in x, in the weight and in the mask, so
  <grad_out, F - bias> = <grad, input> for each of them, with F the
  (separately pinned) forward oracle;
- finite differences: inside one bilinear cell the forward is linear in
  each offset, so a central difference of the forward oracle is exact
  there (offsets on a 2^-12 grid, steps of 2^-10, coordinates at least
  2^-8 from a cell border);
- zero offsets with mask 1: the gradients of a plain convolution
  (torch.nn.grad.conv2d_input / conv2d_weight, with stride, padding,
  dilation and groups);
- samples with every corner outside the image: all gradients 0 but the
  bias's, which is the sum of grad_out.
"""

import numpy as np
import torch
import torch.nn.functional as F

from tests.pins import GEN_SHAPES, SHAPES, _conv_desc, _pair, _rel_err


def _general(s):
    if "stride" in s:
        return dict(s)
    return dict(B=s["B"], C=s["C"], H=s["H"], W=s["W"], O=s["O"], kh=s["kh"], kw=s["kw"],
                stride=1, padding=s["pad"], dilation=1, groups=1, offset_groups=1)


CASES = [_general(s) for s in SHAPES if s["H"] > 1 and s["W"] > 1] + list(GEN_SHAPES)


def _problem(seed, s, off_std=2.5, mask=True):
    g = torch.Generator().manual_seed(seed)
    B, C, H, W, O, kh, kw = (s[k] for k in ("B", "C", "H", "W", "O", "kh", "kw"))
    Ho, Wo = _conv_desc(s).out_size(H, W, kh, kw)
    k, G = kh * kw, s["offset_groups"]
    x = torch.randn(B, C, H, W, generator=g)
    off = torch.randn(B, 2 * G * k, Ho, Wo, generator=g) * off_std
    m = torch.rand(B, G * k, Ho, Wo, generator=g) * 2 if mask else None
    w = torch.randn(O, C // s["groups"], kh, kw, generator=g) * 0.3
    gout = torch.randn(B, O, Ho, Wo, generator=g)
    return x, off, m, w, gout


def _autograd_reference(x, off, m, w, gout, s):
    """Gradients of sum(gout * F) by autograd through grid_sample."""
    B, C, H, W = x.shape
    O, Cg, kh, kw = w.shape
    G, groups = s["offset_groups"], s["groups"]
    k_all, Cq, Og = kh * kw, C // G, O // groups
    sh, sw = _pair(s["stride"])
    ph, pw = _pair(s["padding"])
    dh, dw = _pair(s["dilation"])
    Ho, Wo = off.shape[2], off.shape[3]
    xd = x.double().requires_grad_()
    od = off.double().requires_grad_()
    md = None if m is None else m.double().requires_grad_()
    wd = w.double().requires_grad_()
    bd = torch.zeros(O, dtype=torch.float64, requires_grad=True)
    hh = torch.arange(Ho, dtype=torch.float32).view(1, Ho, 1)
    ww = torch.arange(Wo, dtype=torch.float32).view(1, 1, Wo)
    out = bd.view(1, -1, 1, 1).expand(B, -1, Ho, Wo)
    for q in range(G):
        for i in range(kh):
            for j in range(kw):
                k = q * k_all + i * kw + j
                # the oracle's fp32 coordinate as the value, d/d offset = 1
                py32 = (hh * sh + float(i * dh - ph)) + off[:, 2 * k]
                px32 = (ww * sw + float(j * dw - pw)) + off[:, 2 * k + 1]
                py = py32.double() + (od[:, 2 * k] - od[:, 2 * k].detach())
                px = px32.double() + (od[:, 2 * k + 1] - od[:, 2 * k + 1].detach())
                grid = torch.stack([px * (2.0 / (W - 1)) - 1.0, py * (2.0 / (H - 1)) - 1.0], dim=-1)
                for c0 in range(q * Cq, (q + 1) * Cq):
                    gidx = c0 // Cg
                    samp = F.grid_sample(xd[:, c0:c0 + 1], grid, mode="bilinear",
                                         padding_mode="zeros", align_corners=True)[:, 0]
                    if md is not None:
                        samp = samp * md[:, k]
                    wt = wd[gidx * Og:(gidx + 1) * Og, c0 - gidx * Cg, i, j]
                    contrib = wt.view(1, Og, 1, 1) * samp.unsqueeze(1)
                    pad = (0, 0, 0, 0, gidx * Og, O - (gidx + 1) * Og)
                    out = out + F.pad(contrib, pad)
    (out * gout.double()).sum().backward()
    return {"grad_x": xd.grad.numpy(), "grad_offset": od.grad.numpy(),
            "grad_mask": None if md is None else md.grad.numpy(),
            "grad_weight": wd.grad.numpy(), "grad_bias": bd.grad.numpy()}


def pin_bwd_autograd(orc):
    """Every gradient equals autograd through the library resampler."""
    for n, s in enumerate(CASES):
        for mask in (True, False):
            x, off, m, w, gout = _problem(200 + n, s, mask=mask)
            ref = _autograd_reference(x, off, m, w, gout, s)
            got = orc.backward_ex(x, off, m, w, gout, _conv_desc(s))
            for key in ref:
                if ref[key] is None:
                    assert got[key] is None
                    continue
                err = _rel_err(got[key], ref[key])
                assert err <= 1e-10, f"autograd {key} {s} mask={mask}: rel err {err:.3e}"


def pin_bwd_adjoint(orc):
    """Linearity in x, weight and mask: <grad_out, F - bias> = <grad, input>."""
    for n, s in enumerate(CASES):
        x, off, m, w, gout = _problem(260 + n, s)
        conv = _conv_desc(s)
        g = orc.backward_ex(x, off, m, w, gout, conv)
        f = orc.forward_ex(x, off, m, w, None, conv)
        lhs = float((gout.double().numpy() * f).sum())
        scale = float(np.abs(gout.double().numpy()).sum() * np.abs(f).max()) + 1e-300
        for key, inp in (("grad_x", x), ("grad_weight", w), ("grad_mask", m)):
            rhs = float((g[key] * inp.double().numpy()).sum())
            assert abs(lhs - rhs) <= 1e-12 * scale, f"adjoint {key} {s}: {lhs} vs {rhs}"
        assert np.allclose(g["grad_bias"], gout.double().sum(dim=(0, 2, 3)).numpy(),
                           rtol=0, atol=1e-12 * float(np.abs(gout.numpy()).sum()))


def _quantised_offsets(off, H, W, s):
    """Offsets on a 2^-12 grid whose sampling coordinates lie at least 2^-8
    from every cell border (so +-2^-10 stays inside the cell)."""
    q = torch.round(off * 4096.0) / 4096.0
    frac = q - torch.floor(q)
    # move fractions out of [0, 2^-8) and (1 - 2^-8, 1)
    q = torch.where(frac < 2 ** -8, q + 2 ** -7, q)
    q = torch.where(frac > 1 - 2 ** -8, q - 2 ** -7, q)
    return q


def pin_bwd_finite_diff_offsets(orc):
    """Central differences of the forward in single offsets (exact inside a
    bilinear cell) equal grad_offset."""
    eps = 2.0 ** -10
    for n, s in enumerate(CASES[:6]):
        x, off, m, w, gout = _problem(300 + n, s, off_std=1.5)
        off = _quantised_offsets(off, s["H"], s["W"], s)
        conv = _conv_desc(s)
        g = orc.backward_ex(x, off, m, w, gout, conv)["grad_offset"]
        rng = np.random.default_rng(300 + n)
        B, CH, Ho, Wo = off.shape
        scale = max(float(np.abs(g).max()), 1e-300)
        for _ in range(6):
            b, ch, h, ww = (int(rng.integers(0, v)) for v in (B, CH, Ho, Wo))
            plus, minus = off.clone(), off.clone()
            plus[b, ch, h, ww] += eps
            minus[b, ch, h, ww] -= eps
            pts = np.array([[b, h, ww]], dtype=np.int32)
            fp = orc.forward_points_ex(x, plus, m, w, None, conv, pts)[0]
            fm = orc.forward_points_ex(x, minus, m, w, None, conv, pts)[0]
            fd = float((gout[b, :, h, ww].double().numpy() * (fp - fm)).sum() / (2 * eps))
            assert abs(fd - g[b, ch, h, ww]) <= 1e-9 * scale, \
                f"finite difference {s} at {(b, ch, h, ww)}: {fd} vs {g[b, ch, h, ww]}"


def pin_bwd_direct_conv(orc):
    """Zero offsets, mask 1: the gradients of a plain convolution."""
    for n, s in enumerate(CASES):
        x, off, m, w, gout = _problem(340 + n, s)
        off = torch.zeros_like(off)
        conv = _conv_desc(s)
        kw_ = dict(stride=_pair(s["stride"]), padding=_pair(s["padding"]),
                   dilation=_pair(s["dilation"]), groups=s["groups"])
        for mask in (None, torch.ones_like(m)):
            g = orc.backward_ex(x, off, mask, w, gout, conv)
            gx = torch.nn.grad.conv2d_input(x.shape, w.double(), gout.double(), **kw_)
            gw = torch.nn.grad.conv2d_weight(x.double(), w.shape, gout.double(), **kw_)
            assert _rel_err(g["grad_x"], gx.numpy()) <= 1e-12, f"direct conv grad_x {s}"
            assert _rel_err(g["grad_weight"], gw.numpy()) <= 1e-12, f"direct conv grad_weight {s}"


def pin_bwd_outside(orc):
    """Every corner outside the image: no gradient but the bias's."""
    for n, s in enumerate(CASES[:5]):
        x, off, m, w, gout = _problem(380 + n, s)
        off = off.clone()
        off[:, 0::2] = -(s["H"] + 5.0)
        g = orc.backward_ex(x, off, m, w, gout, _conv_desc(s))
        for key in ("grad_x", "grad_offset", "grad_mask", "grad_weight"):
            assert not np.any(g[key]), f"outside {key} {s}"
        assert np.allclose(g["grad_bias"], gout.double().sum(dim=(0, 2, 3)).numpy(), rtol=1e-13)


ALL_BACKWARD_PINS = [pin_bwd_autograd, pin_bwd_adjoint, pin_bwd_finite_diff_offsets,
                     pin_bwd_direct_conv, pin_bwd_outside]


def check_points_match_full(orc):
    """The per-pixel variant returns the full backward's offset and mask
    gradients at the chosen pixels (the same body; a consistency check)."""
    s = CASES[-2]
    x, off, m, w, gout = _problem(420, s)
    conv = _conv_desc(s)
    full = orc.backward_ex(x, off, m, w, gout, conv)
    B, _, Ho, Wo = off.shape
    pts = np.array([[b, h, ww] for b in range(B) for h in range(0, Ho, 2) for ww in range(0, Wo, 3)],
                   dtype=np.int32)
    goff, gm = orc.backward_points_ex(x, off, m, w, gout, conv, pts)
    for t, (b, h, ww) in enumerate(pts):
        assert np.array_equal(goff[t], full["grad_offset"][b, :, h, ww])
        assert np.array_equal(gm[t], full["grad_mask"][b, :, h, ww])
