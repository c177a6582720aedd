"""Pins of the single-scale deformable sampling backward oracle: checks
against what the mathematics and a library routine fix, independently of
the oracle's own code.

- fp64 autograd through the library bilinear resampler (torch grid_sample)
  and torch's softmax, for the value, offset and weight gradients
  (coordinates at the oracle's fp32 values, moved off cell borders);
- adjoint identities: the output is linear in the value map (and, without
  softmax, in the weights), so <grad_out, out> = <grad_value, value> =
  <grad_weights, weights>, with `out` from the separately pinned forward;
- exact central differences of the forward in single offsets (offsets on a
  2^-10 grid, so that the fp32 coordinates are exact, at least 2^-6 pixel
  from a cell border, where the forward is exactly linear);
- with softmax the weight gradients of each (b, ho, wo, g) sum to zero;
- a constant map sampled with every corner inside: zero offset gradients;
- every corner outside: every gradient exactly zero.
"""

import numpy as np
import torch
import torch.nn.functional as F

from tests.pins_attn import CASES, _problem, _rel


def _grad_out(seed, shape):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g)


def _away_from_borders(off, Ho, Wo, kernel, stride, padding, dilation):
    """Move offsets whose fp32 coordinate lies within 1e-4 of an integer by a
    quarter pixel, so that floor() takes the same cell in fp32 and fp64."""
    off = off.clone()
    kh, kw = kernel
    hs = (torch.arange(Ho) * stride[0] - padding[0]).view(1, Ho, 1, 1)
    ws = (torch.arange(Wo) * stride[1] - padding[1]).view(1, 1, Wo, 1)
    for k in range(kh * kw):
        i, j = k // kw, k % kw
        for axis, base in ((0, hs + i * dilation[0]), (1, ws + j * dilation[1])):
            c = off[:, :, :, :, k, axis]
            p = base.float() + c
            near = (p - torch.round(p)).abs() < 1e-4
            c[near] += 0.25
    return off


def _torch_backward(value, off, w, go, kernel, stride, padding, dilation, softmax):
    B, H, W, G, D = value.shape
    _, Ho, Wo, _, K, _ = off.shape
    kh, kw = kernel
    v = value.double().requires_grad_(True)
    wd = w.double().requires_grad_(True)
    od = off.double().requires_grad_(True)
    a = torch.softmax(wd, dim=-1) if softmax else wd
    out = torch.zeros(B, Ho, Wo, G, D, dtype=torch.float64)
    hs = torch.arange(Ho).view(Ho, 1) * stride[0] - padding[0]
    ws = torch.arange(Wo).view(1, Wo) * stride[1] - padding[1]
    for g in range(G):
        inp = v[:, :, :, g, :].permute(0, 3, 1, 2)
        for k in range(K):
            i, j = k // kw, k % kw
            by, bx = hs + i * dilation[0], ws + j * dilation[1]
            py32 = (by.float() + off[:, :, :, g, k, 0]).double()
            px32 = (bx.float() + off[:, :, :, g, k, 1]).double()
            py = by.double() + od[:, :, :, g, k, 0]
            px = bx.double() + od[:, :, :, g, k, 1]
            py = py + (py32 - py).detach()
            px = px + (px32 - px).detach()
            grid = torch.stack([(2.0 * px + 1.0) / W - 1.0, (2.0 * py + 1.0) / H - 1.0], dim=-1)
            samp = F.grid_sample(inp, grid, mode="bilinear", padding_mode="zeros",
                                 align_corners=False)
            out[:, :, :, g, :] = out[:, :, :, g, :] + samp.permute(0, 2, 3, 1) * a[:, :, :, g, k].unsqueeze(-1)
    (out * go.double()).sum().backward()
    return v.grad.numpy(), od.grad.numpy(), wd.grad.numpy()


def pin_attn_bwd_autograd(orc):
    for n, (B, H, W, G, D, kernel, stride, padding, dilation) in enumerate(CASES):
        value, off, w, Ho, Wo = _problem(800 + n, B, H, W, G, D, kernel, stride, padding, dilation)
        off = _away_from_borders(off, Ho, Wo, kernel, stride, padding, dilation)
        go = _grad_out(810 + n, (B, Ho, Wo, G, D))
        for softmax in (False, True):
            gv, go_, gw = orc.attn_backward(value, off, w, go, kernel, stride, padding, dilation,
                                            softmax)
            rv, ro, rw = _torch_backward(value, off, w, go, kernel, stride, padding, dilation,
                                         softmax)
            for name, got, ref in (("value", gv, rv), ("offsets", go_, ro), ("weights", gw, rw)):
                err = _rel(got, ref)
                assert err <= 1e-9, f"attn backward {name} case {n} softmax={softmax}: {err:.3e}"


def pin_attn_bwd_adjoint(orc):
    for n, (B, H, W, G, D, kernel, stride, padding, dilation) in enumerate(CASES):
        value, off, w, Ho, Wo = _problem(820 + n, B, H, W, G, D, kernel, stride, padding, dilation)
        go = _grad_out(830 + n, (B, Ho, Wo, G, D))
        god = go.double().numpy()
        for softmax in (False, True):
            out = orc.attn_forward(value, off, w, kernel, stride, padding, dilation, softmax)
            gv, _, gw = orc.attn_backward(value, off, w, go, kernel, stride, padding, dilation,
                                          softmax)
            lhs = float((god * out).sum())
            assert abs(lhs - float((gv * value.double().numpy()).sum())) <= 1e-11 * max(1.0, abs(lhs))
            if not softmax:
                assert abs(lhs - float((gw * w.double().numpy()).sum())) <= 1e-11 * max(1.0, abs(lhs))


def pin_attn_bwd_finite_differences(orc):
    B, H, W, G, D, kernel, stride, padding, dilation = CASES[1]
    value, off, w, Ho, Wo = _problem(840, B, H, W, G, D, kernel, stride, padding, dilation)
    go = _grad_out(841, (B, Ho, Wo, G, D))
    god = go.double().numpy()
    rng = np.random.default_rng(842)
    h = 2.0 ** -10
    # offsets on the 2^-10 grid whose fractional part is at least 2^-6 from a border
    m = np.round(off.numpy() / h)
    frac = np.mod(m * h, 1.0)
    m[(frac < 2.0 ** -6) | (frac > 1.0 - 2.0 ** -6)] += 32
    off = torch.from_numpy(m * h).float()
    K = kernel[0] * kernel[1]
    for softmax in (False, True):
        _, go_, _ = orc.attn_backward(value, off, w, go, kernel, stride, padding, dilation, softmax)
        for _ in range(10):
            idx = tuple(int(rng.integers(0, n)) for n in (B, Ho, Wo, G, K, 2))
            op, om = off.clone(), off.clone()
            op[idx] += h
            om[idx] -= h
            fp = float((god * orc.attn_forward(value, op, w, kernel, stride, padding, dilation, softmax)).sum())
            fm = float((god * orc.attn_forward(value, om, w, kernel, stride, padding, dilation, softmax)).sum())
            fd = (fp - fm) / (2.0 * h)
            got = go_[idx]
            assert abs(fd - got) <= 1e-8 * max(1.0, abs(got)), f"offset gradient {idx}: {got} vs {fd}"


def pin_attn_bwd_softmax_sums_to_zero(orc):
    B, H, W, G, D, kernel, stride, padding, dilation = CASES[0]
    value, off, w, Ho, Wo = _problem(850, B, H, W, G, D, kernel, stride, padding, dilation)
    go = _grad_out(851, (B, Ho, Wo, G, D))
    _, _, gw = orc.attn_backward(value, off, w, go, kernel, stride, padding, dilation, True)
    _, _, raw = orc.attn_backward(value, off, w, go, kernel, stride, padding, dilation, False)
    assert np.abs(gw).max() > 0
    assert np.abs(gw.sum(axis=-1)).max() <= 1e-13 * np.abs(raw).max() * gw.shape[-1]


def pin_attn_bwd_constant_map(orc):
    B, H, W, G, D, kernel, stride, padding, dilation = (1, 12, 14, 3, 4, (3, 3), (1, 1), (1, 1), (1, 1))
    value, off, w, Ho, Wo = _problem(860, B, H, W, G, D, kernel, stride, padding, dilation)
    const = torch.randn(G, D)
    value = const.view(1, 1, 1, G, D).expand_as(value).contiguous()
    # every corner strictly inside: positions in [0.5, H-1.5] x [0.5, W-1.5]
    kh, kw = kernel
    for k in range(kh * kw):
        i, j = k // kw, k % kw
        by = (torch.arange(Ho) - padding[0] + i).view(1, Ho, 1, 1).float()
        bx = (torch.arange(Wo) - padding[1] + j).view(1, 1, Wo, 1).float()
        r = torch.rand(B, Ho, Wo, G, 2) - 0.5
        off[..., k, 0] = (by + r[..., 0]).clamp(0.5, H - 1.5) - by
        off[..., k, 1] = (bx + r[..., 1]).clamp(0.5, W - 1.5) - bx
    go = _grad_out(861, (B, Ho, Wo, G, D))
    for softmax in (False, True):
        _, go_, gw = orc.attn_backward(value, off, w, go, kernel, stride, padding, dilation, softmax)
        assert np.abs(go_).max() <= 1e-12 * max(1.0, np.abs(gw).max())


def pin_attn_bwd_outside(orc):
    B, H, W, G, D, kernel, stride, padding, dilation = CASES[0]
    value, off, w, Ho, Wo = _problem(870, B, H, W, G, D, kernel, stride, padding, dilation)
    off[..., 1] = torch.where(torch.rand(off[..., 1].shape) < 0.5, -float(W + 3), float(2 * W + 3))
    go = _grad_out(871, (B, Ho, Wo, G, D))
    for softmax in (False, True):
        gv, go_, gw = orc.attn_backward(value, off, w, go, kernel, stride, padding, dilation, softmax)
        assert not np.any(gv) and not np.any(go_) and not np.any(gw)


ALL_ATTN_BACKWARD_PINS = [pin_attn_bwd_autograd, pin_attn_bwd_adjoint,
                          pin_attn_bwd_finite_differences, pin_attn_bwd_softmax_sums_to_zero,
                          pin_attn_bwd_constant_map, pin_attn_bwd_outside]
