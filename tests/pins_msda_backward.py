"""Pins of the MSDA backward oracle: checks against what the mathematics
and a library routine fix, independently of the oracle's own code.

- autograd through the library bilinear resampler (torch grid_sample, zero
  padding, align_corners=False, fp64) and torch's softmax, for the value,
  location and weight gradients;
- adjoint identities: the output is linear in the value map (and, without
  softmax, in the weights), so <grad_out, out> = <grad_value, value> =
  <grad_weights, weights>, with `out` from the separately pinned forward;
- exact central differences of the forward in single locations (locations
  on a 2^-12 grid, so that the fp32 pixel coordinates are exact, at least
  2^-6 pixel from a cell border, where the forward is exactly linear);
- with softmax the weight gradients of each (b, q, g) sum to zero (the
  normalization is invariant to a common shift of the logits);
- a constant value map sampled with every corner inside: zero location
  gradients;
- every corner outside: every gradient exactly zero.
"""

import numpy as np
import torch
import torch.nn.functional as F

from tests.pins_msda import LEVELS, _problem, _rel


def _away_from_borders(loc, shapes):
    """Move fp32 pixel coordinates that lie within 1e-4 of an integer by a
    quarter pixel, so that floor() takes the same cell in fp32 and fp64."""
    loc = loc.clone()
    for l, (H, W) in enumerate(shapes):
        for axis, n in ((0, W), (1, H)):
            c = loc[:, :, :, l, :, axis]
            p = c * float(n) - 0.5
            near = (p - torch.round(p)).abs() < 1e-4
            c[near] += 0.25 / n
    return loc


def _torch_backward(value, shapes, starts, loc, w, go, softmax):
    """fp64 autograd through grid_sample; the pixel coordinates take the
    oracle's fp32 values (a detached correction) with derivative W_l, H_l."""
    B, S, G, D = value.shape
    _, Q, _, L, K, _ = loc.shape
    v = value.double().requires_grad_(True)
    wd = w.double().requires_grad_(True)
    ld = loc.double().requires_grad_(True)
    a = torch.softmax(wd, dim=-1) if softmax else wd
    out = torch.zeros(B, Q, G, D, dtype=torch.float64)
    for l, (H, W) in enumerate(shapes):
        lvl = v[:, starts[l]:starts[l] + H * W].reshape(B, H, W, G, D)
        for g in range(G):
            inp = lvl[:, :, :, g, :].permute(0, 3, 1, 2)
            px32 = (loc[:, :, g, l, :, 0] * float(W) - 0.5).double()
            py32 = (loc[:, :, g, l, :, 1] * float(H) - 0.5).double()
            px = ld[:, :, g, l, :, 0] * W - 0.5
            py = ld[:, :, g, l, :, 1] * H - 0.5
            px = px + (px32 - px).detach()
            py = py + (py32 - py).detach()
            grid = torch.stack([(2.0 * px + 1.0) / W - 1.0, (2.0 * py + 1.0) / H - 1.0], dim=-1)
            samp = F.grid_sample(inp, grid, mode="bilinear", padding_mode="zeros",
                                 align_corners=False)
            aw = a[:, :, g, l * K:(l + 1) * K]
            out[:, :, g, :] = out[:, :, g, :] + torch.einsum("bdqk,bqk->bqd", samp, aw)
    (out * go.double()).sum().backward()
    return v.grad.numpy(), ld.grad.numpy(), wd.grad.numpy()


def _grad_out(seed, B, Q, G, D):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, Q, G, D, generator=g)


def pin_msda_bwd_autograd(orc):
    for n, (shapes, K, G) in enumerate(LEVELS):
        for softmax in (False, True):
            value, starts, loc, w = _problem(600 + n, shapes, K, G)
            loc = _away_from_borders(loc, shapes)
            go = _grad_out(610 + n, value.shape[0], loc.shape[1], G, value.shape[3])
            gv, gl, gw = orc.msda_backward(value, shapes, starts, loc, w, go, softmax)
            rv, rl, rw = _torch_backward(value, shapes, starts, loc, w, go, softmax)
            for name, got, ref in (("value", gv, rv), ("locations", gl, rl), ("weights", gw, rw)):
                err = _rel(got, ref)
                assert err <= 1e-9, f"msda backward {name} {shapes} softmax={softmax}: {err:.3e}"


def pin_msda_bwd_adjoint(orc):
    for n, (shapes, K, G) in enumerate(LEVELS):
        value, starts, loc, w = _problem(620 + n, shapes, K, G)
        go = _grad_out(630 + n, value.shape[0], loc.shape[1], G, value.shape[3])
        god = go.double().numpy()
        for softmax in (False, True):
            out = orc.msda_forward(value, shapes, starts, loc, w, softmax)
            gv, _, gw = orc.msda_backward(value, shapes, starts, loc, w, go, softmax)
            lhs = float((god * out).sum())
            rv = float((gv * value.double().numpy()).sum())
            assert abs(lhs - rv) <= 1e-11 * max(1.0, abs(lhs)), f"value adjoint {shapes}"
            if not softmax:
                rw = float((gw * w.double().numpy()).sum())
                assert abs(lhs - rw) <= 1e-11 * max(1.0, abs(lhs)), f"weight adjoint {shapes}"


def pin_msda_bwd_finite_differences(orc):
    shapes, K, G = [[8, 16], [4, 8], [2, 4]], 3, 2
    value, starts, loc, w = _problem(640, shapes, K, G)
    B, Q = loc.shape[0], loc.shape[1]
    go = _grad_out(641, B, Q, G, value.shape[3])
    god = go.double().numpy()
    rng = np.random.default_rng(642)
    h = 2.0 ** -12
    # locations on the 2^-12 grid, pixel coordinates at least 2^-6 from a border
    for l, (H, W) in enumerate(shapes):
        for axis, size in ((0, W), (1, H)):
            m = rng.integers(0, 4096, size=loc[:, :, :, l, :, axis].shape)
            frac = np.mod(m * size / 4096.0 - 0.5, 1.0)
            bad = (frac < 2.0 ** -6) | (frac > 1.0 - 2.0 ** -6)
            m[bad] += 8
            loc[:, :, :, l, :, axis] = torch.from_numpy(m * h).float()
    for softmax in (False, True):
        _, gl, _ = orc.msda_backward(value, shapes, starts, loc, w, go, softmax)
        for _ in range(10):
            b, q, g, l, k, ax = (int(rng.integers(0, n)) for n in (B, Q, G, len(shapes), K, 2))
            lp, lm = loc.clone(), loc.clone()
            lp[b, q, g, l, k, ax] += h
            lm[b, q, g, l, k, ax] -= h
            fp = float((god * orc.msda_forward(value, shapes, starts, lp, w, softmax)).sum())
            fm = float((god * orc.msda_forward(value, shapes, starts, lm, w, softmax)).sum())
            fd = (fp - fm) / (2.0 * h)
            got = gl[b, q, g, l, k, ax]
            assert abs(fd - got) <= 1e-8 * max(1.0, abs(got)), \
                f"location gradient {(b, q, g, l, k, ax)}: {got} vs difference {fd}"


def pin_msda_bwd_softmax_sums_to_zero(orc):
    shapes, K, G = [[16, 12], [8, 6], [4, 3]], 4, 2
    value, starts, loc, w = _problem(650, shapes, K, G)
    go = _grad_out(651, value.shape[0], loc.shape[1], G, value.shape[3])
    _, _, gw = orc.msda_backward(value, shapes, starts, loc, w, go, True)
    _, _, raw = orc.msda_backward(value, shapes, starts, loc, w, go, False)
    assert np.abs(gw).max() > 0
    assert np.abs(gw.sum(axis=-1)).max() <= 1e-13 * np.abs(raw).max() * gw.shape[-1]


def pin_msda_bwd_constant_map(orc):
    shapes, K, G = [[16, 12], [8, 6], [4, 4]], 4, 2
    value, starts, loc, w = _problem(660, shapes, K, G)
    const = torch.randn(G, value.shape[3])
    value = const.view(1, 1, G, -1).expand_as(value).contiguous()
    for l, (H, W) in enumerate(shapes):
        loc[:, :, :, l, :, 0] = (1.0 + torch.rand(loc[:, :, :, l, :, 0].shape) * (W - 2)) / W
        loc[:, :, :, l, :, 1] = (1.0 + torch.rand(loc[:, :, :, l, :, 1].shape) * (H - 2)) / H
    go = _grad_out(661, value.shape[0], loc.shape[1], G, value.shape[3])
    for softmax in (False, True):
        _, gl, gw = orc.msda_backward(value, shapes, starts, loc, w, go, softmax)
        assert np.abs(gl).max() <= 1e-12 * max(1.0, np.abs(gw).max())


def pin_msda_bwd_outside(orc):
    shapes, K, G = [[6, 10], [3, 5]], 4, 2
    value, starts, loc, w = _problem(670, shapes, K, G)
    loc[..., 0] = torch.where(torch.rand(loc[..., 0].shape) < 0.5, -0.6, 1.7)
    go = _grad_out(671, value.shape[0], loc.shape[1], G, value.shape[3])
    for softmax in (False, True):
        gv, gl, gw = orc.msda_backward(value, shapes, starts, loc, w, go, softmax)
        assert not np.any(gv) and not np.any(gl) and not np.any(gw)


ALL_MSDA_BACKWARD_PINS = [pin_msda_bwd_autograd, pin_msda_bwd_adjoint,
                          pin_msda_bwd_finite_differences, pin_msda_bwd_softmax_sums_to_zero,
                          pin_msda_bwd_constant_map, pin_msda_bwd_outside]
