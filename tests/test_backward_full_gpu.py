"""Backward pass at the benchmark's full size (the 7x7, C = O = 64,
256 x 256 ASPP workload), in the launch configuration bench.py times.

What the oracle can check there: the offset and mask gradients of sampled
output pixels (they depend on that pixel alone) element by element; the x,
weight and mask gradients through their adjoint identities (the forward
without bias, F, is linear in each of them, so <grad_x, x> =
<grad_weight, weight> = <grad_mask, mask> = sum(grad_out * F), one full
oracle forward); the bias gradient as the sum of grad_out.  Bar: the fp32 one, 1e-4, relative to the compared magnitudes.
"""

import numpy as np
import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300.inputs import WORKLOADS, make_inputs
from tests.helpers import sample_points, to_device

pytestmark = pytest.mark.gpu

BAR = 1e-4


@pytest.fixture(scope="module")
def problem():
    wl = WORKLOADS["aspp7x7"]
    inp = make_inputs(wl)
    g = torch.Generator().manual_seed(1234)
    gout = torch.randn(wl.B, wl.O, wl.Ho, wl.Wo, generator=g).to(inp["x"].dtype)
    d = to_device(inp)
    f32 = dict(dtype=torch.float32, device="cuda")
    gx = torch.empty(d["x"].shape, memory_format=torch.channels_last, **f32)
    goff = torch.empty(d["offset"].shape, **f32)
    gm = torch.empty(d["mask"].shape, **f32)
    gw = torch.empty(d["weight"].shape, **f32)
    gb = torch.empty((wl.O,), **f32)
    gd = gout.cuda().contiguous(memory_format=torch.channels_last)
    with dcn.Handle() as h:
        dcn.dcn_backward(h.h, d["x"], d["offset"], d["mask"], d["weight"], gd, gx, goff, gm, gw, gb,
                         wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, dcn.DCN_BF16)
        assert dcn.dcn_sync_status(h.h) == 0
    got = {"grad_x": gx.cpu(), "grad_offset": goff.cpu(), "grad_mask": gm.cpu(),
           "grad_weight": gw.cpu(), "grad_bias": gb.cpu()}
    return wl, inp, gout, got


def test_offset_and_mask_gradients_at_sampled_pixels(problem):
    wl, inp, gout, got = problem
    pts = sample_points(wl.B, wl.Ho, wl.Wo, 160, seed=5)
    goff, gm = oracle.backward_points_ex(inp["x"], inp["offset"], inp["mask"], inp["weight"], gout,
                                         oracle.ConvDesc(padding=wl.pad), pts)
    b, h, w = pts[:, 0], pts[:, 1], pts[:, 2]
    g_off = got["grad_offset"][b, :, h, w].numpy()
    g_m = got["grad_mask"][b, :, h, w].numpy()
    assert np.abs(g_off - goff).max() <= BAR * np.abs(goff).max()
    assert np.abs(g_m - gm).max() <= BAR * np.abs(gm).max()


def test_x_weight_mask_gradients_by_adjoint(problem):
    """F - bias is linear in x, in the weight and in the mask separately, so
    <grad_x, x> = <grad_weight, weight> = <grad_mask, mask> =
    sum(grad_out * (F - bias)); one oracle forward checks all three."""
    wl, inp, gout, got = problem
    go = gout.double().numpy()
    F = oracle.forward(inp["x"], inp["offset"], inp["mask"], inp["weight"], None, wl.pad)
    lhs, scale = float((go * F).sum()), float(np.abs(go * F).sum())
    for key, v in (("grad_x", inp["x"]), ("grad_weight", inp["weight"]), ("grad_mask", inp["mask"])):
        rhs = float((got[key].double() * v.double()).sum())
        assert abs(lhs - rhs) <= BAR * scale, f"{key} adjoint: {lhs} vs {rhs}"


def test_bias_gradient_is_the_sum(problem):
    wl, inp, gout, got = problem
    exp = gout.double().sum(dim=(0, 2, 3)).numpy()
    assert np.abs(got["grad_bias"].double().numpy() - exp).max() <= BAR * np.abs(exp).max()
