"""Single-scale deformable sampling on the GPU against its oracle.

Whole outputs are compared (the oracle handles every case here in
seconds), with the operand dtype's bar from tests.helpers.TOL: the kernel
computes in fp32 and rounds once to the output dtype.
"""

import numpy as np
import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300.inputs import (ATTN_WORKLOADS, AttnWorkload,
                                                        make_attn_inputs)
from tests.helpers import TOL

pytestmark = pytest.mark.gpu


def check(wl, inp=None):
    inp = make_attn_inputs(wl) if inp is None else inp
    method = "softmax" if wl.softmax else None
    out = dcn.attn(inp["value"].cuda(), inp["offsets"].cuda(), inp["weights"].cuda(), wl.kernel,
                   wl.stride, wl.padding, wl.dilation, method=method)
    torch.cuda.synchronize()
    ref = oracle.attn_forward(inp["value"], inp["offsets"], inp["weights"], wl.kernel, wl.stride,
                              wl.padding, wl.dilation, wl.softmax)
    got = out.float().cpu().numpy()
    assert got.shape == ref.shape
    assert np.isfinite(got).all()
    err = float(np.abs(got - ref).max() / np.abs(ref).max())
    assert err <= TOL[wl.dtype], f"{wl.name}: rel err {err:.3e}"
    return out


@pytest.mark.parametrize("name", sorted(ATTN_WORKLOADS))
def test_attn_workloads(name):
    check(ATTN_WORKLOADS[name])


A = AttnWorkload
CASES = [
    A("attn_f32", 2, 13, 11, 3, 4, dtype="f32", seed=100),
    A("attn_f16", 1, 17, 19, 4, 16, dtype="f16", seed=101),
    A("attn_no_softmax", 1, 12, 15, 2, 32, softmax=False, seed=102),
    A("attn_stride2_dil2", 2, 21, 18, 4, 8, kernel=(3, 3), stride=(2, 2), padding=(2, 2),
      dilation=(2, 2), seed=103),
    A("attn_rect_5x3", 1, 16, 20, 2, 16, kernel=(5, 3), stride=(1, 2), padding=(2, 1), seed=104),
    A("attn_1x1", 1, 9, 10, 5, 8, kernel=(1, 1), padding=(0, 0), seed=105),
    # D not a multiple of 8 (16-bit) / 4 (fp32): one channel per lane
    A("attn_d_odd", 2, 8, 9, 3, 5, seed=106),
    A("attn_d_odd_f32", 1, 7, 6, 2, 3, dtype="f32", softmax=False, seed=107),
    # D = 256: 32 lanes per (pixel, group); D = 24: three chunks over two lanes
    A("attn_d256", 1, 6, 7, 2, 256, seed=108),
    A("attn_d24", 1, 9, 8, 3, 24, dtype="f16", seed=109),
    # offsets large enough that many samples leave the map
    A("attn_far", 1, 10, 12, 4, 16, offset_std=12.0, seed=110),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_attn_cases(wl):
    check(wl)


def test_attn_nonfinite_offsets():
    wl = A("attn_nan", 1, 10, 10, 2, 16, seed=111)
    inp = make_attn_inputs(wl)
    off = inp["offsets"]
    off[0, :2, :, :, :, 0] = float("nan")
    off[0, 2:4, :, :, :, 1] = float("inf")
    off[0, 4:6, :, :, :, 0] = -1e30
    check(wl, inp)


def test_attn_equals_depthwise_deform_conv2d():
    """The operator is a depthwise deformable convolution with unit weights,
    G offset groups and the (normalized) weights as the mask: the library's
    own convolution entry on those inputs gives the same result within the
    bf16 bar."""
    wl = A("attn_vs_conv", 1, 20, 24, 4, 16, softmax=False, seed=112)
    inp = make_attn_inputs(wl)
    out = check(wl, inp).float()
    B, H, W, G, D = inp["value"].shape
    Ho, Wo = wl.out_size()
    K, C = wl.K, G * D
    x = inp["value"].reshape(B, H, W, C).permute(0, 3, 1, 2).cuda().contiguous(
        memory_format=torch.channels_last)
    offset = inp["offsets"].permute(0, 3, 4, 5, 1, 2).reshape(B, 2 * G * K, Ho, Wo).cuda().contiguous()
    mask = inp["weights"].permute(0, 3, 4, 1, 2).reshape(B, G * K, Ho, Wo).cuda().contiguous()
    weight = torch.ones(C, 1, *wl.kernel, dtype=x.dtype, device="cuda")
    conv = dcn.deform_conv2d(x, offset, weight, None, stride=wl.stride, padding=wl.padding,
                             dilation=wl.dilation, mask=mask)
    ref = conv.float().permute(0, 2, 3, 1).reshape(B, Ho, Wo, G, D)
    err = float((out - ref).abs().max() / ref.abs().max())
    assert err <= TOL["bf16"], f"attn vs depthwise deform_conv2d: {err:.3e}"
