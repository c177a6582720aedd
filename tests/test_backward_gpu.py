"""Backward pass on the GPU against the oracle's backward.

Every gradient (x, offset, mask, weight, bias) is compared element by
element with the oracle on the same seeded inputs and the same cotangent.
The kernels compute in fp32 from the operands' exact values for every
operand dtype (the oracle reads the same values and computes in fp64), so
the bar is the fp32 one, max|gpu - ref| / max|ref| <= 1e-4 per gradient --
except the weight gradient of 16-bit operands on the tensor-core path, whose
sampled operand is rounded to the operand type before its GEMM (the
forward's rounding), which takes that dtype's bar.  Shapes cover ragged pixel counts, several output and
channel chunks, C not a multiple of 4 (scalar reductions), offset groups
narrower than four channels, stride, dilation and groups.
"""

import numpy as np
import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300.inputs import GeneralWorkload as GW, make_general_inputs
from tests.helpers import TOL, to_device

pytestmark = pytest.mark.gpu

BAR = 1e-4
KEYS = ("grad_x", "grad_offset", "grad_mask", "grad_weight", "grad_bias")


def _rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def _cotangent(wl, dtype, seed):
    Ho, Wo = wl.out_size()
    g = torch.Generator().manual_seed(seed)
    return torch.randn(wl.B, wl.O, Ho, Wo, generator=g).to(dtype)


def _bar(wl, key, path):
    """The fp32 bar, except for the weight gradient of 16-bit operands on the
    tensor-core path: its sampled operand is rounded to the operand type
    before the contraction (as the forward's is), so it takes that type's
    bar from TOL."""
    if key == "grad_weight" and wl.dtype != "f32" and path != dcn.DCN_PATH_SIMT:
        return TOL[wl.dtype]
    return BAR


def run_backward(wl, inp, gout, path=dcn.DCN_PATH_AUTO):
    d = to_device(inp)
    g = gout.cuda().contiguous(memory_format=torch.channels_last)
    with dcn.Handle(path) as h:
        r = dcn.deform_conv2d_backward(g, d["x"], d["offset"], d["weight"], stride=wl.stride,
                                       padding=wl.padding, dilation=wl.dilation, mask=d["mask"],
                                       handle=h)
        assert dcn.dcn_sync_status(h.h) == 0
        if path != dcn.DCN_PATH_AUTO:
            assert dcn.dcn_last_path(h.h) == path
    return r


def check(wl, path=dcn.DCN_PATH_AUTO, inp=None):
    inp = make_general_inputs(wl) if inp is None else inp
    gout = _cotangent(wl, inp["x"].dtype, wl.seed + 1000)
    got = run_backward(wl, inp, gout, path)
    conv = oracle.ConvDesc(stride=wl.stride, padding=wl.padding, dilation=wl.dilation,
                           groups=wl.groups, offset_groups=wl.offset_groups)
    ref = oracle.backward_ex(inp["x"], inp["offset"], inp["mask"], inp["weight"], gout, conv)
    errs = {}
    for k in KEYS:
        if ref[k] is None:
            assert got[k] is None
            continue
        g = got[k].cpu().numpy()
        assert np.isfinite(g).all(), k
        errs[k] = _rel(g, ref[k])
        bar = _bar(wl, k, path)
        assert errs[k] <= bar, f"{wl.name} {k}: rel err {errs[k]:.3e} > {bar}"
    return errs


CASES = [
    GW("bwd_page3x3", 1, 64, 24, 20, 64, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "bf16", 2.0, True, 1),
    GW("bwd_page3x3_f32", 2, 16, 11, 13, 24, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "f32", 2.0, True, 2),
    GW("bwd_page3x3_f16", 1, 64, 17, 23, 32, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "f16", 2.0, True, 3),
    GW("bwd_7x7_no_mask", 1, 8, 20, 18, 12, 7, 7, (1, 1), (3, 3), (1, 1), 1, 1, "f32", 3.0, False, 4),
    # several output and channel chunks; pixel runs longer than one
    GW("bwd_wide", 1, 160, 26, 30, 144, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "bf16", 1.5, True, 5),
    # C % 4 != 0: scalar reductions into grad_x
    GW("bwd_c_odd", 2, 6, 9, 7, 5, 3, 2, (1, 1), (1, 0), (1, 1), 1, 1, "f32", 2.0, True, 6),
    # stride, dilation, weight groups, offset groups (two channels each)
    GW("bwd_general", 1, 8, 15, 17, 12, 3, 3, (2, 1), (1, 2), (1, 2), 2, 4, "f32", 2.0, True, 7),
    GW("bwd_general_bf16", 2, 128, 12, 10, 64, 3, 3, (1, 2), (2, 1), (2, 1), 2, 2, "bf16", 2.5, True, 8),
    GW("bwd_1x1", 1, 64, 16, 16, 64, 1, 1, (1, 1), (0, 0), (1, 1), 1, 1, "bf16", 1.0, True, 9),
]

# shapes the tensor-core column-gradient kernel takes (16-bit operands, one
# weight group, C and the offset-group width multiples of 64, O a multiple
# of 64 up to 256): ragged tiles, several tiles per CTA, several channel
# blocks and output K-blocks, offset groups, stride and dilation, no mask
TC_CASES = [
    GW("bwdtc_ragged", 2, 64, 13, 21, 64, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "bf16", 2.0, True, 31),
    GW("bwdtc_many_tiles", 1, 64, 150, 150, 64, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "bf16", 2.0, True, 32),
    GW("bwdtc_c128_o128", 1, 128, 20, 24, 128, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "bf16", 1.5, True, 33),
    GW("bwdtc_o256", 1, 64, 12, 17, 256, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "f16", 2.0, True, 34),
    GW("bwdtc_og2", 1, 128, 14, 16, 64, 3, 3, (2, 1), (1, 1), (1, 2), 1, 2, "bf16", 2.0, True, 35),
    GW("bwdtc_5x5_no_mask", 1, 64, 19, 23, 64, 5, 5, (1, 1), (2, 2), (1, 1), 1, 1, "f16", 4.0, False, 36),
    # offsets of std 8: many corners land outside the kernel's grad_x window
    # around the tile (those go straight to grad_x), the rest inside it
    GW("bwdtc_far_offsets", 2, 128, 40, 36, 64, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "bf16", 8.0, True, 37),
    # 49 x 2 (tap, 64-channel) units: more weight-gradient row blocks than a
    # quarter of the SMs, so the weight gradient runs after the data kernel
    # instead of beside it (the cases above take the side-by-side path)
    GW("bwdtc_7x7_c128", 1, 128, 21, 19, 64, 7, 7, (1, 1), (3, 3), (1, 1), 1, 1, "bf16", 2.0, True, 38),
]


@pytest.mark.parametrize("wl", TC_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("path", [dcn.DCN_PATH_TC, dcn.DCN_PATH_SIMT])
def test_backward_both_paths(wl, path):
    check(wl, path=path)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_backward_matches_oracle(wl):
    check(wl)


@pytest.mark.parametrize("path", [dcn.DCN_PATH_TC, dcn.DCN_PATH_SIMT])
def test_backward_nonfinite_offsets(path):
    """Offsets that are NaN, infinite or huge put the sampling coordinate
    outside the image (the kernels clamp it, the oracle's corner tests
    reject it): those taps add nothing to any gradient, nothing is read or
    written out of bounds, and every gradient matches the oracle."""
    wl = GW("bwd_nonfinite", 1, 64, 12, 14, 64, 3, 3, (1, 1), (1, 1), (1, 1), 1, 1, "bf16", 2.0,
            True, 39)
    inp = make_general_inputs(wl)
    off = inp["offset"]
    off[:, 0, :3] = float("nan")
    off[:, 3, 3:6] = float("inf")
    off[:, 5, 6:9] = -float("inf")
    off[:, 7, 9:] = 3e38
    off[:, 10, :, :4] = -1e30
    check(wl, path=path, inp=inp)


def test_backward_all_outside():
    """Every corner outside: every gradient is exactly zero but the bias's."""
    wl = CASES[0]
    inp = make_general_inputs(wl)
    inp["offset"][:, 0::2] = -(wl.H + 5.0)
    gout = _cotangent(wl, inp["x"].dtype, 77)
    got = run_backward(wl, inp, gout)
    for k in ("grad_x", "grad_offset", "grad_mask", "grad_weight"):
        assert not torch.any(got[k]), k
    exp = gout.float().sum(dim=(0, 2, 3))
    assert torch.allclose(got["grad_bias"].cpu(), exp, rtol=1e-5, atol=1e-4)


def test_autograd_function_matches_backward():
    from deformable_convolution_vision_gb300.autograd import deform_conv2d_autograd
    wl = CASES[1]
    inp = make_general_inputs(wl)
    d = to_device(inp)
    leaves = {k: d[k].clone().requires_grad_() for k in ("x", "offset", "mask", "weight", "bias")}
    out = deform_conv2d_autograd(leaves["x"], leaves["offset"], leaves["weight"], leaves["bias"],
                                 stride=wl.stride, padding=wl.padding, dilation=wl.dilation,
                                 mask=leaves["mask"])
    gout = _cotangent(wl, inp["x"].dtype, 99)
    out.backward(gout.cuda().contiguous(memory_format=torch.channels_last))
    conv = oracle.ConvDesc(stride=wl.stride, padding=wl.padding, dilation=wl.dilation)
    ref = oracle.backward_ex(inp["x"], inp["offset"], inp["mask"], inp["weight"], gout, conv)
    for k, name in (("x", "grad_x"), ("offset", "grad_offset"), ("mask", "grad_mask"),
                    ("weight", "grad_weight"), ("bias", "grad_bias")):
        assert _rel(leaves[k].grad.cpu().numpy(), ref[name]) <= BAR, name
