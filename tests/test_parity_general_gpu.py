"""The general form (stride, per-axis padding, dilation, weight groups,
offset groups, more than 256 outputs) on the GPU against the oracle.

Both kernels are checked: the tensor-core path where the shape allows it
(one launch per weight group and per 256 outputs; offset groups as virtual
taps), and the CUDA-core path, which takes every shape.  Whole outputs are
compared with the tolerances of the page-1 tests; larger cases on
sampled pixels aimed at the 8 x 16 tile seams.  Every compared element is
also held to the per-element rounding bound of tests.helpers.
"""

import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300 import DCN_PATH_AUTO, DCN_PATH_SIMT, DCN_PATH_TC, Handle
from deformable_convolution_vision_gb300.inputs import GeneralWorkload as GW, make_general_inputs
from tests.helpers import (TOL, abs_inputs, compare_full, compare_points, elementwise_bound,
                           elementwise_ratio, sample_points, to_device)

pytestmark = pytest.mark.gpu

FULL_LIMIT = 3e9


def _conv(wl):
    return oracle.ConvDesc(stride=wl.stride, padding=wl.padding, dilation=wl.dilation,
                           groups=wl.groups, offset_groups=wl.offset_groups)


def _cost(wl):
    Ho, Wo = wl.out_size()
    return wl.B * Ho * Wo * wl.O * wl.kh * wl.kw * (wl.C // wl.groups) * 4


def run(wl, path=DCN_PATH_AUTO):
    inp = make_general_inputs(wl)
    d = to_device(inp)
    with Handle(path) as h:
        out = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], stride=wl.stride,
                                padding=wl.padding, dilation=wl.dilation, mask=d["mask"], handle=h)
        st = dcn.dcn_sync_status(h.h)
        assert st == 0, dcn.dcn_status_string(st)
        taken = dcn.dcn_last_path(h.h)
    return inp, out, taken


def check(wl, path=DCN_PATH_AUTO, expect_path=None):
    inp, out, taken = run(wl, path)
    if expect_path is not None:
        assert taken == expect_path, f"{wl.name}: path {taken}, expected {expect_path}"
    args = (inp["x"], inp["offset"], inp["mask"], inp["weight"], inp["bias"], _conv(wl))
    ai = abs_inputs(inp)
    aargs = (ai["x"], ai["offset"], ai["mask"], ai["weight"], None, _conv(wl))
    if _cost(wl) <= FULL_LIMIT:
        ref = oracle.forward_ex(*args)
        absref = oracle.forward_ex(*aargs)
        err = compare_full(out, ref)
        got = out.float().cpu().numpy()
    else:
        Ho, Wo = wl.out_size()
        nkb = wl.kh * wl.kw * -(-(wl.C // wl.groups) // 64)
        pts = sample_points(wl.B, Ho, Wo, 256, seed=wl.seed, nkb=nkb)
        ref = oracle.forward_points_ex(*args, pts)
        absref = oracle.forward_points_ex(*aargs, pts)
        err = compare_points(out, ref, pts)
        got = out.float().cpu()[pts[:, 0], :, pts[:, 1], pts[:, 2]].numpy()
    assert err <= TOL[wl.dtype], f"{wl.name} path {taken}: rel err {err:.3e}"
    K = wl.kh * wl.kw * (wl.C // wl.groups)
    ratio = elementwise_ratio(got, ref, elementwise_bound(absref, ref, wl.dtype, K))
    assert ratio <= 1.0, f"{wl.name} path {taken}: an element exceeds its error bound by {ratio:.2f}x"
    return out


# bf16 shapes the tensor-core kernel takes
TC_GENERAL = [
    GW("stride2", 2, 64, 33, 47, 64, 3, 3, stride=(2, 2), padding=(1, 1), seed=40),
    GW("stride_hw", 1, 64, 40, 36, 48, 3, 3, stride=(1, 2), padding=(1, 1), seed=41),
    GW("dilation2", 1, 64, 30, 34, 64, 3, 3, padding=(2, 2), dilation=(2, 2), seed=42),
    GW("pad_asym_rect", 1, 64, 21, 26, 32, 3, 5, padding=(0, 3), dilation=(1, 2), seed=43),
    GW("groups2", 2, 128, 17, 20, 64, 3, 3, padding=(1, 1), groups=2, seed=44),
    GW("offset_groups2", 1, 128, 18, 22, 64, 3, 3, padding=(1, 1), offset_groups=2, seed=45),
    # weight groups of 128 channels, offset groups of 64: two virtual taps per tap
    GW("g2_og4", 1, 256, 12, 17, 128, 3, 3, padding=(1, 1), groups=2, offset_groups=4, seed=46),
    # offset groups of 128 channels over weight groups of 64
    GW("g4_og2", 1, 256, 12, 15, 64, 3, 3, padding=(1, 1), groups=4, offset_groups=2, seed=47),
    # more than 256 outputs: two launches of 256 and 64
    GW("o320", 1, 64, 13, 18, 320, 3, 3, padding=(1, 1), seed=48),
    # grouped, strided and over the SM count in tiles: stream-K per launch
    GW("streamk_groups", 1, 128, 129, 170, 64, 3, 3, stride=(1, 1), padding=(1, 1), groups=2,
       offset_groups=2, seed=49),
    GW("streamk_stride2", 2, 64, 260, 200, 32, 5, 5, stride=(2, 2), padding=(2, 2), dilation=(1, 1),
       offset_std=3.0, seed=50),
    GW("no_mask_groups", 1, 128, 16, 19, 32, 3, 3, padding=(1, 1), groups=2, offset_groups=2,
       mask=False, seed=51),
]

# shapes only the CUDA-core kernel takes, both dtypes
SIMT_GENERAL = [
    GW("f32_all", 2, 6, 11, 13, 9, 3, 2, stride=(2, 1), padding=(1, 2), dilation=(1, 2), groups=3,
       offset_groups=2, dtype="f32", seed=60),
    GW("f32_og_straddle", 1, 12, 9, 8, 8, 3, 3, padding=(1, 1), groups=2, offset_groups=3,
       dtype="f32", seed=61),
    GW("f32_depthwise", 1, 16, 10, 12, 16, 3, 3, padding=(1, 1), groups=16, offset_groups=4,
       dtype="f32", seed=62),
    GW("f32_stride3_dil3", 1, 5, 23, 19, 7, 3, 3, stride=(3, 3), padding=(2, 0), dilation=(3, 2),
       dtype="f32", seed=63),
    GW("bf16_og32", 1, 96, 14, 15, 40, 3, 3, padding=(1, 1), offset_groups=3, seed=64),
    GW("bf16_groups3_o24", 1, 192, 9, 10, 24, 3, 3, padding=(1, 1), groups=3, seed=65),
]


@pytest.mark.parametrize("wl", TC_GENERAL, ids=lambda w: w.name)
def test_general_tc(wl):
    check(wl, expect_path=DCN_PATH_TC)


@pytest.mark.parametrize("wl", TC_GENERAL[:9], ids=lambda w: w.name)
def test_general_tc_shapes_on_cuda_cores(wl):
    check(wl, path=DCN_PATH_SIMT, expect_path=DCN_PATH_SIMT)


@pytest.mark.parametrize("wl", SIMT_GENERAL, ids=lambda w: w.name)
def test_general_simt(wl):
    check(wl, expect_path=DCN_PATH_SIMT)


def test_forced_tc_on_unsupported_general_shape_launches_nothing():
    wl = SIMT_GENERAL[-2]
    with pytest.raises(dcn.DcnError) as e:
        run(wl, DCN_PATH_TC)
    assert "UNSUPPORTED" in str(e.value)


def test_page_form_equals_general_form():
    """dcn_forward and dcn_forward_ex with stride 1, dilation 1, one group
    give the same bits."""
    wl = GW("page", 1, 64, 20, 24, 64, 3, 3, padding=(1, 1), seed=70)
    inp = make_general_inputs(wl)
    d = to_device(inp)
    Ho, Wo = wl.out_size()
    a = torch.empty((1, 64, Ho, Wo), dtype=torch.bfloat16, device="cuda",
                    memory_format=torch.channels_last)
    b = torch.empty_like(a)
    with Handle() as h:
        dcn.dcn_forward(h.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], a,
                        1, 64, 20, 24, 64, 3, 3, 1, dcn.DCN_BF16)
        desc = dcn.ConvDesc(1, 64, 20, 24, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1, 1)
        dcn.dcn_forward_ex(h.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], b, desc,
                           dcn.DCN_BF16)
        assert dcn.dcn_sync_status(h.h) == 0
    assert torch.equal(a, b)


def test_packed_halves_general():
    wl = TC_GENERAL[6]
    inp = make_general_inputs(wl)
    d = to_device(inp)
    Ho, Wo = wl.out_size()
    desc = dcn.ConvDesc(wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, *wl.stride, *wl.padding,
                        *wl.dilation, wl.groups, wl.offset_groups)
    ref = check(wl)
    out = torch.empty_like(ref)
    with Handle() as h:
        dcn.dcn_pack_weight_ex(h.h, d["weight"], desc, dcn.DCN_BF16)
        dcn.dcn_forward_packed_ex(h.h, d["x"], d["offset"], d["mask"], d["bias"], out, desc,
                                  dcn.DCN_BF16)
        assert dcn.dcn_sync_status(h.h) == 0
        # a different pack key is refused
        bad = dcn.ConvDesc(wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, *wl.stride, *wl.padding,
                           *wl.dilation, 1, wl.offset_groups)
        with pytest.raises(dcn.DcnError):
            dcn.dcn_forward_packed_ex(h.h, d["x"], d["offset"], d["mask"], d["bias"], out, bad,
                                      dcn.DCN_BF16)
    assert torch.equal(out, ref)
