"""fp16 operands on the GPU against the oracle.

The same method with x, weight and out in IEEE half precision: the
bilinear combine in fp16 (or fp32 when selected), tcgen05 kind::f16 with
fp16 A and B and fp32 accumulation, the CUDA-core kernel for shapes outside
the tensor-core envelope.  The oracle reads the fp16 inputs' exact values
and computes in fp64; the bar is tests.helpers.TOL["f16"].
"""

import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300 import (DCN_PATH_SIMT, DCN_PATH_TC, DCN_SAMPLE_F32,
                                                 DCN_SAMPLE_INPUT_DTYPE, Handle)
from deformable_convolution_vision_gb300.inputs import (GeneralWorkload as GW, WORKLOADS,
                                                        make_inputs, make_general_inputs)
from tests.helpers import TOL, compare_full, compare_points, to_device
from tests.test_parity_gpu import TC_SHAPES, check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["decoder3x3", "aspp7x7", "backbone3x3", "boundary5x5"])
def test_workload_f16(name):
    # full size, compared on the seam-aimed pixels (the bf16 runs compare whole)
    check(WORKLOADS[name].with_(dtype="f16"), expect_path=DCN_PATH_TC, full_limit=4e9)


@pytest.mark.parametrize("idx", [0, 1, 4, 7, 10, 12])
def test_tc_shapes_f16(idx):
    wl = TC_SHAPES[idx]
    check(wl.with_(dtype="f16", name=wl.name + "_f16"), expect_path=DCN_PATH_TC,
          samples=(DCN_SAMPLE_INPUT_DTYPE, DCN_SAMPLE_F32))


@pytest.mark.parametrize("path", [DCN_PATH_SIMT, DCN_PATH_TC])
def test_both_f16_paths(path):
    wl = WORKLOADS["decoder3x3"].with_(dtype="f16", H=40, W=56, seed=41)
    check(wl, path=path, expect_path=path)


def test_simt_odd_f16():
    # C % 16 != 0: only the CUDA-core kernel takes it
    wl = WORKLOADS["decoder3x3"].with_(dtype="f16", C=24, O=40, H=10, W=9, seed=42)
    check(wl, expect_path=DCN_PATH_SIMT)


def test_all_samples_outside_give_bias_f16():
    wl = WORKLOADS["decoder3x3"].with_(H=32, W=32, dtype="f16", seed=43)
    inp = make_inputs(wl)
    inp["offset"][:, 0::2] = -(wl.H + 5.0)
    d = to_device(inp)
    out = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=wl.pad,
                            mask=d["mask"]).float().cpu()
    exp = inp["bias"].to(torch.float16).float()
    assert torch.equal(out, exp.view(1, -1, 1, 1).expand_as(out))


@pytest.mark.parametrize("wl", [
    GW("f16_groups_og", 1, 128, 30, 34, 64, 3, 3, (2, 1), (1, 2), (1, 2), 2, 2, "f16", 2.0, True, 44),
    GW("f16_og4_o320", 2, 256, 12, 14, 320, 3, 3, (1, 1), (1, 1), (1, 1), 1, 4, "f16", 2.0, True, 45),
], ids=lambda w: w.name)
def test_general_f16(wl):
    inp = make_general_inputs(wl)
    d = to_device(inp)
    with Handle() as h:
        out = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], stride=wl.stride,
                                padding=wl.padding, dilation=wl.dilation, mask=d["mask"], handle=h)
        assert dcn.dcn_sync_status(h.h) == 0
        assert dcn.dcn_last_path(h.h) == DCN_PATH_TC
    conv = oracle.ConvDesc(stride=wl.stride, padding=wl.padding, dilation=wl.dilation,
                           groups=wl.groups, offset_groups=wl.offset_groups)
    ref = oracle.forward_ex(inp["x"], inp["offset"], inp["mask"], inp["weight"], inp["bias"], conv)
    assert compare_full(out, ref) <= TOL["f16"]
