"""The NCHW <-> NHWC layout kernels and the torchvision-layout entry.

The copies must be exact (they move bytes); the NCHW entry must give bit
for bit the channels-last entry's result, in NCHW."""

import pytest
import torch

import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300.inputs import WORKLOADS, make_inputs
from tests.helpers import TOL, compare_full, oracle_full, to_device

pytestmark = pytest.mark.gpu

CODE = {torch.float32: dcn.DCN_F32, torch.bfloat16: dcn.DCN_BF16, torch.float16: dcn.DCN_F16}


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(1, 64, 33, 40), (3, 5, 7, 9), (2, 96, 1, 1), (1, 1, 65, 31)])
def test_layout_copies_are_exact(shape, dtype):
    B, C, H, W = shape
    g = torch.Generator().manual_seed(sum(shape))
    a = torch.randn(shape, generator=g).to(dtype).cuda()
    nhwc = torch.empty((B, H, W, C), dtype=dtype, device="cuda")
    dcn.dcn_nchw_to_nhwc(a, nhwc, B, C, H, W, CODE[dtype])
    back = torch.empty_like(a)
    dcn.dcn_nhwc_to_nchw(nhwc, back, B, C, H, W, CODE[dtype])
    torch.cuda.synchronize()
    assert torch.equal(nhwc, a.permute(0, 2, 3, 1))
    assert torch.equal(back, a)


@pytest.mark.parametrize("name", ["decoder3x3", "tiny"])
def test_nchw_entry_matches_channels_last_entry(name):
    wl = WORKLOADS[name].with_(H=min(WORKLOADS[name].H, 40), W=min(WORKLOADS[name].W, 36))
    inp = make_inputs(wl)
    d = to_device(inp)
    x_nchw = inp["x"].cuda().contiguous()
    out = dcn.deform_conv2d_nchw(x_nchw, d["offset"], d["weight"], d["bias"], padding=wl.pad,
                                 mask=d["mask"])
    ref = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=wl.pad,
                            mask=d["mask"])
    torch.cuda.synchronize()
    assert out.is_contiguous()
    assert torch.equal(out, ref.contiguous())
    assert compare_full(out, oracle_full(inp, wl.pad)) <= TOL[wl.dtype]
