"""Channel counts that are not a multiple of 64 on the tensor-core kernel.

The kernel contracts 64 channels of one tap per K-block.  For C % 16 == 0
and C % 64 != 0 the packed weight completes each tap's last block with
zero rows; the sampler lanes whose channels lie past C fill their A
columns from the last 16 real channels, which those zero rows cancel, so
every shape here must match the oracle like the whole-block shapes do.
Cases cover one, two and three blocks per tap with 16, 32 and 48 real
channels in the last one, the
persistent stream-K schedule (one and two blocks per tap), both combine
precisions, fp16, the general form (weight groups whose width is not a
multiple of 64), the CUDA-core kernel reading the padded pack, and the
pack / packed-forward halves.
"""

import pytest
import torch

import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300 import (DCN_PATH_SIMT, DCN_PATH_TC, DCN_SAMPLE_F32,
                                                 DCN_SAMPLE_INPUT_DTYPE, Handle)
from deformable_convolution_vision_gb300.inputs import GeneralWorkload as GW
from deformable_convolution_vision_gb300.inputs import Workload, make_inputs
from tests.helpers import to_device
from tests.test_parity_gpu import check
from tests.test_parity_general_gpu import check as check_general

pytestmark = pytest.mark.gpu

PAD_SHAPES = [
    Workload("tc_c16", 1, 16, 13, 11, 32, 3, 3, 1, "bf16", 2.0, "sigmoid", 0.0, 0.1, 80),
    Workload("tc_c32", 2, 32, 20, 17, 64, 3, 3, 1, "bf16", 2.0, "uniform", 0.0, 0.1, 81),
    Workload("tc_c48_7x7_no_mask", 1, 48, 24, 30, 64, 7, 7, 3, "bf16", 5.0, "none", 0.0, 0.0, 82),
    # two blocks per tap, the second one half real
    Workload("tc_c96_o112", 1, 96, 15, 19, 112, 3, 3, 1, "bf16", 2.0, "sigmoid", 0.0, 0.1, 83),
    # three blocks per tap, 16 real channels in the last
    Workload("tc_c144_5x5", 1, 144, 11, 13, 48, 5, 5, 2, "bf16", 3.0, "uniform_zero10", 0.0, 0.1, 84),
    Workload("tc_c208_o256", 1, 208, 9, 10, 256, 3, 3, 1, "bf16", 1.5, "sigmoid", 0.0, 0.1, 85),
    # more tiles than SMs: stream-K with one (alternate taps per team) and
    # two blocks per tap
    Workload("tc_streamk_c32", 2, 32, 64, 160, 64, 3, 3, 1, "bf16", 2.0, "sigmoid", 0.0, 0.1, 86),
    Workload("tc_streamk_c80", 1, 80, 96, 208, 32, 3, 3, 1, "bf16", 2.0, "uniform", 0.0, 0.1, 87),
]


@pytest.mark.parametrize("wl", PAD_SHAPES, ids=lambda w: w.name)
def test_padded_blocks_on_tensor_cores(wl):
    check(wl, expect_path=DCN_PATH_TC, samples=(DCN_SAMPLE_INPUT_DTYPE, DCN_SAMPLE_F32))


@pytest.mark.parametrize("idx", [0, 3, 4, 6])
def test_padded_blocks_f16(idx):
    wl = PAD_SHAPES[idx]
    check(wl.with_(dtype="f16", name=wl.name + "_f16"), expect_path=DCN_PATH_TC)


@pytest.mark.parametrize("idx", [1, 4])
def test_padded_pack_on_cuda_cores(idx):
    # the CUDA-core kernel reads the same zero-padded, permuted pack
    check(PAD_SHAPES[idx], path=DCN_PATH_SIMT, expect_path=DCN_PATH_SIMT)


PAD_GENERAL = [
    GW("groups2_cg48", 1, 96, 17, 20, 64, 3, 3, padding=(1, 1), groups=2, seed=90),
    # weight groups of 32 inside offset groups of 64: one virtual tap per tap
    GW("groups4_cg32_og2", 1, 128, 14, 18, 64, 3, 3, padding=(1, 1), groups=4, offset_groups=2,
       seed=91),
    GW("stride2_c96", 2, 96, 33, 41, 48, 3, 3, stride=(2, 2), padding=(1, 1), seed=92),
    GW("dil2_c112_o320", 1, 112, 16, 19, 320, 3, 3, padding=(2, 2), dilation=(2, 2), seed=93),
]


@pytest.mark.parametrize("wl", PAD_GENERAL, ids=lambda w: w.name)
def test_padded_blocks_general(wl):
    check_general(wl, expect_path=DCN_PATH_TC)


def test_packed_halves_with_padded_pack():
    wl = PAD_SHAPES[3]
    d = to_device(make_inputs(wl))
    outs = []
    with Handle() as h:
        for halves in (False, True):
            out = torch.empty((wl.B, wl.O, wl.Ho, wl.Wo), dtype=torch.bfloat16, device="cuda",
                              memory_format=torch.channels_last)
            args = (wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, dcn.DCN_BF16)
            if halves:
                dcn.dcn_pack_weight(h.h, d["weight"], wl.O, wl.C, wl.kh, wl.kw, dcn.DCN_BF16)
                dcn.dcn_forward_packed(h.h, d["x"], d["offset"], d["mask"], d["bias"], out, *args)
            else:
                dcn.dcn_forward(h.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], out,
                                *args)
            assert dcn.dcn_sync_status(h.h) == 0
            assert dcn.dcn_last_path(h.h) == DCN_PATH_TC
            outs.append(out)
    assert torch.equal(outs[0], outs[1])
