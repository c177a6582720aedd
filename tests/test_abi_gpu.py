"""C-ABI behaviour on a GB300: argument errors, forced paths, the packed
weight halves, the host-buffer entry point and the bounded-wait status."""

import numpy as np
import pytest
import torch

import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300 import binding
from deformable_convolution_vision_gb300.inputs import WORKLOADS, make_inputs
from tests.helpers import TOL, compare_full, oracle_full, to_device

pytestmark = pytest.mark.gpu

E = binding.STATUS_CODE


@pytest.fixture
def handle():
    with dcn.Handle() as h:
        yield h


def _args(d, wl):
    return [d["x"].data_ptr(), d["offset"].data_ptr(),
            None if d["mask"] is None else d["mask"].data_ptr(), d["weight"].data_ptr(),
            None if d["bias"] is None else d["bias"].data_ptr()]


def test_argument_errors(handle):
    lib = binding.load()
    wl = WORKLOADS["tiny"]
    d = to_device(make_inputs(wl))
    out = torch.empty(wl.B * wl.Ho * wl.Wo * wl.O, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    x, off, m, w, b = _args(d, wl)
    ok = [wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, 0]

    def call(xx=x, oo=off, ww=w, out_p=out.data_ptr(), dims=ok):
        return lib.dcn_forward(handle.h, xx, oo, m, ww, b, out_p, *dims, s)

    assert call() == E["DCN_OK"]
    assert call(xx=None) == E["DCN_ERR_INVALID_ARG"]
    assert call(oo=None) == E["DCN_ERR_INVALID_ARG"]
    assert call(ww=None) == E["DCN_ERR_INVALID_ARG"]
    assert call(out_p=None) == E["DCN_ERR_INVALID_ARG"]
    assert call(xx=x + 2) == E["DCN_ERR_INVALID_ARG"]           # misaligned fp32
    for bad in ([0] + ok[1:], ok[:1] + [-1] + ok[2:], ok[:7] + [-1, 0], ok[:8] + [7],
                [1, 4, 2, 2, 3, 5, 5, 0, 0],                       # Ho <= 0
                [1 << 16, 1 << 16, 1, 1, 1, 1, 1, 0, 0]):          # B*H*W*C >= 2^31
        assert call(dims=bad) == E["DCN_ERR_INVALID_ARG"], bad
    assert dcn.dcn_sync_status(handle.h) == 0


def test_forced_tc_path_rejects_unsupported_shapes(handle):
    dcn.dcn_set_path(handle.h, dcn.DCN_PATH_TC)
    wl = WORKLOADS["tiny"]  # fp32: no tensor-core path
    inp = make_inputs(wl)
    d = to_device(inp)
    out = torch.empty((wl.B, wl.O, wl.Ho, wl.Wo), device="cuda", memory_format=torch.channels_last)
    with pytest.raises(dcn.DcnError) as e:
        dcn.dcn_forward(handle.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], out,
                        wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, dcn.DCN_F32)
    assert e.value.status == E["DCN_ERR_UNSUPPORTED"]
    wl2 = WORKLOADS["decoder3x3"].with_(C=24, H=16, W=16)  # C % 16 != 0
    d2 = to_device(make_inputs(wl2))
    out2 = torch.empty((1, wl2.O, wl2.Ho, wl2.Wo), dtype=torch.bfloat16, device="cuda",
                       memory_format=torch.channels_last)
    with pytest.raises(dcn.DcnError) as e:
        dcn.dcn_forward(handle.h, d2["x"], d2["offset"], d2["mask"], d2["weight"], d2["bias"],
                        out2, 1, 24, 16, 16, wl2.O, 3, 3, 1, dcn.DCN_BF16)
    assert e.value.status == E["DCN_ERR_UNSUPPORTED"]
    assert dcn.dcn_sync_status(handle.h) == 0


def test_packed_halves_match_forward(handle):
    wl = WORKLOADS["decoder3x3"].with_(H=48, W=40)
    inp = make_inputs(wl)
    d = to_device(inp)
    shape = (wl.B, wl.O, wl.Ho, wl.Wo)
    a = torch.empty(shape, dtype=torch.bfloat16, device="cuda", memory_format=torch.channels_last)
    b = torch.empty_like(a)
    dims = (wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, dcn.DCN_BF16)
    dcn.dcn_forward(handle.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], a, *dims)
    dcn.dcn_pack_weight(handle.h, d["weight"], wl.O, wl.C, wl.kh, wl.kw, dcn.DCN_BF16)
    dcn.dcn_forward_packed(handle.h, d["x"], d["offset"], d["mask"], d["bias"], b, *dims)
    assert dcn.dcn_sync_status(handle.h) == 0
    assert torch.equal(a, b)
    # a packed weight of another shape is refused
    with pytest.raises(dcn.DcnError) as e:
        dcn.dcn_forward_packed(handle.h, d["x"], d["offset"], d["mask"], d["bias"], b,
                               wl.B, wl.C, wl.H, wl.W, wl.O, 5, 5, 2, dcn.DCN_BF16)
    assert e.value.status == E["DCN_ERR_INVALID_ARG"]


@pytest.mark.parametrize("name", ["tiny", "decoder3x3"])
def test_host_entry_point_matches_device(handle, name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    # host buffers in the ABI layouts, pinned
    x = inp["x"].permute(0, 2, 3, 1).contiguous().pin_memory()
    off = inp["offset"].pin_memory()
    m = inp["mask"].pin_memory()
    w = inp["weight"].contiguous().pin_memory()
    bias = inp["bias"].pin_memory()
    out = torch.empty((wl.B, wl.Ho, wl.Wo, wl.O), dtype=x.dtype).pin_memory()
    code = dcn.DCN_F32 if wl.dtype == "f32" else dcn.DCN_BF16
    dcn.dcn_forward_host(handle.h, x, off, m, w, bias, out, wl.B, wl.C, wl.H, wl.W, wl.O,
                         wl.kh, wl.kw, wl.pad, code)
    d = to_device(inp)
    ref = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=wl.pad,
                            mask=d["mask"])
    assert torch.equal(out, ref.permute(0, 2, 3, 1).cpu())
    assert compare_full(out.permute(0, 3, 1, 2), oracle_full(inp, wl.pad)) <= TOL[wl.dtype]


def test_bounded_wait_reports_timeout_and_context_survives(handle):
    dcn.dcn_selftest_timeout(handle.h, 20_000_000)  # 20 ms
    assert dcn.dcn_sync_status(handle.h) == E["DCN_ERR_TIMEOUT"]
    assert dcn.dcn_sync_status(handle.h) == 0       # the word is cleared once read
    wl = WORKLOADS["tiny"]
    inp = make_inputs(wl)
    d = to_device(inp)
    out = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=wl.pad,
                            mask=d["mask"], handle=handle)
    assert dcn.dcn_sync_status(handle.h) == 0
    assert compare_full(out, oracle_full(inp, wl.pad)) <= TOL["f32"]


def _host_call(handle, wl, inp, code):
    x = inp["x"].permute(0, 2, 3, 1).contiguous().pin_memory()
    off = inp["offset"].pin_memory()
    m = None if inp["mask"] is None else inp["mask"].pin_memory()
    w = inp["weight"].contiguous().pin_memory()
    bias = None if inp["bias"] is None else inp["bias"].pin_memory()
    out = torch.empty((wl.B, wl.Ho, wl.Wo, wl.O), dtype=x.dtype).pin_memory()
    dcn.dcn_forward_host(handle.h, x, off, m, w, bias, out, wl.B, wl.C, wl.H, wl.W, wl.O,
                         wl.kh, wl.kw, wl.pad, code)
    return out.permute(0, 3, 1, 2)


@pytest.mark.parametrize("wl", [
    # three bands of 96, 96 and 64 rows (the benchmark's end-to-end call)
    WORKLOADS["aspp7x7"],
    # two images, two bands each, both ragged (27 and 16 rows of Ho = 43)
    WORKLOADS["decoder3x3"].with_(B=2, H=43, W=50, seed=81),
    # five images: one band per image; no mask, no bias
    WORKLOADS["decoder3x3"].with_(B=5, H=20, W=24, mask="none", bias_std=0.0, seed=82),
    # fp16, and fp32 on the CUDA-core kernel, banded
    WORKLOADS["decoder3x3"].with_(H=70, W=33, dtype="f16", seed=83),
    WORKLOADS["decoder3x3"].with_(C=16, O=24, H=66, W=30, dtype="f32", seed=84),
], ids=["aspp7x7", "b2_ragged", "b5_nomask", "f16", "f32"])
def test_host_entry_point_bands(handle, wl):
    """The host-buffer entry runs as a pipeline over bands of output rows
    (uploads, kernels and downloads on separate streams); every band's
    result must match the oracle."""
    import oracle
    from tests.helpers import compare_points, sample_points
    inp = make_inputs(wl)
    code = {"f32": dcn.DCN_F32, "bf16": dcn.DCN_BF16, "f16": dcn.DCN_F16}[wl.dtype]
    out = _host_call(handle, wl, inp, code)
    assert dcn.dcn_sync_status(handle.h) == 0
    if wl.pixels * wl.O * wl.taps * wl.C <= 1e9:
        assert compare_full(out, oracle_full(inp, wl.pad)) <= TOL[wl.dtype]
    else:
        pts = sample_points(wl.B, wl.Ho, wl.Wo, 256, seed=wl.seed)
        ref = oracle.forward_points(inp["x"], inp["offset"], inp["mask"], inp["weight"],
                                    inp["bias"], wl.pad, pts)
        assert compare_points(out, ref, pts) <= TOL[wl.dtype]
    # a second call on the same handle (streams and events reused) agrees
    again = _host_call(handle, wl, inp, code)
    assert torch.equal(out, again)


def test_host_entry_point_pageable_memory(handle):
    """dcn_forward_host with pageable (not pinned) host buffers: slower,
    the same result as with pinned ones."""
    wl = WORKLOADS["decoder3x3"].with_(H=40, W=48, seed=85)
    inp = make_inputs(wl)
    pinned = _host_call(handle, wl, inp, dcn.DCN_BF16)
    x = inp["x"].permute(0, 2, 3, 1).contiguous()
    out = torch.empty((wl.B, wl.Ho, wl.Wo, wl.O), dtype=x.dtype)
    dcn.dcn_forward_host(handle.h, x, inp["offset"].contiguous(), inp["mask"].contiguous(),
                         inp["weight"].contiguous(), inp["bias"].contiguous(), out, wl.B, wl.C,
                         wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, dcn.DCN_BF16)
    assert dcn.dcn_sync_status(handle.h) == 0
    assert torch.equal(out.permute(0, 3, 1, 2), pinned)


def test_python_entries_refuse_wrong_buffers():
    """``out`` of another dtype or layout, and a bias longer than O, are
    refused before the library is called.  Every wrong buffer here is at
    least as large as the right one, so nothing could be written out of
    bounds even if a check were missing."""
    from deformable_convolution_vision_gb300.inputs import (ATTN_WORKLOADS, MSDA_WORKLOADS,
                                                            make_attn_inputs, make_msda_inputs)
    wl = WORKLOADS["decoder3x3"].with_(H=24, W=40)
    d = to_device(make_inputs(wl))
    shape = (wl.B, wl.O, wl.Ho, wl.Wo)
    wrong = {
        "fp32 out": torch.empty(shape, device="cuda", memory_format=torch.channels_last),
        "NCHW out": torch.empty(shape, dtype=torch.bfloat16, device="cuda"),
    }
    for name, out in wrong.items():
        with pytest.raises(ValueError, match="out must be"):
            dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=wl.pad,
                              mask=d["mask"], out=out)
    long_bias = torch.zeros(wl.O + 1, device="cuda")
    with pytest.raises(ValueError, match="bias must be"):
        dcn.deform_conv2d(d["x"], d["offset"], d["weight"], long_bias, padding=wl.pad,
                          mask=d["mask"])
    ref = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=wl.pad,
                            mask=d["mask"])
    out = torch.empty_like(ref)
    dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=wl.pad,
                      mask=d["mask"], out=out)
    assert torch.equal(out, ref)

    m = MSDA_WORKLOADS["msda_page"]
    mi = {k: v.cuda() for k, v in make_msda_inputs(m).items()}
    with pytest.raises(ValueError, match="out must be"):
        dcn.msda(mi["value"], m.shapes, m.starts, mi["locations"], mi["weights"],
                 out=torch.empty((m.B, m.Q, m.G, m.D), device="cuda"))
    a = ATTN_WORKLOADS["attn_page"]
    ai = {k: v.cuda() for k, v in make_attn_inputs(a).items()}
    Ho, Wo = a.out_size()
    with pytest.raises(ValueError, match="out must be"):
        dcn.attn(ai["value"], ai["offsets"], ai["weights"], a.kernel, a.stride, a.padding,
                 a.dilation, out=torch.empty((a.B, Ho, Wo, a.G, a.D), device="cuda"))
