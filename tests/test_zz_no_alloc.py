"""The allocation-free entry point, dcn_forward_noalloc.

It serves callers that must not let a library allocate device memory
(plugin hosts that own all device memory, processes with a fixed memory
budget, loops where cudaMalloc/cudaFree would stall other streams).  Its
scratch lives in fixed device arrays shared by every call, so this test
calls it twice in a row, on different workloads that take different
kernels, and checks each result against dcn_forward's within the parity
tolerance and against the oracle.  A second test checks the entry
point's contract itself: once the first calls on the device have loaded
the kernels and looked up the scratch arrays, further calls change neither
the device's free memory nor the memory torch's allocator holds.  It is
collected last so that, if it fails, a run that stops at the first failure
has already run every other test.
"""

import gc

import numpy as np
import pytest
import torch

import deformable_convolution_vision_gb300 as dcn
import oracle
from deformable_convolution_vision_gb300 import binding
from deformable_convolution_vision_gb300.inputs import WORKLOADS, make_inputs
from tests.helpers import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


def _with_handle(wl, d):
    out = torch.empty((wl.B, wl.O, wl.Ho, wl.Wo), dtype=d["x"].dtype, device="cuda",
                      memory_format=torch.channels_last)
    with dcn.Handle() as h:
        dcn.dcn_forward(h.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], out,
                        wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad,
                        dcn.DCN_BF16 if wl.dtype == "bf16" else dcn.DCN_F32)
        assert dcn.dcn_sync_status(h.h) == 0
    return out


def _noalloc(wl, d):
    # poison the output so that a call which writes nothing cannot pass
    out = torch.full((wl.B, wl.O, wl.Ho, wl.Wo), float("nan"), dtype=d["x"].dtype, device="cuda")
    out = out.contiguous(memory_format=torch.channels_last)
    dcn.binding.dcn_forward_noalloc(d["x"], d["offset"], d["mask"], d["weight"], d["bias"], out,
                                    wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad,
                                    dcn.DCN_BF16 if wl.dtype == "bf16" else dcn.DCN_F32)
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    # tensor-core path, CUDA-core path, then the tensor-core path with a
    # zero-padded last channel block (C = 96)
    cases = [WORKLOADS["decoder3x3"], WORKLOADS["tiny"],
             WORKLOADS["decoder3x3"].with_(C=96, H=24, W=20, seed=95)]
    results = []
    for wl in cases:
        inp = make_inputs(wl)
        d = to_device(inp)
        results.append((wl, inp, _with_handle(wl, d), _noalloc(wl, d)))
    for wl, inp, ref, got in results:
        g = got.float().cpu().numpy()
        assert np.isfinite(g).all(), wl.name
        err = rel_err(g, ref.float().cpu().numpy())
        assert err <= TOL[wl.dtype], f"{wl.name}: {err:.3e} against dcn_forward"
        want = oracle.forward(inp["x"], inp["offset"], inp["mask"], inp["weight"], inp["bias"],
                              wl.pad)
        err = rel_err(g, want)
        assert err <= TOL[wl.dtype], f"{wl.name}: {err:.3e} against the oracle"


def test_noalloc_allocates_nothing():
    # the tensor-core and CUDA-core paths, inputs and outputs made up front
    cases = [WORKLOADS["decoder3x3"].with_(H=40, W=36, seed=96), WORKLOADS["tiny"]]
    prepared = []
    for wl in cases:
        d = to_device(make_inputs(wl))
        out = torch.empty((wl.B, wl.O, wl.Ho, wl.Wo), dtype=d["x"].dtype, device="cuda",
                          memory_format=torch.channels_last)
        prepared.append((wl, d, out))

    def call_all():
        for wl, d, out in prepared:
            dcn.binding.dcn_forward_noalloc(d["x"], d["offset"], d["mask"], d["weight"], d["bias"],
                                            out, wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad,
                                            dcn.DCN_BF16 if wl.dtype == "bf16" else dcn.DCN_F32)

    # the first calls may load the kernels and map the scratch arrays
    call_all()
    torch.cuda.synchronize()
    # tensors of earlier tests that the garbage collector frees in between
    # would move torch's own count: collect them first
    gc.collect()
    free0, _ = torch.cuda.mem_get_info()
    held0 = torch.cuda.memory_allocated()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(5):
        call_all()
    torch.cuda.synchronize()
    gc.collect()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    assert torch.cuda.memory_allocated() == held0
    assert torch.cuda.memory_reserved() == reserved0


def test_noalloc_rejects_weights_beyond_the_scratch():
    lib = binding.load()
    # 7x7, C = O = 512, bf16: 25.7 MB of packed weight > 8 MiB; nothing is launched
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    rc = lib.dcn_forward_noalloc(p, p, None, p, None, p, 1, 512, 8, 8, 512, 7, 7, 3,
                                 dcn.DCN_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == binding.STATUS_CODE["DCN_ERR_UNSUPPORTED"]
