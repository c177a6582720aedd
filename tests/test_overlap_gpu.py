"""The fused kernel overlaps the weight pack of the same dcn_forward call
(a programmatic dependent launch whose weight loads wait for the pack).
Once a handle's workspace exists, every later call on it takes that path;
a kernel that read the packed weight early would see the previous call's
weight.  Each case runs a call with one weight and then calls with others on
the same handle, and checks each output bit for bit against a fresh handle's
(whose first call is an ordinary launch) and against the oracle."""

import pytest
import torch

import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300 import DCN_PATH_TC, Handle
from deformable_convolution_vision_gb300.inputs import WORKLOADS, make_inputs
from tests.helpers import TOL, compare_full, oracle_full, to_device

pytestmark = pytest.mark.gpu


def _call(h, d, wl, weight):
    out = torch.empty((wl.B, wl.O, wl.Ho, wl.Wo), dtype=d["x"].dtype, device="cuda",
                      memory_format=torch.channels_last)
    code = {torch.bfloat16: dcn.DCN_BF16, torch.float16: dcn.DCN_F16}[d["x"].dtype]
    dcn.dcn_forward(h.h, d["x"], d["offset"], d["mask"], weight, d["bias"], out,
                    wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, code)
    return out


@pytest.mark.parametrize("wl", [
    # one tile per CTA (fewer tiles than SMs)
    WORKLOADS["decoder3x3"].with_(H=40, W=48, seed=51),
    # persistent stream-K launch (more tiles than SMs)
    WORKLOADS["decoder3x3"].with_(B=2, H=96, W=160, seed=52),
    WORKLOADS["decoder3x3"].with_(H=40, W=48, dtype="f16", seed=53),
], ids=["one_tile", "streamk", "f16"])
def test_calls_on_one_handle_see_their_own_weight(wl):
    inp = make_inputs(wl)
    d = to_device(inp)
    g = torch.Generator().manual_seed(wl.seed + 100)
    weights = [d["weight"]] + [
        (torch.randn(d["weight"].shape, generator=g) / (wl.taps * wl.C) ** 0.5)
        .to(d["weight"].dtype).cuda() for _ in range(3)]
    with Handle() as h:
        outs = [_call(h, d, wl, w) for w in weights]
        assert dcn.dcn_sync_status(h.h) == 0
        assert dcn.dcn_last_path(h.h) == DCN_PATH_TC
    for w, out in zip(weights, outs):
        with Handle() as fresh:
            ref = _call(fresh, d, wl, w)
            assert dcn.dcn_sync_status(fresh.h) == 0
        assert torch.equal(out, ref)
        cpu = dict(inp, weight=w.cpu())
        assert compare_full(out, oracle_full(cpu, wl.pad)) <= TOL[wl.dtype]


@pytest.mark.parametrize("name", ["aspp7x7", "boundary5x5"])
def test_full_size_in_the_bench_configuration(name):
    """The benchmark's launch configuration: one handle, repeated
    dcn_forward calls (so every call after the first overlaps its weight
    pack), the persistent stream-K launch.  The third call's output is
    compared with the oracle on sampled pixels."""
    import oracle
    from tests.helpers import compare_points, sample_points
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    d = to_device(inp)
    with Handle() as h:
        outs = [_call(h, d, wl, d["weight"]) for _ in range(3)]
        assert dcn.dcn_sync_status(h.h) == 0
        assert dcn.dcn_last_path(h.h) == DCN_PATH_TC
    assert torch.equal(outs[0], outs[2])
    pts = sample_points(wl.B, wl.Ho, wl.Wo, 256, seed=wl.seed + 9)
    ref = oracle.forward_points(inp["x"], inp["offset"], inp["mask"], inp["weight"], inp["bias"],
                                wl.pad, pts)
    assert compare_points(outs[2], ref, pts) <= TOL[wl.dtype]
