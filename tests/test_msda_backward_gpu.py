"""The MSDA backward on the GPU against the MSDA backward oracle.

Every gradient is compared whole (the oracle handles every case here,
the 21760-query encoder workload included, in seconds).  The kernel takes
the same 16-bit value and cotangent as the oracle and accumulates in fp32,
so the bar is the fp32 one: max |gpu - oracle| / max |oracle| <= 1e-4 per
gradient.  The value gradient is a sum of fp32 reductions whose order
varies between runs; the location and weight gradients are written once
and must repeat bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300.autograd import msda_autograd
from deformable_convolution_vision_gb300.inputs import (MSDA_WORKLOADS, MsdaWorkload,
                                                        make_msda_grad_out, make_msda_inputs)
from tests.test_msda_gpu import CASES

pytestmark = pytest.mark.gpu

BAR = 1e-4


def _rel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def run(wl, inp, go):
    method = "softmax" if wl.softmax else None
    r = dcn.msda_backward(go.cuda(), inp["value"].cuda(), wl.shapes, wl.starts,
                          inp["locations"].cuda(), inp["weights"].cuda(), method=method)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in r]


def check(wl, inp=None):
    inp = make_msda_inputs(wl) if inp is None else inp
    go = make_msda_grad_out(wl)
    got = run(wl, inp, go)
    ref = oracle.msda_backward(inp["value"], wl.shapes, wl.starts, inp["locations"],
                               inp["weights"], go, wl.softmax)
    for name, g, r in zip(("grad_value", "grad_locations", "grad_weights"), got, ref):
        assert g.shape == r.shape, name
        assert np.isfinite(g).all(), f"{wl.name} {name}: non-finite"
        err = _rel(g, r)
        assert err <= BAR, f"{wl.name} {name}: rel err {err:.3e}"
    return inp, go, got


@pytest.mark.parametrize("name", sorted(MSDA_WORKLOADS))
def test_msda_backward_workloads(name):
    check(MSDA_WORKLOADS[name])


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_msda_backward_cases(wl):
    check(wl)


EXTRA = [
    # one level, one point, one head: the smallest problem
    MsdaWorkload("msda_bwd_min", 1, 1, 8, ((4, 4),), 1, 1, "bf16", False, 0.0, 1.0, 80),
    # D = 256: 32 lanes per (query, head)
    MsdaWorkload("msda_bwd_d256", 1, 2, 256, ((9, 11), (5, 6)), 13, 4, "bf16", True, -0.1, 1.1, 81),
    # D = 24: three 8-channel chunks over two lanes
    MsdaWorkload("msda_bwd_d24", 2, 3, 24, ((7, 9), (4, 5)), 17, 4, "f16", True, -0.1, 1.1, 82),
    # many queries onto a 2x2 level: heavy contention on a few value rows
    MsdaWorkload("msda_bwd_contention", 1, 2, 32, ((2, 2),), 4096, 8, "bf16", True, 0.0, 1.0, 83),
]


@pytest.mark.parametrize("wl", EXTRA, ids=lambda w: w.name)
def test_msda_backward_extra(wl):
    check(wl)


def test_msda_backward_repeats_except_value_order():
    wl = MSDA_WORKLOADS["msda_encoder"]
    inp, go, a = check(wl)
    b = run(wl, inp, go)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    # another order of the same fp32 sums (each entry has tens of terms
    # that partly cancel): an order of magnitude inside the parity bar
    assert _rel(a[0], b[0]) <= BAR / 10


def test_msda_backward_nonfinite_locations():
    wl = MsdaWorkload("msda_bwd_nan", 1, 2, 32, ((8, 8), (4, 4)), 40, 4, "bf16", True, 0.0, 1.0, 84)
    inp = make_msda_inputs(wl)
    loc = inp["locations"]
    loc[0, :10, :, :, :, 0] = float("nan")
    loc[0, 10:20, :, :, :, 1] = float("inf")
    loc[0, 20:30, :, :, :, 0] = -1e30
    check(wl, inp)


def test_msda_autograd_matches_backward():
    wl = MSDA_WORKLOADS["msda_page"]
    inp = make_msda_inputs(wl)
    go = make_msda_grad_out(wl).cuda()
    v = inp["value"].cuda().requires_grad_(True)
    loc = inp["locations"].cuda().requires_grad_(True)
    w = inp["weights"].cuda().requires_grad_(True)
    out = msda_autograd(v, wl.shapes, wl.starts, loc, w, method="softmax")
    out.backward(go)
    gv, gl, gw = dcn.msda_backward(go, inp["value"].cuda(), wl.shapes, wl.starts,
                                   inp["locations"].cuda(), inp["weights"].cuda(), method="softmax")
    assert torch.equal(loc.grad, gl) and torch.equal(w.grad, gw)
    assert _rel(v.grad.float().cpu().numpy(), gv.to(v.dtype).float().cpu().numpy()) <= 1e-2
