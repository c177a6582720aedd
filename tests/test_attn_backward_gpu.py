"""The single-scale sampling backward on the GPU against its oracle.

Every gradient is compared whole.  The kernel takes the same 16-bit value
and cotangent as the oracle and accumulates in fp32, so the bar is the
fp32 one: max |gpu - oracle| / max |oracle| <= 1e-4 per gradient.  The
value gradient is a sum of fp32 reductions whose order varies between
runs; the offset and weight gradients are written once and must repeat
bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300.autograd import attn_autograd
from deformable_convolution_vision_gb300.inputs import (ATTN_WORKLOADS, AttnWorkload,
                                                        make_attn_grad_out, make_attn_inputs)
from tests.test_attn_gpu import CASES

pytestmark = pytest.mark.gpu

BAR = 1e-4


def _rel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def run(wl, inp, go):
    method = "softmax" if wl.softmax else None
    r = dcn.attn_backward(go.cuda(), inp["value"].cuda(), inp["offsets"].cuda(),
                          inp["weights"].cuda(), wl.kernel, wl.stride, wl.padding, wl.dilation,
                          method=method)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in r]


def check(wl, inp=None):
    inp = make_attn_inputs(wl) if inp is None else inp
    go = make_attn_grad_out(wl)
    got = run(wl, inp, go)
    ref = oracle.attn_backward(inp["value"], inp["offsets"], inp["weights"], go, wl.kernel,
                               wl.stride, wl.padding, wl.dilation, wl.softmax)
    for name, g, r in zip(("grad_value", "grad_offsets", "grad_weights"), got, ref):
        assert g.shape == r.shape, name
        assert np.isfinite(g).all(), f"{wl.name} {name}: non-finite"
        err = _rel(g, r)
        assert err <= BAR, f"{wl.name} {name}: rel err {err:.3e}"
    return inp, go, got


@pytest.mark.parametrize("name", sorted(ATTN_WORKLOADS))
def test_attn_backward_workloads(name):
    check(ATTN_WORKLOADS[name])


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_attn_backward_cases(wl):
    check(wl)


def test_attn_backward_repeats_except_value_order():
    wl = ATTN_WORKLOADS["attn_page"]
    inp, go, a = check(wl)
    b = run(wl, inp, go)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert _rel(a[0], b[0]) <= BAR / 10


def test_attn_backward_nonfinite_offsets():
    wl = AttnWorkload("attn_bwd_nan", 1, 10, 10, 2, 16, seed=120)
    inp = make_attn_inputs(wl)
    off = inp["offsets"]
    off[0, :2, :, :, :, 0] = float("nan")
    off[0, 2:4, :, :, :, 1] = float("inf")
    off[0, 4:6, :, :, :, 0] = -1e30
    check(wl, inp)


def test_attn_autograd_matches_backward():
    wl = ATTN_WORKLOADS["attn_page"]
    inp = make_attn_inputs(wl)
    go = make_attn_grad_out(wl).cuda()
    v = inp["value"].cuda().requires_grad_(True)
    off = inp["offsets"].cuda().requires_grad_(True)
    w = inp["weights"].cuda().requires_grad_(True)
    out = attn_autograd(v, off, w, wl.kernel, wl.stride, wl.padding, wl.dilation, method="softmax")
    out.backward(go)
    gv, go_, gw = dcn.attn_backward(go, inp["value"].cuda(), inp["offsets"].cuda(),
                                    inp["weights"].cuda(), wl.kernel, wl.stride, wl.padding,
                                    wl.dilation, method="softmax")
    assert torch.equal(off.grad, go_) and torch.equal(w.grad, gw)
    assert _rel(v.grad.float().cpu().numpy(), gv.to(v.dtype).float().cpu().numpy()) <= 1e-2
