"""A seeded sweep of random general-form problems against the oracle.

Hand-picked shapes cover the cases the kernels were designed around; this
sweep draws 40 more from a fixed seed: batch, channel counts (multiples of
16 and of 64 for the tensor-core path, odd ones for the CUDA-core path),
output counts, map sizes, kernel sizes, stride, per-axis padding,
dilation, weight groups, offset groups, mask or none, bias or none, and
the operand dtype.  Each is compared whole with the oracle at the dtype's
bar; whichever kernel the library picks must agree.
"""

import numpy as np
import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300 import Handle
from deformable_convolution_vision_gb300.inputs import GeneralWorkload as GW, make_general_inputs
from tests.helpers import TOL, compare_full, to_device

pytestmark = pytest.mark.gpu


def _draw(n, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        dtype = rng.choice(["bf16", "bf16", "f16", "f32"])
        groups = int(rng.choice([1, 1, 1, 2, 4]))
        ogroups = int(rng.choice([1, 1, 2, 4]))
        step = int(rng.choice([16, 64, 8, 3]))
        cg = step * int(rng.integers(1, 5))
        C = cg * groups
        if C % ogroups or C > 512:
            continue
        og = 16 * int(rng.integers(1, 9))
        O = og * groups
        kh, kw = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        sh, sw = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        dh, dw = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        ph, pw = int(rng.integers(0, kh * dh // 2 + 2)), int(rng.integers(0, kw * dw // 2 + 2))
        H, W = int(rng.integers(4, 40)), int(rng.integers(4, 48))
        B = int(rng.integers(1, 3))
        wl = GW(f"rand{len(out):02d}", B, C, H, W, O, kh, kw, stride=(sh, sw), padding=(ph, pw),
                dilation=(dh, dw), groups=groups, offset_groups=ogroups, dtype=str(dtype),
                offset_std=float(rng.choice([0.5, 2.0, 6.0])), mask=bool(rng.integers(0, 2)),
                seed=3000 + len(out))
        Ho, Wo = wl.out_size()
        if Ho <= 0 or Wo <= 0 or B * Ho * Wo * O * kh * kw * cg > 3e8:
            continue
        out.append(wl)
    return out


CASES = _draw(40)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_random_general_shape(wl):
    inp = make_general_inputs(wl)
    d = to_device(inp)
    with Handle() as h:
        out = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], stride=wl.stride,
                                padding=wl.padding, dilation=wl.dilation, mask=d["mask"], handle=h)
        assert dcn.dcn_sync_status(h.h) == 0
    conv = oracle.ConvDesc(stride=wl.stride, padding=wl.padding, dilation=wl.dilation,
                           groups=wl.groups, offset_groups=wl.offset_groups)
    ref = oracle.forward_ex(inp["x"], inp["offset"], inp["mask"], inp["weight"], inp["bias"], conv)
    err = compare_full(out, ref)
    assert err <= TOL[wl.dtype], f"{wl}: rel err {err:.3e}"
