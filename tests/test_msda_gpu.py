"""Multi-scale deformable attention on the GPU against the MSDA oracle.

Whole outputs are compared (the oracle handles every case here in
seconds), with the operand dtype's bar from tests.helpers.TOL: the kernel
computes in fp32 and rounds once to the output dtype.
"""

import numpy as np
import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300.inputs import (MSDA_WORKLOADS, MsdaWorkload,
                                                        make_msda_inputs)
from tests.helpers import TOL

pytestmark = pytest.mark.gpu


def check(wl, inp=None):
    inp = make_msda_inputs(wl) if inp is None else inp
    out = dcn.msda(inp["value"].cuda(), wl.shapes, wl.starts, inp["locations"].cuda(),
                   inp["weights"].cuda(), method="softmax" if wl.softmax else None)
    torch.cuda.synchronize()
    ref = oracle.msda_forward(inp["value"], wl.shapes, wl.starts, inp["locations"], inp["weights"],
                              wl.softmax)
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    err = float(np.abs(got - ref).max() / np.abs(ref).max())
    assert err <= TOL[wl.dtype], f"{wl.name}: rel err {err:.3e}"
    return out


@pytest.mark.parametrize("name", sorted(MSDA_WORKLOADS))
def test_msda_workloads(name):
    check(MSDA_WORKLOADS[name])


CASES = [
    MsdaWorkload("msda_f32", 2, 4, 16, ((10, 12), (5, 6)), 37, 4, "f32", True, -0.1, 1.1, 70),
    MsdaWorkload("msda_f16", 1, 8, 32, ((16, 16), (8, 8), (4, 4)), 99, 8, "f16", True, -0.2, 1.2, 71),
    MsdaWorkload("msda_no_softmax", 1, 2, 64, ((9, 7),), 50, 4, "bf16", False, -0.1, 1.1, 72),
    # D not a multiple of 8 / 4: one channel per thread
    MsdaWorkload("msda_d_odd", 2, 3, 6, ((7, 5), (3, 3)), 21, 2, "bf16", True, -0.1, 1.1, 73),
    MsdaWorkload("msda_d_odd_f32", 1, 2, 5, ((6, 6),), 11, 3, "f32", False, -0.1, 1.1, 74),
    # eight lanes per (query, head) sharing eight points; a last warp that the
    # rows fill only in part (15 rows x 4 lanes)
    MsdaWorkload("msda_d64_k8", 1, 4, 64, ((12, 10), (6, 5)), 23, 8, "bf16", True, -0.1, 1.1, 76),
    MsdaWorkload("msda_partial_warp", 1, 3, 32, ((8, 8), (4, 4)), 5, 4, "bf16", True, -0.1, 1.1, 77),
    # five levels, eight points, many samples outside
    MsdaWorkload("msda_5lvl", 1, 4, 32, ((20, 24), (10, 12), (5, 6), (3, 3), (1, 2)), 64, 8, "bf16",
                 True, -0.5, 1.5, 75),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_msda_cases(wl):
    check(wl)


def test_msda_nonfinite_locations_do_not_fault():
    wl = CASES[0]
    inp = make_msda_inputs(wl)
    inp["locations"][0, :5, 0, 0, 0, 0] = float("nan")
    inp["locations"][0, 5:10, 1, 1, 1, 1] = float("inf")
    inp["locations"][1, :5, 2, 0, 2, 0] = -float("inf")
    inp["locations"][1, 5:10, 3, 1, 3, 1] = 3e38
    check(wl, inp)


def test_msda_rejects_too_many_levels():
    wl = MsdaWorkload("msda_9lvl", 1, 1, 8, tuple((2, 2) for _ in range(9)), 3, 1, "f32")
    inp = make_msda_inputs(wl)
    with pytest.raises(dcn.DcnError):
        dcn.msda(inp["value"].cuda(), wl.shapes, wl.starts, inp["locations"].cuda(),
                 inp["weights"].cuda())
