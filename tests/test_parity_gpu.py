"""CUDA path vs the oracle on seeded inputs (GB300).

Every output is compared whole, element by element, the five workloads at
full size included (the oracle runs on all host cores; its result is
shared by the two combine precisions).  Two checks on every element set:

- the spec bar: max|gpu - ref| / max|ref| <= 1e-4 for fp32 and
  <= 2e-2 for bf16 operands with fp32 accumulation;
- a per-element bound derived from the path's roundings (tests.helpers.
  elementwise_bound): |gpu - ref| <= c * u * (magnitude sum of the
  element's terms) + 1.1 u |ref|, the magnitude sum from the oracle run on
  |x|, |mask| and |weight|.  It holds for small outputs too, so a wrong
  element of small magnitude fails it where the max-relative bar would not.
"""

import numpy as np
import pytest
import torch

import oracle
from deformable_convolution_vision_gb300 import (DCN_PATH_AUTO, DCN_PATH_SIMT, DCN_PATH_TC,
                                                 DCN_SAMPLE_F32, DCN_SAMPLE_INPUT_DTYPE, Handle,
                                                 dcn_last_path)
from deformable_convolution_vision_gb300.inputs import MAIN, WORKLOADS, Workload, make_inputs
from tests.helpers import (TOL, abs_inputs, compare_full, compare_points, elementwise_bound,
                           elementwise_ratio, oracle_full, run_cuda, sample_points)

pytestmark = pytest.mark.gpu

# whole-output comparison up to this much oracle work (MACs x 4): every
# workload here, the 5x5 boundary one at full size included
FULL_LIMIT = 1.5e11


def _oracle_cost(wl):
    return wl.pixels * wl.O * wl.taps * wl.C * 4


def _run(wl, inp, path, sample):
    with Handle(path, sample) as h:
        out = run_cuda(inp, wl.pad, handle=h)
        taken = dcn_last_path(h.h)
    return out, taken


def check(wl, path=DCN_PATH_AUTO, inp=None, expect_path=None, n_points=256,
          samples=(DCN_SAMPLE_INPUT_DTYPE,), full_limit=FULL_LIMIT):
    """Run the CUDA path in each combine precision of `samples` and compare
    it with the oracle: whole when the oracle's work allows, else on the
    seam-aimed pixels of sample_points."""
    inp = make_inputs(wl) if inp is None else inp
    K = wl.taps * wl.C
    whole = _oracle_cost(wl) <= full_limit
    if whole:
        ref = oracle_full(inp, wl.pad)
        absref = oracle_full(abs_inputs(inp), wl.pad)
    else:
        tiles_k = wl.taps * -(-wl.C // 64)
        pts = sample_points(wl.B, wl.Ho, wl.Wo, n_points, seed=wl.seed, nkb=tiles_k)
        ai = abs_inputs(inp)
        ref = oracle.forward_points(inp["x"], inp["offset"], inp["mask"], inp["weight"],
                                    inp["bias"], wl.pad, pts)
        absref = oracle.forward_points(ai["x"], ai["offset"], ai["mask"], ai["weight"],
                                       None, wl.pad, pts)
    errs = []
    for sample in samples:
        out, taken = _run(wl, inp, path, sample)
        if expect_path is not None:
            assert taken == expect_path, f"{wl.name}: path {taken}, expected {expect_path}"
        if whole:
            err = compare_full(out, ref)
            got = out.float().cpu().numpy()
        else:
            err = compare_points(out, ref, pts)
            got = out.float().cpu()[pts[:, 0], :, pts[:, 1], pts[:, 2]].numpy()
        assert err <= TOL[wl.dtype], f"{wl.name} path {taken}: rel err {err:.3e} > {TOL[wl.dtype]}"
        bound = elementwise_bound(absref, ref, wl.dtype, K,
                                  sample_f32=(sample == DCN_SAMPLE_F32 and taken == DCN_PATH_TC))
        ratio = elementwise_ratio(got, ref, bound)
        assert ratio <= 1.0, f"{wl.name} path {taken}: an element exceeds its error bound by {ratio:.2f}x"
        errs.append(err)
    return max(errs), out


@pytest.mark.parametrize("name", MAIN)
def test_workload(name):
    """The five workloads at full size, whole, in both combine precisions."""
    wl = WORKLOADS[name]
    expect = DCN_PATH_SIMT if wl.dtype == "f32" else DCN_PATH_TC
    check(wl, expect_path=expect, samples=(DCN_SAMPLE_INPUT_DTYPE, DCN_SAMPLE_F32))


@pytest.mark.parametrize("ks", [1, 3, 7])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_page_selftest_shapes(ks, dtype):
    wl = WORKLOADS[f"selftest{ks}x{ks}"].with_(dtype=dtype)
    check(wl, expect_path=DCN_PATH_SIMT if dtype == "f32" else DCN_PATH_TC)


@pytest.mark.parametrize("path", [DCN_PATH_SIMT, DCN_PATH_TC])
def test_both_bf16_paths(path):
    check(WORKLOADS["decoder3x3"], path=path, expect_path=path)


# ragged tile counts, non-square kernels, small maps, no mask / no bias
TC_SHAPES = [
    Workload("tc_ragged_a", 1, 64, 13, 11, 48, 3, 3, 1, "bf16", 2.0, "sigmoid", 0.0, 0.1, 11),
    Workload("tc_ragged_b", 3, 128, 7, 9, 16, 5, 5, 2, "bf16", 3.0, "uniform", 0.0, 0.1, 12),
    Workload("tc_one_tile", 2, 192, 10, 10, 256, 3, 3, 0, "bf16", 1.5, "sigmoid", 0.0, 0.1, 13),
    Workload("tc_one_pixel", 1, 64, 1, 1, 32, 3, 3, 1, "bf16", 0.7, "sigmoid", 0.0, 0.1, 14),
    Workload("tc_no_mask_bias", 1, 64, 40, 37, 64, 7, 7, 3, "bf16", 5.0, "none", 0.0, 0.0, 15),
    Workload("tc_rect_kernel", 1, 64, 12, 20, 64, 3, 5, 2, "bf16", 2.0, "sigmoid", 0.0, 0.1, 16),
    Workload("tc_o_112", 2, 64, 9, 30, 112, 3, 3, 1, "bf16", 2.0, "uniform_zero10", 0.0, 0.1, 17),
    # more 8x16 tiles than a GB300 has SMs: the persistent stream-K schedule,
    # with tiles split between CTAs (one and two channel blocks per tap, and
    # a 5x5 kernel whose CTA runs start in the middle of a group of taps)
    Workload("tc_streamk_3x3", 3, 64, 64, 128, 64, 3, 3, 1, "bf16", 2.0, "sigmoid", 0.0, 0.1, 18),
    Workload("tc_streamk_c128", 2, 128, 64, 160, 32, 3, 3, 1, "bf16", 1.5, "sigmoid", 0.0, 0.1, 19),
    Workload("tc_streamk_5x5", 1, 64, 96, 208, 32, 5, 5, 2, "bf16", 4.0, "uniform_zero10", 0.0, 0.1, 20),
    # one K-block per tile (1x1, C = 64) on the persistent schedule: every
    # segment is one K-block, so one sampler team has nothing to sample in it
    # and the accumulator's reuse rests on the "read out" barrier alone; with
    # O = 64 two accumulators alternate, with O = 256 one is reused
    Workload("tc_streamk_1x1", 2, 64, 64, 160, 64, 1, 1, 0, "bf16", 1.0, "sigmoid", 0.0, 0.1, 21),
    Workload("tc_streamk_1x1_o256", 2, 64, 64, 160, 256, 1, 1, 0, "bf16", 1.0, "sigmoid", 0.0, 0.1, 22),
    # 160 tiles x 9 K-blocks in runs of 10: the run of the ninth CTA starts on
    # a tile's last K-block (a one-K-block tail segment)
    Workload("tc_streamk_tail1", 2, 64, 64, 160, 64, 3, 3, 1, "bf16", 2.0, "uniform", 0.0, 0.1, 23),
]

SIMT_SHAPES = [
    Workload("simt_odd", 2, 3, 9, 7, 5, 3, 3, 1, "f32", 2.0, "sigmoid", 0.0, 0.1, 21),
    Workload("simt_wide", 1, 17, 11, 13, 70, 5, 3, 2, "f32", 3.0, "uniform", 0.0, 0.1, 22),
    Workload("simt_no_mask", 1, 33, 6, 5, 8, 2, 2, 0, "f32", 1.0, "none", 0.0, 0.0, 23),
    Workload("simt_bf16_odd", 2, 24, 10, 9, 40, 3, 3, 1, "bf16", 2.0, "sigmoid", 0.0, 0.1, 24),
    Workload("simt_pad_big", 1, 8, 4, 5, 9, 3, 3, 3, "f32", 1.0, "sigmoid", 0.0, 0.1, 25),
    # a long packed weight row (7 * 7 * 272 fp32 = 53 KB), C not a multiple
    # of the 16-channel step
    Workload("simt_long_row", 1, 272, 7, 6, 8, 7, 7, 3, "f32", 1.5, "sigmoid", 0.0, 0.1, 26),
]


@pytest.mark.parametrize("wl", TC_SHAPES, ids=lambda w: w.name)
def test_tc_shapes(wl):
    check(wl, expect_path=DCN_PATH_TC, samples=(DCN_SAMPLE_INPUT_DTYPE, DCN_SAMPLE_F32))


@pytest.mark.parametrize("wl", SIMT_SHAPES, ids=lambda w: w.name)
def test_simt_shapes(wl):
    check(wl, expect_path=DCN_PATH_SIMT)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_samples_outside_give_bias(dtype):
    wl = WORKLOADS["decoder3x3"].with_(H=32, W=32, dtype=dtype, seed=30)
    inp = make_inputs(wl)
    inp["offset"][:, 0::2] = -(wl.H + 5.0)
    out = run_cuda(inp, wl.pad).float().cpu()
    exp = inp["bias"].to(torch.bfloat16 if dtype == "bf16" else torch.float32).float()
    assert torch.equal(out, exp.view(1, -1, 1, 1).expand_as(out))


def test_mask_zero_gives_bias():
    wl = WORKLOADS["decoder3x3"].with_(H=24, W=40, seed=31)
    inp = make_inputs(wl)
    inp["mask"].zero_()
    out = run_cuda(inp, wl.pad).float().cpu()
    exp = inp["bias"].to(torch.bfloat16).float()
    assert torch.equal(out, exp.view(1, -1, 1, 1).expand_as(out))


def test_nonfinite_offsets_do_not_fault():
    """The pages leave non-finite offsets open; the kernels clamp the sampling
    coordinate, so such taps contribute nothing and nothing is read out of
    bounds."""
    wl = WORKLOADS["decoder3x3"].with_(H=16, W=16, seed=32)
    inp = make_inputs(wl)
    inp["offset"][:, 0, :4] = float("nan")
    inp["offset"][:, 3, 4:8] = float("inf")
    inp["offset"][:, 5, 8:12] = -float("inf")
    inp["offset"][:, 7, 12:] = 3e38
    out = run_cuda(inp, wl.pad)
    ref = oracle_full(inp, wl.pad)
    assert compare_full(out, ref) <= TOL["bf16"]


@pytest.mark.parametrize("name", ["decoder3x3", "tiny"])
def test_deterministic(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    a = run_cuda(inp, wl.pad)
    b = run_cuda(inp, wl.pad)
    assert torch.equal(a, b)


def test_output_guard_bands_untouched():
    """Only the output's own bytes are written: canaries on both sides stay."""
    import deformable_convolution_vision_gb300 as dcn
    from tests.helpers import to_device
    wl = TC_SHAPES[0]
    inp = make_inputs(wl)
    d = to_device(inp)
    n = wl.pixels * wl.O
    guard = 4096
    buf = torch.full((guard + n + guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    out_view = buf[guard:guard + n]
    with Handle() as h:
        dcn.dcn_forward(h.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], out_view,
                        wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, 1)
        assert dcn.dcn_sync_status(h.h) == 0
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + n:] == 7.0)
    out = out_view.view(wl.B, wl.Ho, wl.Wo, wl.O).permute(0, 3, 1, 2)
    assert compare_full(out, oracle_full(inp, wl.pad)) <= TOL["bf16"]
