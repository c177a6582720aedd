"""Invariants of the forward on the GPU that hold whatever the oracle says.

- Mask linearity, exactly: with no bias, scaling the mask by 1/2 halves
  every output bit for bit.  A power-of-two scale commutes with every
  rounding on the path (the corner weights rounded to the operand type,
  the 16-bit combine, the fp32 accumulation, the final rounding) as long
  as nothing reaches the subnormal range: so bf16 and fp32, whose exponent
  range is fp32's, and not fp16, whose small corner-weight products would.
- Batch splitting: a batch gives the same output as its images one by
  one.  With every tile computed by one CTA (no more (tile, K-block)
  units than SMs, so no split schedule) the order of every sum is the
  same, so the bits are equal; when the persistent schedule splits tiles
  between CTAs at other places, the
  partial sums meet in another order: the fp32 sum moves by a few units
  of fp32 roundoff of the sum of its terms' magnitudes, which the output
  rounding can turn into one unit in the last place of the output type,
  plus that absolute amount where the output is near zero (a result of
  cancellation).
"""

import pytest
import torch

import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300 import DCN_PATH_SIMT, DCN_PATH_TC, Handle
from deformable_convolution_vision_gb300.inputs import Workload, make_inputs
from tests.helpers import to_device

pytestmark = pytest.mark.gpu


def _forward(d, wl, path, mask=None, bias=None):
    with Handle(path) as h:
        out = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], bias, padding=wl.pad,
                                mask=d["mask"] if mask is None else mask, handle=h)
        assert dcn.dcn_sync_status(h.h) == 0
        assert dcn.dcn_last_path(h.h) == path
    return out


@pytest.mark.parametrize("path,dtype", [(DCN_PATH_TC, "bf16"), (DCN_PATH_SIMT, "bf16"),
                                        (DCN_PATH_SIMT, "f32")])
def test_mask_linearity_is_exact(path, dtype):
    wl = Workload("inv_mask", 2, 64, 40, 56, 64, 3, 3, 1, dtype, 2.0, "uniform", 0.0, 0.0, 130)
    d = to_device(make_inputs(wl))
    full = _forward(d, wl, path)
    half = _forward(d, wl, path, mask=d["mask"] * 0.5)
    assert torch.equal(half, full * 0.5)


@pytest.mark.parametrize("wl", [
    # 3 x 2 x 2 = 12 tiles x 9 K-blocks: one CTA per tile, the same sums in
    # the same order
    Workload("inv_batch_small", 3, 64, 16, 30, 64, 3, 3, 1, "bf16", 2.0, "sigmoid", 0.0, 0.1, 131),
    # 2 x 16 x 10 = 320 tiles: the persistent schedule splits tiles
    Workload("inv_batch_streamk", 2, 128, 128, 160, 32, 5, 5, 2, "bf16", 3.0, "sigmoid", 0.0, 0.1, 132),
], ids=lambda w: w.name)
def test_batch_split(wl):
    inp = make_inputs(wl)
    d = to_device(inp)
    whole = _forward(d, wl, DCN_PATH_TC, bias=d["bias"])
    parts = []
    for b in range(wl.B):
        db = {"x": d["x"][b:b + 1].contiguous(memory_format=torch.channels_last),
              "offset": d["offset"][b:b + 1].contiguous(),
              "mask": d["mask"][b:b + 1].contiguous(), "weight": d["weight"]}
        parts.append(_forward(db, wl.with_(B=1), DCN_PATH_TC, bias=d["bias"]))
    split = torch.cat(parts, 0)
    tiles = wl.B * ((wl.Ho + 7) // 8) * ((wl.Wo + 15) // 16)
    units = tiles * wl.taps * ((wl.C + 63) // 64)
    if units <= torch.cuda.get_device_properties(0).multi_processor_count:
        assert torch.equal(whole, split)
    else:
        a, b = whole.float(), split.float()
        # one bf16 unit in the last place at each element's magnitude, plus
        # the fp32 reordering: K = 3200 products of magnitude <~ 1 per output
        # give sums of magnitudes <~ 100, whose fp32 roundoff is ~1e-5
        ulp = torch.maximum(a.abs(), b.abs()) * 2.0 ** -7
        diff = (a - b).abs()
        assert bool((diff <= ulp + 1e-4).all()), f"max excess {float((diff - ulp).max()):.3e}"
        assert float((diff > ulp).float().mean()) < 1e-3
