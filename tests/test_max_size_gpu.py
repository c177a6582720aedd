"""The forward at the largest sizes the ABI accepts (GB300).

Every tensor of the problem must hold fewer than 2^31 elements; this one
puts x and out right under that limit: B = 1, C = O = 64, H = W = 5792,
so x and out each hold 2,147,024,896 elements (4.3 GB in bf16), with a
3x3 kernel.  Both kernels run it (the tensor-core path and, forced, the
CUDA-core path), on inputs drawn on the device from a seeded generator.

The oracle cannot take the whole problem, so each sampled output pixel is
checked against the oracle run on a window of x around it: the offsets are
bounded by 3 pixels, so every corner the pixel can reach lies inside the
window, and where the window is cut by the image border it is the image's
own border, so the outside rule is the same.  The pixels are the image
corners, borders, pixels either side of 128-pixel tile seams of the
flattened order, and random ones.  The bar is the bf16 one from TOL.
"""

import numpy as np
import pytest
import torch

import oracle
import deformable_convolution_vision_gb300 as dcn
from deformable_convolution_vision_gb300.inputs import Workload, make_device_inputs
from tests.helpers import TOL, rel_err, sample_points

pytestmark = pytest.mark.gpu

MAX_WL = Workload("max_x_5792", 1, 64, 5792, 5792, 64, 3, 3, 1, "bf16", 3.0, "sigmoid", 0.0, 0.1, 97)
BOUND = 3.0


def _window_reference(d, wl, pts):
    """Oracle value of out[b, :, oh, ow] for each point, from a crop of x."""
    reach = wl.pad + int(BOUND) + 1             # rows / columns a corner can lie from the tap grid
    refs = []
    w_cpu = d["weight"].float().cpu()
    b_cpu = d["bias"].float().cpu()
    for b, oh, ow in pts.tolist():
        r0 = max(0, oh - reach)
        r1 = min(wl.H, oh + wl.kh + reach)
        c0 = max(0, ow - reach)
        c1 = min(wl.W, ow + wl.kw + reach)
        xs = d["x"][b:b + 1, :, r0:r1, c0:c1].float().cpu().contiguous()
        hs, ws = r1 - r0, c1 - c0
        hos, wos = hs + 2 * wl.pad - wl.kh + 1, ws + 2 * wl.pad - wl.kw + 1
        oh_s, ow_s = oh - r0, ow - c0
        assert 0 <= oh_s < hos and 0 <= ow_s < wos
        off = torch.zeros((1, 2 * wl.taps, hos, wos))
        msk = torch.zeros((1, wl.taps, hos, wos))
        off[0, :, oh_s, ow_s] = d["offset"][b, :, oh, ow].cpu()
        msk[0, :, oh_s, ow_s] = d["mask"][b, :, oh, ow].cpu()
        ref = oracle.forward_points(xs, off, msk, w_cpu, b_cpu, wl.pad,
                                    np.array([[0, oh_s, ow_s]], dtype=np.int32))
        refs.append(ref[0])
    return np.stack(refs)


@pytest.fixture(scope="module")
def max_inputs():
    free, _ = torch.cuda.mem_get_info()
    if free < 24 << 30:
        pytest.skip("needs about 20 GB of free device memory")
    d = make_device_inputs(MAX_WL, offset_bound=BOUND)
    assert d["x"].numel() < 2 ** 31 and d["offset"].numel() < 2 ** 31
    pts = sample_points(MAX_WL.B, MAX_WL.Ho, MAX_WL.Wo, 48, seed=MAX_WL.seed)
    # also the middle of every border and a pixel next to each corner
    H, W = MAX_WL.Ho, MAX_WL.Wo
    extra = [(0, 0, W // 2), (0, H - 1, W // 2), (0, H // 2, 0), (0, H // 2, W - 1),
             (0, 1, 1), (0, H - 2, W - 2)]
    pts = np.unique(np.concatenate([pts, np.array(extra, dtype=np.int32)]), axis=0)
    ref = _window_reference(d, MAX_WL, pts)
    yield d, pts, ref
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", [dcn.DCN_PATH_TC, dcn.DCN_PATH_SIMT])
def test_forward_at_the_index_limit(max_inputs, path):
    d, pts, ref = max_inputs
    wl = MAX_WL
    out = torch.empty((wl.B, wl.O, wl.Ho, wl.Wo), dtype=torch.bfloat16, device="cuda",
                      memory_format=torch.channels_last)
    assert out.numel() < 2 ** 31
    with dcn.Handle(path) as h:
        dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=wl.pad,
                          mask=d["mask"], handle=h, out=out)
        assert dcn.dcn_sync_status(h.h) == 0
        assert dcn.dcn_last_path(h.h) == path
    idx = torch.from_numpy(pts).long()
    got = out[idx[:, 0], :, idx[:, 1], idx[:, 2]].float().cpu().numpy()
    del out
    assert np.isfinite(got).all()
    err = rel_err(got, ref)
    assert err <= TOL["bf16"], f"path {path}: rel err {err:.3e} at the index limit"
