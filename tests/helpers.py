"""Shared test plumbing: run the CUDA path on seeded inputs and compare it
with the oracle.  Parity metric (the pages print max|diff| beside max|ref|):
err = max|gpu - ref| / max|ref| over the compared outputs."""

import numpy as np
import torch

# fp32 and bf16: the spec bars.  fp16 keeps the bf16 bar's form but
# scales it by the ratio of unit roundoffs, 2^-11 / 2^-8 = 1/8 (every
# rounding on the path -- corner weights, combine, sample, output -- is one
# unit roundoff of the operand type), with a factor 2 of margin: 2e-2 / 4.
TOL = {"f32": 1e-4, "bf16": 2e-2, "f16": 5e-3}


def to_device(inp, device="cuda"):
    """Inputs dict (CPU, logical NCHW) -> device tensors in the ABI layouts."""
    d = {}
    d["x"] = inp["x"].to(device).contiguous(memory_format=torch.channels_last)
    d["offset"] = inp["offset"].to(device).contiguous()
    d["mask"] = None if inp["mask"] is None else inp["mask"].to(device).contiguous()
    d["weight"] = inp["weight"].to(device).contiguous()
    d["bias"] = None if inp["bias"] is None else inp["bias"].to(device).contiguous()
    return d


def run_cuda(inp, pad, handle=None):
    import deformable_convolution_vision_gb300 as dcn
    d = to_device(inp)
    out = dcn.deform_conv2d(d["x"], d["offset"], d["weight"], d["bias"], padding=pad,
                            mask=d["mask"], handle=handle)
    if handle is not None:
        st = dcn.dcn_sync_status(handle.h)
        assert st == 0, f"device status {dcn.dcn_status_string(st)}"
    return out


def oracle_full(inp, pad):
    import oracle
    return oracle.forward(inp["x"], inp["offset"], inp["mask"], inp["weight"], inp["bias"], pad)


def sample_points(B, Ho, Wo, n, seed=0, tile=128):
    """Pixels (b, h, w) to check at full size: random ones plus the first and
    last pixel, image corners and both sides of several 128-pixel tile
    boundaries in the flattened (b, h, w) order."""
    P = B * Ho * Wo
    g = np.random.default_rng(seed)
    flat = set(g.integers(0, P, size=n).tolist())
    flat.update([0, P - 1])
    for t in range(1, min(P // tile, 6) + 1):
        flat.update([t * tile - 1, min(t * tile, P - 1)])
    for b in range(B):
        for h, w in [(0, 0), (0, Wo - 1), (Ho - 1, 0), (Ho - 1, Wo - 1)]:
            flat.add((b * Ho + h) * Wo + w)
    flat = np.array(sorted(flat))
    b = flat // (Ho * Wo)
    r = flat % (Ho * Wo)
    return np.stack([b, r // Wo, r % Wo], axis=1).astype(np.int32)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def compare_full(out, ref):
    """out: CUDA [B,O,Ho,Wo]; ref: numpy fp64 [B,O,Ho,Wo]."""
    got = out.float().cpu().numpy()
    assert got.shape == ref.shape
    assert np.isfinite(got).all()
    return rel_err(got, ref)


def compare_points(out, ref_pts, pts):
    """out: CUDA [B,O,Ho,Wo]; ref_pts: [n,O] fp64 at pts [n,3]."""
    o = out.float().cpu()
    got = o[pts[:, 0], :, pts[:, 1], pts[:, 2]].numpy()
    assert np.isfinite(got).all()
    return rel_err(got, ref_pts)
