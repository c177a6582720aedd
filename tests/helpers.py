"""Shared test plumbing: run the CUDA path on seeded inputs and compare it
with the oracle.  Parity metric (the pages print max|diff| beside max|ref|):
err = max|gpu - ref| / max|ref| over the compared outputs.  Alongside it,
every element is held to a bound derived from the path's roundings (see
elementwise_bound), which also sees a wrong small-magnitude element."""

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


# The tensor-core kernel's output tile: 8 rows x 16 columns of one image.
TILE_H, TILE_W = 8, 16


def split_tiles(B, Ho, Wo, nkb, sm_count=152):
    """Tiles (b, tile row, tile column) that the tensor-core kernel's
    persistent stream-K schedule splits between two CTAs: with more tiles
    than SMs every CTA takes an equal run of (tile, K-block) units, and a
    tile is split where a run starts inside it."""
    ty, tx = -(-Ho // TILE_H), -(-Wo // TILE_W)
    tiles = B * ty * tx
    if tiles <= sm_count:
        return []
    units = -(-tiles * nkb // sm_count)
    out = set()
    for start in range(units, tiles * nkb, units):
        if start % nkb:
            t = start // nkb
            out.add((t // (ty * tx), (t % (ty * tx)) // tx, t % tx))
    return sorted(out)


def sample_points(B, Ho, Wo, n, seed=0, nkb=None, sm_count=152):
    """Pixels (b, h, w) to check at full size, aimed at the tensor-core
    kernel's seams: random pixels; every image's corners; both sides of the
    8-row and 16-column tile boundaries along the first, a middle and the
    last rows and columns; the ragged last tile row and column; and, given
    the K-blocks per tile (nkb), the corners and a few inner pixels of tiles
    that the stream-K schedule splits between two CTAs."""
    g = np.random.default_rng(seed)
    pts = set()
    for f in g.integers(0, B * Ho * Wo, size=n).tolist():
        pts.add((f // (Ho * Wo), (f // Wo) % Ho, f % Wo))
    rows = sorted({0, Ho // 2, Ho - 1})
    cols = sorted({0, Wo // 2, Wo - 1})
    hseams = [h for k in range(TILE_H, Ho, TILE_H) for h in (k - 1, k)]
    wseams = [w for k in range(TILE_W, Wo, TILE_W) for w in (k - 1, k)]
    for b in sorted({0, B - 1}):
        for h, w in [(0, 0), (0, Wo - 1), (Ho - 1, 0), (Ho - 1, Wo - 1)]:
            pts.add((b, h, w))
        for h in rows:
            pts.update((b, h, w) for w in wseams[:24] + wseams[-4:])
        for w in cols:
            pts.update((b, h, w) for h in hseams[:24] + hseams[-4:])
        # the ragged last tile row and column (or the last whole ones)
        h_last = (Ho - 1) // TILE_H * TILE_H
        w_last = (Wo - 1) // TILE_W * TILE_W
        pts.update((b, h, w) for h in range(h_last, Ho) for w in (0, Wo // 2, Wo - 1))
        pts.update((b, h, w) for w in range(w_last, Wo) for h in (0, Ho // 2, Ho - 1))
    if nkb is not None:
        for b, ty, tx in split_tiles(B, Ho, Wo, nkb, sm_count)[:64]:
            h0, w0 = ty * TILE_H, tx * TILE_W
            h1, w1 = min(h0 + TILE_H, Ho) - 1, min(w0 + TILE_W, Wo) - 1
            pts.update([(b, h0, w0), (b, h0, w1), (b, h1, w0), (b, h1, w1)])
            for _ in range(2):
                pts.add((b, int(g.integers(h0, h1 + 1)), int(g.integers(w0, w1 + 1))))
    return np.array(sorted(pts), dtype=np.int32)


# unit roundoff of the operand types
UNIT = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -24}


def abs_inputs(inp):
    """The inputs with x, mask and weight replaced by their magnitudes and no
    bias: the oracle on them gives, per output element, the magnitude sum
    sum_k |W_k| * |m_k| * sum_corners w_corner * |x_corner| that bounds every
    rounding error of the path (the corner weights are >= 0)."""
    return {"x": inp["x"].abs(), "offset": inp["offset"],
            "mask": None if inp["mask"] is None else inp["mask"].abs(),
            "weight": inp["weight"].abs(), "bias": None}


def elementwise_bound(absref, ref, dtype, K, sample_f32=False):
    """Per-element error bound of the CUDA path against the oracle.

    16-bit operands: each sampled element is a four-term weighted sum whose
    weights are rounded to the operand type and each of whose fused
    multiply-adds rounds once (the input-dtype combine), so its error is at
    most about 5u times the sum of the corner terms' magnitudes (u the unit
    roundoff); with the fp32 combine it is one rounding, u.  The contraction
    over K = taps * C accumulates in fp32 (at most K + 2 roundings of 2^-24
    on the magnitude sum) and the output is rounded once more (u |out|).
    fp32 operands: the combine and the K-term contraction are fp32 through,
    at most K + 12 roundings of 2^-24 on the magnitude sum.  absref is the
    oracle on abs_inputs, ref the oracle output."""
    u = UNIT[dtype]
    absref = np.asarray(absref, dtype=np.float64)
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    if dtype == "f32":
        return (K + 12) * u * absref + 2 * u * ref + 1e-30
    comb = 1.1 * u if sample_f32 else 6.0 * u
    return (comb + (K + 2) * 2.0 ** -23) * absref + 1.1 * u * ref + 1e-30


def elementwise_ratio(got, ref, bound):
    """max over elements of |got - ref| / bound (must be <= 1)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float((np.abs(got - ref) / bound).max())


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
