"""Seeded synthetic inputs for the deformable convolution workloads.

This module draws random tensors and nothing else: it holds none of the
operator's arithmetic, so the CUDA path and the oracle can both be fed from
it without sharing any of the method.

Shapes and value distributions are those of the five workloads the library
is measured on (a tiny fp32 case, a decoder 3x3, the BiRefNet-style ASPP 7x7
at 256x256 that the "birefnet-lite-1024-webgpu patch_deform.py" page sizes
at 392 MB of gathered fp16, a batched backbone 3x3 and a non-square 5x5
boundary case), plus the three kernel sizes of the self-test on the page
"litert-community/Idol ... deform_conv.py" (x [1,64,33,40] ~ N(0,1),
offsets N(0,1)*4, mask U(0,2), weight N(0,1)*0.05, no bias).

Every tensor is generated in logical NCHW / OIHW order in fp32 on the CPU,
then x and weight are rounded to the compute dtype.  Offsets, mask and bias
stay fp32.
"""

from dataclasses import dataclass, replace

import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    C: int
    H: int
    W: int
    O: int
    kh: int
    kw: int
    pad: int
    dtype: str            # "f32", "bf16" or "f16": dtype of x, weight and out
    offset_std: float
    mask: str             # "sigmoid", "uniform", "uniform_zero10", "uniform2", "none"
    weight_std: float     # 0 -> 1/sqrt(kh*kw*C)
    bias_std: float       # 0 -> no bias
    seed: int

    @property
    def Ho(self):
        return self.H + 2 * self.pad - self.kh + 1

    @property
    def Wo(self):
        return self.W + 2 * self.pad - self.kw + 1

    @property
    def taps(self):
        return self.kh * self.kw

    @property
    def pixels(self):
        """Output pixels P = B * Ho * Wo."""
        return self.B * self.Ho * self.Wo

    @property
    def flops(self):
        """Effective FLOPs of the contraction, 2 * B*Ho*Wo * O * kh*kw * C."""
        return 2 * self.pixels * self.O * self.taps * self.C

    def with_(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 1, 4, 8, 8, 3, 3, 3, 1, "f32", 1.5, "sigmoid", 0.0, 0.1, 0),
        Workload("decoder3x3", 1, 64, 128, 128, 64, 3, 3, 1, "bf16", 2.0, "sigmoid", 0.0, 0.1, 1),
        Workload("aspp7x7", 1, 64, 256, 256, 64, 7, 7, 3, "bf16", 3.0, "sigmoid", 0.0, 0.1, 2),
        Workload("backbone3x3", 8, 256, 64, 64, 256, 3, 3, 1, "bf16", 1.0, "sigmoid", 0.0, 0.1, 3),
        Workload("boundary5x5", 2, 128, 160, 224, 128, 5, 5, 2, "bf16", 8.0, "uniform_zero10", 0.0, 0.1, 4),
        # the page's self-test shapes (ks, pad) = (1, 0), (3, 1), (7, 3)
        Workload("selftest1x1", 1, 64, 33, 40, 256, 1, 1, 0, "f32", 4.0, "uniform2", 0.05, 0.0, 0),
        Workload("selftest3x3", 1, 64, 33, 40, 256, 3, 3, 1, "f32", 4.0, "uniform2", 0.05, 0.0, 0),
        Workload("selftest7x7", 1, 64, 33, 40, 256, 7, 7, 3, "f32", 4.0, "uniform2", 0.05, 0.0, 0),
    ]
}

# The five measured workloads, in order.
MAIN = ["tiny", "decoder3x3", "aspp7x7", "backbone3x3", "boundary5x5"]

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def make_inputs(wl: Workload, seed=None):
    """Return a dict of CPU tensors for workload ``wl``.

    x [B,C,H,W] and weight [O,C,kh,kw] are in the compute dtype;
    offset [B,2*kh*kw,Ho,Wo], mask [B,kh*kw,Ho,Wo] (or None) and bias [O]
    (or None) are fp32.
    """
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    k = wl.taps
    x = torch.randn(wl.B, wl.C, wl.H, wl.W, generator=g)
    offset = torch.randn(wl.B, 2 * k, wl.Ho, wl.Wo, generator=g) * wl.offset_std
    if wl.mask == "sigmoid":
        mask = torch.sigmoid(torch.randn(wl.B, k, wl.Ho, wl.Wo, generator=g))
    elif wl.mask == "uniform":
        mask = torch.rand(wl.B, k, wl.Ho, wl.Wo, generator=g)
    elif wl.mask == "uniform2":
        mask = torch.rand(wl.B, k, wl.Ho, wl.Wo, generator=g) * 2
    elif wl.mask == "uniform_zero10":
        mask = torch.rand(wl.B, k, wl.Ho, wl.Wo, generator=g)
        drop = torch.rand(wl.B, k, wl.Ho, wl.Wo, generator=g) < 0.1
        mask = torch.where(drop, torch.zeros_like(mask), mask)
    elif wl.mask == "none":
        mask = None
    else:
        raise ValueError(f"unknown mask kind {wl.mask!r}")
    wstd = wl.weight_std if wl.weight_std > 0 else 1.0 / (k * wl.C) ** 0.5
    weight = torch.randn(wl.O, wl.C, wl.kh, wl.kw, generator=g) * wstd
    bias = torch.randn(wl.O, generator=g) * wl.bias_std if wl.bias_std > 0 else None
    dt = TORCH_DTYPE[wl.dtype]
    return {
        "x": x.to(dt),
        "offset": offset.float().contiguous(),
        "mask": None if mask is None else mask.float().contiguous(),
        "weight": weight.to(dt),
        "bias": None if bias is None else bias.float().contiguous(),
    }


@dataclass(frozen=True)
class GeneralWorkload:
    """A problem of the general form: stride, per-axis padding, dilation,
    weight groups and offset groups.  Inputs follow make_inputs' recipe
    (x ~ N(0,1), offsets ~ N(0, offset_std), sigmoid mask, weight std
    1/sqrt(kh*kw*C/groups), bias ~ N(0, 0.1)); offsets and mask carry one
    block of planes per offset group."""
    name: str
    B: int
    C: int
    H: int
    W: int
    O: int
    kh: int
    kw: int
    stride: tuple = (1, 1)
    padding: tuple = (0, 0)
    dilation: tuple = (1, 1)
    groups: int = 1
    offset_groups: int = 1
    dtype: str = "bf16"
    offset_std: float = 2.0
    mask: bool = True
    seed: int = 0

    def out_size(self):
        def one(n, k, s, p, d):
            span = n + 2 * p - d * (k - 1) - 1
            return span // s + 1 if span >= 0 else 0
        return (one(self.H, self.kh, self.stride[0], self.padding[0], self.dilation[0]),
                one(self.W, self.kw, self.stride[1], self.padding[1], self.dilation[1]))


def make_general_inputs(wl: GeneralWorkload):
    """CPU tensors for a GeneralWorkload (layouts as make_inputs, with
    weight [O, C/groups, kh, kw], offset [B, 2*G*kh*kw, Ho, Wo] and mask
    [B, G*kh*kw, Ho, Wo], G = offset_groups)."""
    g = torch.Generator().manual_seed(wl.seed)
    Ho, Wo = wl.out_size()
    k, G = wl.kh * wl.kw, wl.offset_groups
    Cg = wl.C // wl.groups
    x = torch.randn(wl.B, wl.C, wl.H, wl.W, generator=g)
    offset = torch.randn(wl.B, 2 * G * k, Ho, Wo, generator=g) * wl.offset_std
    mask = torch.sigmoid(torch.randn(wl.B, G * k, Ho, Wo, generator=g)) if wl.mask else None
    weight = torch.randn(wl.O, Cg, wl.kh, wl.kw, generator=g) / (k * Cg) ** 0.5
    bias = torch.randn(wl.O, generator=g) * 0.1
    dt = TORCH_DTYPE[wl.dtype]
    return {
        "x": x.to(dt),
        "offset": offset.contiguous(),
        "mask": None if mask is None else mask.contiguous(),
        "weight": weight.to(dt),
        "bias": bias.contiguous(),
    }


@dataclass(frozen=True)
class MsdaWorkload:
    """Multi-scale deformable attention (the deformops page's functional
    form): value [B, S, G, D] ~ N(0, 1) in the compute dtype, locations
    [B, Q, G, L, K, 2] ~ U(lo, hi) (normalized; beyond [0, 1] some corners
    fall outside), weights [B, Q, G, L*K] ~ U(0, 1) raw logits (softmax
    applied in the operator when `softmax`)."""
    name: str
    B: int
    G: int
    D: int
    shapes: tuple          # ((H, W), ...) per level
    Q: int
    K: int
    dtype: str = "bf16"
    softmax: bool = True
    loc_lo: float = 0.0
    loc_hi: float = 1.0
    seed: int = 0

    @property
    def starts(self):
        out, s = [], 0
        for h, w in self.shapes:
            out.append(s)
            s += h * w
        return out

    @property
    def S(self):
        return sum(h * w for h, w in self.shapes)

    @property
    def L(self):
        return len(self.shapes)


def make_msda_inputs(wl: MsdaWorkload):
    g = torch.Generator().manual_seed(wl.seed)
    value = torch.randn(wl.B, wl.S, wl.G, wl.D, generator=g)
    loc = torch.rand(wl.B, wl.Q, wl.G, wl.L, wl.K, 2, generator=g) * (wl.loc_hi - wl.loc_lo) + wl.loc_lo
    weights = torch.rand(wl.B, wl.Q, wl.G, wl.L * wl.K, generator=g)
    return {"value": value.to(TORCH_DTYPE[wl.dtype]), "locations": loc.contiguous(),
            "weights": weights.contiguous()}


def make_device_inputs(wl: Workload, device="cuda", offset_bound=3.0):
    """Inputs for problems too large to build on the host, drawn on the
    device from a seeded device generator: x ~ N(0, 1) in the compute dtype
    (channels-last), offsets ~ U(-offset_bound, offset_bound) (bounded, so
    that the corners a pixel reaches lie within a small window of it),
    sigmoid mask of N(0, 1), weight ~ N(0, 1/(kh*kw*C)), bias ~ N(0, 0.1),
    all in the ABI layouts."""
    g = torch.Generator(device=device).manual_seed(wl.seed)
    dt = TORCH_DTYPE[wl.dtype]
    x = torch.empty((wl.B, wl.C, wl.H, wl.W), dtype=dt, device=device,
                    memory_format=torch.channels_last)
    # fill in slabs of rows so that no fp32 temporary of x's size exists
    for h0 in range(0, wl.H, 256):
        h1 = min(wl.H, h0 + 256)
        x[:, :, h0:h1] = torch.randn((wl.B, wl.C, h1 - h0, wl.W), generator=g, device=device).to(dt)
    off = (torch.rand((wl.B, 2 * wl.taps, wl.Ho, wl.Wo), generator=g, device=device) * 2.0 - 1.0)
    off.mul_(offset_bound)
    mask = torch.sigmoid(torch.randn((wl.B, wl.taps, wl.Ho, wl.Wo), generator=g, device=device))
    weight = (torch.randn((wl.O, wl.C, wl.kh, wl.kw), generator=g, device=device)
              / math.sqrt(wl.taps * wl.C)).to(dt)
    bias = torch.randn(wl.O, generator=g, device=device) * 0.1
    return {"x": x, "offset": off, "mask": mask, "weight": weight, "bias": bias}


def make_msda_grad_out(wl: MsdaWorkload):
    """A cotangent for the backward: grad_out [B, Q, G, D] ~ N(0, 1) in the
    compute dtype, from its own seed (the workload's + 1000)."""
    g = torch.Generator().manual_seed(wl.seed + 1000)
    return torch.randn(wl.B, wl.Q, wl.G, wl.D, generator=g).to(TORCH_DTYPE[wl.dtype])


@dataclass(frozen=True)
class AttnWorkload:
    """Single-scale deformable sampling (the deformops page's attn, the DCNv3
    operator): value [B, H, W, G, D] ~ N(0, 1) in the compute dtype,
    offsets [B, Ho, Wo, G, K, 2] ~ N(0, offset_std) pixels (dy, dx), weights
    [B, Ho, Wo, G, K] ~ U(0, 1) raw logits (softmax applied in the operator
    when `softmax`)."""
    name: str
    B: int
    H: int
    W: int
    G: int
    D: int
    kernel: tuple = (3, 3)
    stride: tuple = (1, 1)
    padding: tuple = (1, 1)
    dilation: tuple = (1, 1)
    dtype: str = "bf16"
    softmax: bool = True
    offset_std: float = 2.0
    seed: int = 0

    def out_size(self):
        def one(n, k, s, p, d):
            return (n + 2 * p - d * (k - 1) - 1) // s + 1
        return (one(self.H, self.kernel[0], self.stride[0], self.padding[0], self.dilation[0]),
                one(self.W, self.kernel[1], self.stride[1], self.padding[1], self.dilation[1]))

    @property
    def K(self):
        return self.kernel[0] * self.kernel[1]


def make_attn_inputs(wl: AttnWorkload):
    g = torch.Generator().manual_seed(wl.seed)
    Ho, Wo = wl.out_size()
    value = torch.randn(wl.B, wl.H, wl.W, wl.G, wl.D, generator=g)
    off = torch.randn(wl.B, Ho, Wo, wl.G, wl.K, 2, generator=g) * wl.offset_std
    weights = torch.rand(wl.B, Ho, Wo, wl.G, wl.K, generator=g)
    return {"value": value.to(TORCH_DTYPE[wl.dtype]), "offsets": off.contiguous(),
            "weights": weights.contiguous()}


def make_attn_grad_out(wl: AttnWorkload):
    """A cotangent for the backward: grad_out [B, Ho, Wo, G, D] ~ N(0, 1) in
    the compute dtype, from its own seed (the workload's + 1000)."""
    g = torch.Generator().manual_seed(wl.seed + 1000)
    Ho, Wo = wl.out_size()
    return torch.randn(wl.B, Ho, Wo, wl.G, wl.D, generator=g).to(TORCH_DTYPE[wl.dtype])


ATTN_WORKLOADS = {
    w.name: w for w in [
        # the page's layer example: DeformSample2d(dim=64, kernel_size=3,
        # groups=4) on a 32 x 32 map
        AttnWorkload("attn_page", 1, 32, 32, 4, 16, seed=90),
        # a DCNv3 layer at the first stage of an InternImage-scale backbone on
        # a 1024 x 1024 image (256 x 256 map, 112 channels in 7 groups of 16),
        # two images
        AttnWorkload("attn_stage1_1024", 2, 256, 256, 7, 16, seed=91),
    ]
}


_PAGE_LEVELS = ((64, 64), (32, 32), (16, 16), (8, 8))
MSDA_WORKLOADS = {
    w.name: w for w in [
        # the page's layer example: 300 queries over four levels
        MsdaWorkload("msda_page", 1, 8, 32, _PAGE_LEVELS, 300, 4, seed=60),
        # encoder scale: every pixel of the four levels is a query (5440)
        MsdaWorkload("msda_encoder", 1, 8, 32, _PAGE_LEVELS, 5440, 4, seed=61),
        # the upper end of the page's 5k-22k queries per call
        MsdaWorkload("msda_encoder_22k", 1, 8, 32, ((128, 128), (64, 64), (32, 32), (16, 16)),
                     21760, 4, seed=62),
    ]
}
