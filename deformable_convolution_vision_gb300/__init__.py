"""GB300 (sm_103a) modulated deformable convolution: forward and backward.

torchvision ``deform_conv2d`` semantics -- stride, per-axis padding,
dilation, weight groups and offset groups -- computed by hand-written CUDA
kernels behind the C ABI declared in ``include/dcn.h``.  This package is the
thin Python side: ``binding`` maps the C entry points one to one,
``deform_conv2d`` and ``deform_conv2d_backward`` below shape PyTorch tensors
into one call each, and ``autograd.DeformConv2dFunction`` joins the two for
torch's autograd.
"""

from . import binding
from .binding import (DCN_BF16, DCN_F16, DCN_F32, DCN_PATH_AUTO, DCN_PATH_SIMT, DCN_PATH_TC,
                      DCN_SAMPLE_F32, DCN_SAMPLE_INPUT_DTYPE, ConvDesc, DcnError, dcn_create,
                      dcn_backward, dcn_backward_ex, dcn_destroy, dcn_forward, dcn_forward_ex,
                      dcn_attn_backward, dcn_attn_forward, dcn_msda_backward, dcn_msda_forward, dcn_nchw_to_nhwc,
                      dcn_nhwc_to_nchw,
                      dcn_forward_host,
                      dcn_forward_packed, dcn_forward_packed_ex, dcn_last_path, dcn_out_size,
                      dcn_pack_weight, dcn_pack_weight_ex, dcn_selftest_timeout, dcn_set_path,
                      dcn_set_sample_precision, dcn_status_string, dcn_sync_status)

__all__ = ["binding", "deform_conv2d", "Handle", "DcnError", "DCN_F32", "DCN_BF16", "DCN_F16",
           "DCN_PATH_AUTO", "DCN_PATH_SIMT", "DCN_PATH_TC", "DCN_SAMPLE_INPUT_DTYPE",
           "DCN_SAMPLE_F32", "dcn_set_sample_precision", "dcn_create", "dcn_destroy",
           "dcn_forward", "dcn_forward_host", "dcn_forward_packed", "dcn_pack_weight",
           "dcn_set_path", "dcn_last_path", "dcn_sync_status", "dcn_selftest_timeout",
           "dcn_status_string", "ConvDesc", "dcn_forward_ex", "dcn_pack_weight_ex",
           "dcn_forward_packed_ex", "dcn_out_size", "dcn_backward", "dcn_backward_ex",
           "deform_conv2d_backward", "dcn_msda_forward", "msda", "dcn_msda_backward",
           "msda_backward", "dcn_attn_forward", "attn", "dcn_attn_backward",
           "attn_backward", "dcn_nchw_to_nhwc",
           "dcn_nhwc_to_nchw", "deform_conv2d_nchw"]


class Handle:
    """Owns one ``dcn_handle_t`` (workspace + status word) on the current device."""

    def __init__(self, path=DCN_PATH_AUTO, sample=DCN_SAMPLE_INPUT_DTYPE):
        self.h = dcn_create()
        if path != DCN_PATH_AUTO:
            dcn_set_path(self.h, path)
        if sample != DCN_SAMPLE_INPUT_DTYPE:
            dcn_set_sample_precision(self.h, sample)

    def close(self):
        if self.h is not None:
            dcn_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return DCN_F32
    if t.dtype == torch.bfloat16:
        return DCN_BF16
    if t.dtype == torch.float16:
        return DCN_F16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32, bfloat16 or float16")


def _pair(v, name):
    if isinstance(v, int):
        return (v, v)
    v = tuple(int(t) for t in v)
    if len(v) != 2:
        raise ValueError(f"{name} must be an int or a pair")
    return v


def _on_device_of(name):
    """Run the wrapped entry point with the device of its tensor argument
    ``name`` current: the C library launches on the current device, takes
    the current device's stream by default and refuses a handle made on
    another device, so a tensor on cuda:1 while cuda:0 is current would
    otherwise reach the wrong GPU."""
    import functools
    import inspect

    def wrap(fn):
        sig = inspect.signature(fn)

        @functools.wraps(fn)
        def run(*args, **kwargs):
            import torch
            t = sig.bind_partial(*args, **kwargs).arguments.get(name)
            if isinstance(t, torch.Tensor) and t.is_cuda:
                with torch.cuda.device(t.device):
                    return fn(*args, **kwargs)
            return fn(*args, **kwargs)
        return run
    return wrap


def _check_devices(device, **named):
    """Every given tensor (None is skipped) must live on ``device``: the
    kernels take raw device pointers and cannot tell a host or another
    GPU's pointer from their own."""
    for name, t in named.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} must be on {device}, not {t.device}")


def _check_out(out, shape, dtype, device, channels_last=False):
    """A caller-supplied output must be exactly what the kernel writes: its
    shape, dtype, device and dense layout (a smaller or strided buffer would
    be written out of bounds)."""
    import torch
    fmt = torch.channels_last if channels_last else torch.contiguous_format
    if tuple(out.shape) != tuple(shape) or out.dtype != dtype or out.device != device or \
            not out.is_contiguous(memory_format=fmt):
        layout = "channels_last" if channels_last else "contiguous"
        raise ValueError(f"out must be {tuple(shape)} {dtype} on {device}, {layout}")


def _out_size(n, k, s, p, d):
    span = n + 2 * p - d * (k - 1) - 1
    return span // s + 1 if span >= 0 else 0


def _describe(x, offset, weight, stride, padding, dilation, mask):
    """Check layouts and dtypes (never convert them); the problem's ConvDesc
    and output size."""
    import torch
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    _check_devices(x.device, offset=offset, weight=weight, mask=mask)
    if not x.is_contiguous(memory_format=torch.channels_last):
        raise ValueError("x must be channels_last contiguous")
    for name, t in (("offset", offset), ("weight", weight), ("mask", mask)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if offset.dtype != torch.float32 or (mask is not None and mask.dtype != torch.float32):
        raise TypeError("offset and mask must be float32")
    if weight.dtype != x.dtype:
        raise TypeError("weight must have x's dtype")
    B, C, H, W = x.shape
    O, Cg, kh, kw = weight.shape
    if Cg <= 0 or C % Cg != 0 or O % (C // Cg) != 0:
        raise ValueError("weight's channel count must divide C, and the group count O")
    groups = C // Cg
    (sh, sw), (ph, pw), (dh, dw) = _pair(stride, "stride"), _pair(padding, "padding"), \
        _pair(dilation, "dilation")
    Ho, Wo = _out_size(H, kh, sh, ph, dh), _out_size(W, kw, sw, pw, dw)
    k = kh * kw
    if offset.dim() != 4 or offset.shape[1] % (2 * k) != 0:
        raise ValueError("offset must be [B, 2*G*kh*kw, Ho, Wo]")
    G = offset.shape[1] // (2 * k)
    if G <= 0 or C % G != 0 or tuple(offset.shape) != (B, 2 * G * k, Ho, Wo):
        raise ValueError(f"offset must be {(B, 2 * G * k, Ho, Wo)} with G dividing C")
    if mask is not None and tuple(mask.shape) != (B, G * k, Ho, Wo):
        raise ValueError(f"mask must be {(B, G * k, Ho, Wo)}")
    return ConvDesc(B, C, H, W, O, kh, kw, sh, sw, ph, pw, dh, dw, groups, G), Ho, Wo


@_on_device_of("x")
def deform_conv2d(x, offset, weight, bias=None, stride=1, padding=0, dilation=1, mask=None,
                  handle=None, out=None, stream=None):
    """Modulated deformable convolution forward on CUDA tensors, with
    torchvision ``deform_conv2d``'s argument order.

    x       [B, C, H, W] float32/bfloat16/float16, channels_last memory format
    offset  [B, 2*G*kh*kw, Ho, Wo] float32, contiguous ((dy, dx) per tap,
            offset group after offset group); G = offset groups
    weight  [O, C/groups, kh, kw] same dtype as x, contiguous; groups = C / its dim 1
    bias    [O] float32 or None
    mask    [B, G*kh*kw, Ho, Wo] float32 or None
    stride, padding, dilation: int or (h, w)
    Returns out [B, O, Ho, Wo] in x's dtype, channels_last memory format.
    Layouts are checked, never converted.
    """
    import torch
    if bias is not None and (not bias.is_contiguous() or bias.dtype != torch.float32):
        raise TypeError("bias must be contiguous float32")
    desc, Ho, Wo = _describe(x, offset, weight, stride, padding, dilation, mask)
    if bias is not None:
        _check_devices(x.device, bias=bias)
        if tuple(bias.shape) != (desc.O,):
            raise ValueError(f"bias must be {(desc.O,)}")
    if out is None:
        out = torch.empty((desc.B, desc.O, Ho, Wo), dtype=x.dtype, device=x.device,
                          memory_format=torch.channels_last)
    else:
        _check_out(out, (desc.B, desc.O, Ho, Wo), x.dtype, x.device, channels_last=True)
    own = handle is None
    h = Handle() if own else handle
    try:
        dcn_forward_ex(h.h, x, offset, mask, weight, bias, out, desc, _dtype_code(x), stream)
        if own:
            st = dcn_sync_status(h.h, stream)
            if st != 0:
                raise DcnError(st, "deform_conv2d")
    finally:
        if own:
            h.close()
    return out


@_on_device_of("x")
def deform_conv2d_backward(grad_out, x, offset, weight, stride=1, padding=0, dilation=1,
                           mask=None, bias=True, handle=None, stream=None):
    """Gradients of ``deform_conv2d`` given ``grad_out`` [B, O, Ho, Wo]
    (channels_last, x's dtype).  Returns a dict of fp32 CUDA tensors:
    grad_x [B, C, H, W] (channels_last), grad_offset, grad_mask (None
    without a mask), grad_weight [O, C/groups, kh, kw] and grad_bias [O]
    (None when ``bias`` is False).  Layouts are checked, never converted."""
    import torch
    desc, Ho, Wo = _describe(x, offset, weight, stride, padding, dilation, mask)
    _check_devices(x.device, grad_out=grad_out)
    if tuple(grad_out.shape) != (desc.B, desc.O, Ho, Wo) or grad_out.dtype != x.dtype or \
            not grad_out.is_contiguous(memory_format=torch.channels_last):
        raise ValueError(f"grad_out must be {(desc.B, desc.O, Ho, Wo)} channels_last in x's dtype")
    f32 = dict(dtype=torch.float32, device=x.device)
    gx = torch.empty(x.shape, memory_format=torch.channels_last, **f32)
    goff = torch.empty(offset.shape, **f32)
    gm = None if mask is None else torch.empty(mask.shape, **f32)
    gw = torch.empty(weight.shape, **f32)
    gb = torch.empty((desc.O,), **f32) if bias else None
    own = handle is None
    h = Handle() if own else handle
    try:
        dcn_backward_ex(h.h, x, offset, mask, weight, grad_out, gx, goff, gm, gw, gb, desc,
                        _dtype_code(x), stream)
    finally:
        if own:
            h.close()
    return {"grad_x": gx, "grad_offset": goff, "grad_mask": gm, "grad_weight": gw,
            "grad_bias": gb}


@_on_device_of("value")
def msda(value, shapes, starts, locations, weights, method=None, out=None, stream=None):
    """Multi-scale deformable attention forward (the deformops functional
    form): value [B, S, G, D] (float32/bfloat16/float16, contiguous),
    shapes [L, 2] of (H, W) and starts [L] (any sequence or tensor; read on
    the host), locations [B, Q, G, L, K, 2] float32 normalized (x, y),
    weights [B, Q, G, L*K] float32, method None (weights as given) or
    "softmax".  Returns out [B, Q, G, D] in value's dtype.  Layouts are
    checked, never converted."""
    import torch
    if method not in (None, "softmax"):
        raise ValueError("method must be None or 'softmax'")
    shapes = [tuple(int(v) for v in hw) for hw in (shapes.tolist() if hasattr(shapes, "tolist") else shapes)]
    starts = [int(v) for v in (starts.tolist() if hasattr(starts, "tolist") else starts)]
    if len(shapes) != len(starts):
        raise ValueError("shapes and starts must describe the same levels")
    for name, t in (("value", value), ("locations", locations), ("weights", weights)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if locations.dtype != torch.float32 or weights.dtype != torch.float32:
        raise TypeError("locations and weights must be float32")
    B, S, G, D = value.shape
    Bq, Q, G2, L, K, two = locations.shape
    if (Bq, G2, L, two) != (B, G, len(shapes), 2) or tuple(weights.shape) != (B, Q, G, L * K):
        raise ValueError("locations must be [B, Q, G, L, K, 2] and weights [B, Q, G, L*K]")
    _check_devices(value.device, locations=locations, weights=weights)
    if out is None:
        out = torch.empty((B, Q, G, D), dtype=value.dtype, device=value.device)
    else:
        _check_out(out, (B, Q, G, D), value.dtype, value.device)
    dcn_msda_forward(value, shapes, starts, locations, weights, out, B, S, G, D, Q, K,
                     method == "softmax", _dtype_code(value), stream)
    return out


@_on_device_of("value")
def msda_backward(grad_out, value, shapes, starts, locations, weights, method=None, stream=None):
    """Gradients of ``msda`` for the cotangent grad_out [B, Q, G, D] (value's
    dtype, contiguous): returns (grad_value [B, S, G, D], grad_locations
    [B, Q, G, L, K, 2], grad_weights [B, Q, G, L*K]), all float32 (the
    kernel accumulates them in fp32).  Same argument rules as ``msda``."""
    import torch
    if method not in (None, "softmax"):
        raise ValueError("method must be None or 'softmax'")
    shapes = [tuple(int(v) for v in hw) for hw in (shapes.tolist() if hasattr(shapes, "tolist") else shapes)]
    starts = [int(v) for v in (starts.tolist() if hasattr(starts, "tolist") else starts)]
    if len(shapes) != len(starts):
        raise ValueError("shapes and starts must describe the same levels")
    for name, t in (("value", value), ("locations", locations), ("weights", weights),
                    ("grad_out", grad_out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if locations.dtype != torch.float32 or weights.dtype != torch.float32:
        raise TypeError("locations and weights must be float32")
    if grad_out.dtype != value.dtype:
        raise TypeError("grad_out must have value's dtype")
    B, S, G, D = value.shape
    Bq, Q, G2, L, K, two = locations.shape
    if (Bq, G2, L, two) != (B, G, len(shapes), 2) or tuple(weights.shape) != (B, Q, G, L * K):
        raise ValueError("locations must be [B, Q, G, L, K, 2] and weights [B, Q, G, L*K]")
    if tuple(grad_out.shape) != (B, Q, G, D):
        raise ValueError("grad_out must be [B, Q, G, D]")
    _check_devices(value.device, locations=locations, weights=weights, grad_out=grad_out)
    dev = value.device
    gv = torch.empty((B, S, G, D), dtype=torch.float32, device=dev)
    gl = torch.empty((B, Q, G, L, K, 2), dtype=torch.float32, device=dev)
    gw = torch.empty((B, Q, G, L * K), dtype=torch.float32, device=dev)
    dcn_msda_backward(value, shapes, starts, locations, weights, grad_out, gv, gl, gw,
                      B, S, G, D, Q, K, method == "softmax", _dtype_code(value), stream)
    return gv, gl, gw


@_on_device_of("value")
def attn(value, offsets, weights, kernel_size, stride=1, padding=0, dilation=1, method=None,
         out=None, stream=None):
    """Single-scale deformable sampling (the deformops functional form attn,
    the DCNv3 operator): value [B, H, W, G, D] (float32/bfloat16/float16,
    contiguous channels-last), offsets [B, Ho, Wo, G, K, 2] float32 (dy, dx)
    in pixels, weights [B, Ho, Wo, G, K] float32, method None (weights as
    given) or "softmax" (over the K taps).  kernel_size, stride, padding and
    dilation are ints or (h, w) pairs, with the convolution's meaning.
    Returns out [B, Ho, Wo, G, D] in value's dtype.  Layouts are checked,
    never converted."""
    import torch
    if method not in (None, "softmax"):
        raise ValueError("method must be None or 'softmax'")
    pair = lambda v: (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))  # noqa: E731
    (kh, kw), (sh, sw), (ph, pw), (dh, dw) = (pair(v) for v in (kernel_size, stride, padding, dilation))
    for name, t in (("value", value), ("offsets", offsets), ("weights", weights)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if offsets.dtype != torch.float32 or weights.dtype != torch.float32:
        raise TypeError("offsets and weights must be float32")
    B, H, W, G, D = value.shape
    Ho = dcn_out_size(H, kh, sh, ph, dh)
    Wo = dcn_out_size(W, kw, sw, pw, dw)
    K = kh * kw
    if tuple(offsets.shape) != (B, Ho, Wo, G, K, 2) or tuple(weights.shape) != (B, Ho, Wo, G, K):
        raise ValueError("offsets must be [B, Ho, Wo, G, K, 2] and weights [B, Ho, Wo, G, K]")
    _check_devices(value.device, offsets=offsets, weights=weights)
    if out is None:
        out = torch.empty((B, Ho, Wo, G, D), dtype=value.dtype, device=value.device)
    else:
        _check_out(out, (B, Ho, Wo, G, D), value.dtype, value.device)
    dcn_attn_forward(value, offsets, weights, out, B, H, W, G, D, kh, kw, sh, sw, ph, pw, dh, dw,
                     method == "softmax", _dtype_code(value), stream)
    return out


@_on_device_of("value")
def attn_backward(grad_out, value, offsets, weights, kernel_size, stride=1, padding=0, dilation=1,
                  method=None, stream=None):
    """Gradients of ``attn`` for the cotangent grad_out [B, Ho, Wo, G, D]
    (value's dtype, contiguous): returns (grad_value [B, H, W, G, D],
    grad_offsets [B, Ho, Wo, G, K, 2], grad_weights [B, Ho, Wo, G, K]), all
    float32.  Same argument rules as ``attn``."""
    import torch
    if method not in (None, "softmax"):
        raise ValueError("method must be None or 'softmax'")
    pair = lambda v: (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))  # noqa: E731
    (kh, kw), (sh, sw), (ph, pw), (dh, dw) = (pair(v) for v in (kernel_size, stride, padding, dilation))
    for name, t in (("value", value), ("offsets", offsets), ("weights", weights),
                    ("grad_out", grad_out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if offsets.dtype != torch.float32 or weights.dtype != torch.float32:
        raise TypeError("offsets and weights must be float32")
    if grad_out.dtype != value.dtype:
        raise TypeError("grad_out must have value's dtype")
    B, H, W, G, D = value.shape
    Ho = dcn_out_size(H, kh, sh, ph, dh)
    Wo = dcn_out_size(W, kw, sw, pw, dw)
    K = kh * kw
    if tuple(offsets.shape) != (B, Ho, Wo, G, K, 2) or tuple(weights.shape) != (B, Ho, Wo, G, K):
        raise ValueError("offsets must be [B, Ho, Wo, G, K, 2] and weights [B, Ho, Wo, G, K]")
    if tuple(grad_out.shape) != (B, Ho, Wo, G, D):
        raise ValueError("grad_out must be [B, Ho, Wo, G, D]")
    _check_devices(value.device, offsets=offsets, weights=weights, grad_out=grad_out)
    dev = value.device
    gv = torch.empty((B, H, W, G, D), dtype=torch.float32, device=dev)
    go = torch.empty((B, Ho, Wo, G, K, 2), dtype=torch.float32, device=dev)
    gw = torch.empty((B, Ho, Wo, G, K), dtype=torch.float32, device=dev)
    dcn_attn_backward(value, offsets, weights, grad_out, gv, go, gw, B, H, W, G, D, kh, kw, sh, sw,
                      ph, pw, dh, dw, method == "softmax", _dtype_code(value), stream)
    return gv, go, gw


@_on_device_of("input")
def deform_conv2d_nchw(input, offset, weight, bias=None, stride=1, padding=0, dilation=1,
                       mask=None, handle=None, stream=None):
    """torchvision's argument order and layouts: input [B, C, H, W] and the
    result in plain (contiguous) NCHW.  The library's layout kernels copy
    input to channels-last and the result back; offset, mask and bias stay
    float32 and contiguous as for ``deform_conv2d``."""
    import torch
    if not input.is_cuda or not input.is_contiguous():
        raise ValueError("input must be a contiguous (NCHW) CUDA tensor")
    B, C, H, W = input.shape
    code = _dtype_code(input)
    x = torch.empty((B, C, H, W), dtype=input.dtype, device=input.device,
                    memory_format=torch.channels_last)
    dcn_nchw_to_nhwc(input, x, B, C, H, W, code, stream)
    out_cl = deform_conv2d(x, offset, weight, bias, stride=stride, padding=padding,
                           dilation=dilation, mask=mask, handle=handle, stream=stream)
    Bo, O, Ho, Wo = out_cl.shape
    out = torch.empty((Bo, O, Ho, Wo), dtype=out_cl.dtype, device=out_cl.device)
    dcn_nhwc_to_nchw(out_cl, out, Bo, O, Ho, Wo, code, stream)
    return out
