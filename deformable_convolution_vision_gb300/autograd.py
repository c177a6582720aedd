"""torch.autograd glue: the forward and backward entry points of the C ABI
as one differentiable function.  Argument marshalling only; both passes run
in the library's kernels."""

import torch

from . import attn, attn_backward, deform_conv2d, deform_conv2d_backward, msda, msda_backward


class DeformConv2dFunction(torch.autograd.Function):
    """out = deform_conv2d(x, offset, weight, bias, stride, padding,
    dilation, mask); gradients for x, offset, mask, weight and bias, each
    returned in its input's dtype (the kernels compute them in fp32)."""

    @staticmethod
    def forward(ctx, x, offset, mask, weight, bias, stride=1, padding=0, dilation=1):
        out = deform_conv2d(x, offset, weight, bias, stride=stride, padding=padding,
                            dilation=dilation, mask=mask)
        ctx.save_for_backward(x, offset, mask, weight)
        ctx.conv = (stride, padding, dilation)
        ctx.has_bias = bias is not None
        return out

    @staticmethod
    def backward(ctx, grad_out):
        x, offset, mask, weight = ctx.saved_tensors
        stride, padding, dilation = ctx.conv
        g = grad_out.to(x.dtype).contiguous(memory_format=torch.channels_last)
        r = deform_conv2d_backward(g, x, offset, weight, stride=stride, padding=padding,
                                   dilation=dilation, mask=mask, bias=ctx.has_bias)
        gm = None if mask is None else r["grad_mask"]
        gb = r["grad_bias"] if ctx.has_bias else None
        return (r["grad_x"].to(x.dtype), r["grad_offset"], gm, r["grad_weight"].to(weight.dtype),
                gb, None, None, None)


def deform_conv2d_autograd(x, offset, weight, bias=None, stride=1, padding=0, dilation=1,
                           mask=None):
    """deform_conv2d that records the graph for torch.autograd."""
    return DeformConv2dFunction.apply(x, offset, mask, weight, bias, stride, padding, dilation)


class MsdaFunction(torch.autograd.Function):
    """out = msda(value, shapes, starts, locations, weights, method);
    gradients for value (in its dtype), locations and weights (float32)."""

    @staticmethod
    def forward(ctx, value, locations, weights, shapes, starts, method=None):
        out = msda(value, shapes, starts, locations, weights, method=method)
        ctx.save_for_backward(value, locations, weights)
        ctx.meta = (shapes, starts, method)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        value, locations, weights = ctx.saved_tensors
        shapes, starts, method = ctx.meta
        gv, gl, gw = msda_backward(grad_out.to(value.dtype).contiguous(), value, shapes, starts,
                                   locations, weights, method=method)
        return gv.to(value.dtype), gl, gw, None, None, None


def msda_autograd(value, shapes, starts, locations, weights, method=None):
    """msda that records the graph for torch.autograd."""
    return MsdaFunction.apply(value, locations, weights, shapes, starts, method)


class AttnFunction(torch.autograd.Function):
    """out = attn(value, offsets, weights, kernel_size, stride, padding,
    dilation, method); gradients for value (in its dtype), offsets and
    weights (float32)."""

    @staticmethod
    def forward(ctx, value, offsets, weights, kernel_size, stride=1, padding=0, dilation=1,
                method=None):
        out = attn(value, offsets, weights, kernel_size, stride, padding, dilation, method=method)
        ctx.save_for_backward(value, offsets, weights)
        ctx.meta = (kernel_size, stride, padding, dilation, method)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        value, offsets, weights = ctx.saved_tensors
        kernel_size, stride, padding, dilation, method = ctx.meta
        gv, go, gw = attn_backward(grad_out.to(value.dtype).contiguous(), value, offsets, weights,
                                   kernel_size, stride, padding, dilation, method=method)
        return gv.to(value.dtype), go, gw, None, None, None, None, None


def attn_autograd(value, offsets, weights, kernel_size, stride=1, padding=0, dilation=1,
                  method=None):
    """attn that records the graph for torch.autograd."""
    return AttnFunction.apply(value, offsets, weights, kernel_size, stride, padding, dilation,
                              method)
