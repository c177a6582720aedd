"""Oracle for the modulated deformable convolution forward pass and its
gradients.

TEST INFRASTRUCTURE ONLY.  The plain C definition in ``dcn_oracle.c`` is
what the CUDA path is checked against.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package; the product library never loads it, and it shares no code with the
CUDA sources.

The arithmetic follows the page "litert-community/Idol ... deform_conv.py"
(module docstring and the four-corner loop of ``deform_conv2d_gather``):
bilinear samples at (h - pad + i + dy_k, w - pad + j + dx_k), corners
outside the image count as 0, each sample scaled by mask_k, contracted over
(tap, channel) with the weight, plus bias.  Accumulation is fp64; the
sampling coordinate is fp32 (the page builds its grid in the input dtype,
fp32 for the fp32 offsets).

All arrays cross this boundary in logical NCHW order:
x [B,C,H,W] fp32, offset [B,2k,Ho,Wo] fp32, mask [B,k,Ho,Wo] fp32 or None,
weight [O,C,kh,kw] fp32, bias [O] fp32 or None; results are fp64.  The
general form (``forward_ex``) adds stride, per-axis padding, dilation,
weight groups and offset groups (``ConvDesc``): offset
[B,2*G*k,Ho,Wo], mask [B,G*k,Ho,Wo], weight [O,C/groups,kh,kw].
"""

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "dcn_oracle.c")
LIBRARY = os.path.join(_HERE, "libdcn_oracle.so")

# -ffp-contract=off: no fused multiply-add, so x86 and Arm hosts give the
# same bits.  No -ffast-math: floor, comparisons and NaN must follow IEEE.
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


MSDA_SOURCE = os.path.join(_HERE, "msda_oracle.c")
ATTN_SOURCE = os.path.join(_HERE, "attn_oracle.c")


def compile_oracle(source=SOURCE, output=LIBRARY, extra=(MSDA_SOURCE, ATTN_SOURCE)):
    """Compile the oracle's C sources into a shared library (gcc)."""
    cmd = ["gcc", *CFLAGS, source, *extra, "-o", output, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def _stale(source, output):
    if not os.path.exists(output):
        return True
    built = os.path.getmtime(output)
    return any(os.path.getmtime(s) > built for s in (source, MSDA_SOURCE, ATTN_SOURCE))


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path=LIBRARY, source=SOURCE):
        if path == LIBRARY and _stale(source, path):
            compile_oracle(source, path)
        self.path = path
        lib = ctypes.CDLL(path)
        f = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_dcn_forward.argtypes = [f, f, f, f, f, f] + [i] * 9
        lib.oracle_dcn_forward.restype = i
        lib.oracle_dcn_forward_points.argtypes = [f, f, f, f, f, f, i, f] + [i] * 9
        lib.oracle_dcn_forward_points.restype = i
        lib.oracle_dcn_forward_ex.argtypes = [f, f, f, f, f, f, f, i]
        lib.oracle_dcn_forward_ex.restype = i
        lib.oracle_dcn_forward_points_ex.argtypes = [f, f, f, f, f, f, i, f, f, i]
        lib.oracle_dcn_forward_points_ex.restype = i
        lib.oracle_dcn_backward_ex.argtypes = [f] * 10 + [f, i]
        lib.oracle_dcn_backward_ex.restype = i
        lib.oracle_dcn_backward_points_ex.argtypes = [f] * 5 + [f, i, f, f, f, i]
        lib.oracle_dcn_backward_points_ex.restype = i
        if hasattr(lib, "oracle_msda_forward"):
            lib.oracle_msda_forward.argtypes = [f, f, f, i, f, f, i, f] + [i] * 7
            lib.oracle_msda_forward.restype = i
        if hasattr(lib, "oracle_attn_forward"):
            lib.oracle_attn_forward.argtypes = [f, f, f, i, f] + [i] * 14
            lib.oracle_attn_forward.restype = i
        if hasattr(lib, "oracle_attn_backward"):
            lib.oracle_attn_backward.argtypes = [f, f, f, i, f, f, f, f] + [i] * 14
            lib.oracle_attn_backward.restype = i
        if hasattr(lib, "oracle_msda_backward"):
            lib.oracle_msda_backward.argtypes = [f, f, f, i, f, f, i, f, f, f, f] + [i] * 7
            lib.oracle_msda_backward.restype = i
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i
        self._lib = lib

    def max_threads(self):
        return int(self._lib.oracle_max_threads())

    @staticmethod
    def _f32(a):
        if a is None:
            return None
        if hasattr(a, "detach"):  # torch tensor
            a = a.detach().to("cpu").float().numpy()
        return np.ascontiguousarray(a, dtype=np.float32)

    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    def _prepare(self, x, offset, mask, weight, bias, pad):
        x, offset, mask, weight, bias = (self._f32(t) for t in (x, offset, mask, weight, bias))
        B, C, H, W = x.shape
        O, C2, kh, kw = weight.shape
        if C2 != C:
            raise ValueError("weight channel count does not match x")
        Ho, Wo = H + 2 * pad - kh + 1, W + 2 * pad - kw + 1
        if offset.shape != (B, 2 * kh * kw, Ho, Wo):
            raise ValueError(f"offset shape {offset.shape} != {(B, 2 * kh * kw, Ho, Wo)}")
        if mask is not None and mask.shape != (B, kh * kw, Ho, Wo):
            raise ValueError(f"mask shape {mask.shape} != {(B, kh * kw, Ho, Wo)}")
        if bias is not None and bias.shape != (O,):
            raise ValueError("bias must have shape [O]")
        return (x, offset, mask, weight, bias), (B, C, H, W, O, kh, kw, pad), (Ho, Wo)

    def forward(self, x, offset, mask, weight, bias, pad, nthreads=0):
        """Whole output [B, O, Ho, Wo] in fp64."""
        arrs, dims, (Ho, Wo) = self._prepare(x, offset, mask, weight, bias, pad)
        B, O = dims[0], dims[4]
        out = np.empty((B, O, Ho, Wo), dtype=np.float64)
        rc = self._lib.oracle_dcn_forward(*(self._ptr(a) for a in arrs), self._ptr(out),
                                          *dims, int(nthreads))
        if rc != 0:
            raise ValueError("oracle_dcn_forward rejected its arguments")
        return out

    def forward_points(self, x, offset, mask, weight, bias, pad, points, nthreads=0):
        """Selected pixels: points is an int array [n, 3] of (b, h, w);
        returns [n, O] fp64."""
        arrs, dims, _ = self._prepare(x, offset, mask, weight, bias, pad)
        pts = np.ascontiguousarray(points, dtype=np.int32).reshape(-1, 3)
        n = pts.shape[0]
        out = np.empty((n, dims[4]), dtype=np.float64)
        rc = self._lib.oracle_dcn_forward_points(*(self._ptr(a) for a in arrs),
                                                 self._ptr(pts), n, self._ptr(out),
                                                 *dims, int(nthreads))
        if rc != 0:
            raise ValueError("oracle_dcn_forward_points rejected its arguments")
        return out


    # ---------------------------------------------------------- general form

    def _prepare_ex(self, x, offset, mask, weight, bias, conv):
        """conv: ConvDesc (or a dict with its fields)."""
        c = conv if isinstance(conv, ConvDesc) else ConvDesc(**conv)
        x, offset, mask, weight, bias = (self._f32(t) for t in (x, offset, mask, weight, bias))
        B, C, H, W = x.shape
        O, Cg, kh, kw = weight.shape
        if c.groups <= 0 or C % c.groups or O % c.groups or Cg != C // c.groups:
            raise ValueError("weight shape does not match x and groups")
        if c.offset_groups <= 0 or C % c.offset_groups:
            raise ValueError("offset_groups must divide C")
        Ho, Wo = c.out_size(H, W, kh, kw)
        if Ho <= 0 or Wo <= 0:
            raise ValueError("empty output")
        k, G = kh * kw, c.offset_groups
        if offset.shape != (B, 2 * G * k, Ho, Wo):
            raise ValueError(f"offset shape {offset.shape} != {(B, 2 * G * k, Ho, Wo)}")
        if mask is not None and mask.shape != (B, G * k, Ho, Wo):
            raise ValueError(f"mask shape {mask.shape} != {(B, G * k, Ho, Wo)}")
        if bias is not None and bias.shape != (O,):
            raise ValueError("bias must have shape [O]")
        desc = np.array([B, C, H, W, O, kh, kw, c.stride[0], c.stride[1], c.padding[0],
                         c.padding[1], c.dilation[0], c.dilation[1], c.groups, G], dtype=np.int32)
        return (x, offset, mask, weight, bias), desc, (B, O, Ho, Wo)

    def forward_ex(self, x, offset, mask, weight, bias, conv, nthreads=0):
        """Whole output [B, O, Ho, Wo] in fp64 of the general problem."""
        arrs, desc, (B, O, Ho, Wo) = self._prepare_ex(x, offset, mask, weight, bias, conv)
        out = np.empty((B, O, Ho, Wo), dtype=np.float64)
        rc = self._lib.oracle_dcn_forward_ex(*(self._ptr(a) for a in arrs), self._ptr(out),
                                             self._ptr(desc), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_dcn_forward_ex rejected its arguments")
        return out

    def forward_points_ex(self, x, offset, mask, weight, bias, conv, points, nthreads=0):
        """Selected pixels (b, h, w) of the general problem: [n, O] fp64."""
        arrs, desc, (B, O, Ho, Wo) = self._prepare_ex(x, offset, mask, weight, bias, conv)
        pts = np.ascontiguousarray(points, dtype=np.int32).reshape(-1, 3)
        n = pts.shape[0]
        out = np.empty((n, O), dtype=np.float64)
        rc = self._lib.oracle_dcn_forward_points_ex(*(self._ptr(a) for a in arrs),
                                                    self._ptr(pts), n, self._ptr(out),
                                                    self._ptr(desc), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_dcn_forward_points_ex rejected its arguments")
        return out


    # ----------------------------------------------------------- backward

    def backward_ex(self, x, offset, mask, weight, grad_out, conv, nthreads=0):
        """Gradients of the general problem's forward with respect to x,
        offset, mask, weight and bias, given grad_out [B, O, Ho, Wo]: a dict
        of fp64 arrays in the inputs' layouts (grad_mask None without a
        mask)."""
        arrs, desc, (B, O, Ho, Wo) = self._prepare_ex(x, offset, mask, weight, None, conv)
        x, offset, mask, weight, _ = arrs
        go = self._f32(grad_out)
        if go.shape != (B, O, Ho, Wo):
            raise ValueError(f"grad_out shape {go.shape} != {(B, O, Ho, Wo)}")
        gx = np.empty(x.shape, dtype=np.float64)
        goff = np.empty(offset.shape, dtype=np.float64)
        gm = None if mask is None else np.empty(mask.shape, dtype=np.float64)
        gw = np.empty(weight.shape, dtype=np.float64)
        gb = np.empty((O,), dtype=np.float64)
        rc = self._lib.oracle_dcn_backward_ex(
            self._ptr(x), self._ptr(offset), self._ptr(mask), self._ptr(weight), self._ptr(go),
            self._ptr(gx), self._ptr(goff), self._ptr(gm), self._ptr(gw), self._ptr(gb),
            self._ptr(desc), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_dcn_backward_ex rejected its arguments")
        return {"grad_x": gx, "grad_offset": goff, "grad_mask": gm, "grad_weight": gw,
                "grad_bias": gb}

    def backward_points_ex(self, x, offset, mask, weight, grad_out, conv, points, nthreads=0):
        """grad_offset [n, 2*G*k] and grad_mask [n, G*k] (None without a
        mask) at output pixels points [n, 3] of (b, h, w)."""
        arrs, desc, (B, O, Ho, Wo) = self._prepare_ex(x, offset, mask, weight, None, conv)
        x, offset, mask, weight, _ = arrs
        go = self._f32(grad_out)
        if go.shape != (B, O, Ho, Wo):
            raise ValueError(f"grad_out shape {go.shape} != {(B, O, Ho, Wo)}")
        pts = np.ascontiguousarray(points, dtype=np.int32).reshape(-1, 3)
        n = pts.shape[0]
        goff = np.empty((n, offset.shape[1]), dtype=np.float64)
        gm = None if mask is None else np.empty((n, mask.shape[1]), dtype=np.float64)
        rc = self._lib.oracle_dcn_backward_points_ex(
            self._ptr(x), self._ptr(offset), self._ptr(mask), self._ptr(weight), self._ptr(go),
            self._ptr(pts), n, self._ptr(goff), self._ptr(gm), self._ptr(desc), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_dcn_backward_points_ex rejected its arguments")
        return goff, gm

    def backward(self, x, offset, mask, weight, grad_out, pad, nthreads=0):
        """backward_ex for the page-1 problem (stride 1, dilation 1, one
        padding, one weight group, one offset group)."""
        return self.backward_ex(x, offset, mask, weight, grad_out, ConvDesc(padding=pad),
                                nthreads)


    # --------------------------------------------------------------- MSDA

    def msda_forward(self, value, shapes, starts, locations, weights, softmax=False, nthreads=0):
        """Multi-scale deformable attention: value [B, S, G, D], shapes [L, 2]
        (H, W), starts [L], locations [B, Q, G, L, K, 2], weights
        [B, Q, G, L*K]; returns out [B, Q, G, D] in fp64."""
        value, locations, weights = (self._f32(t) for t in (value, locations, weights))
        shapes = np.ascontiguousarray(np.asarray(shapes), dtype=np.int32).reshape(-1, 2)
        starts = np.ascontiguousarray(np.asarray(starts), dtype=np.int32).reshape(-1)
        B, S, G, D = value.shape
        L = shapes.shape[0]
        Bq, Q, G2, L2, K, two = locations.shape
        if (Bq, G2, L2, two) != (B, G, L, 2) or weights.shape != (B, Q, G, L * K) or starts.shape != (L,):
            raise ValueError("msda shapes do not match")
        out = np.empty((B, Q, G, D), dtype=np.float64)
        rc = self._lib.oracle_msda_forward(self._ptr(value), self._ptr(shapes), self._ptr(starts), L,
                                           self._ptr(locations), self._ptr(weights), int(bool(softmax)),
                                           self._ptr(out), B, S, G, D, Q, K, int(nthreads))
        if rc != 0:
            raise ValueError("oracle_msda_forward rejected its arguments")
        return out

    def attn_forward(self, value, offsets, weights, kernel_size, stride=1, padding=0, dilation=1,
                     softmax=False, nthreads=0):
        """Single-scale deformable sampling: value [B, H, W, G, D], offsets
        [B, Ho, Wo, G, K, 2] as (dy, dx), weights [B, Ho, Wo, G, K]; returns
        out [B, Ho, Wo, G, D] in fp64.  kernel_size, stride, padding and
        dilation are ints or (h, w) pairs."""
        pair = lambda v: (int(v), int(v)) if np.isscalar(v) else (int(v[0]), int(v[1]))  # noqa: E731
        (kh, kw), (sh, sw), (ph, pw), (dh, dw) = (pair(v) for v in
                                                  (kernel_size, stride, padding, dilation))
        value, offsets, weights = (self._f32(t) for t in (value, offsets, weights))
        B, H, W, G, D = value.shape
        K = kh * kw
        Ho = (H + 2 * ph - dh * (kh - 1) - 1) // sh + 1
        Wo = (W + 2 * pw - dw * (kw - 1) - 1) // sw + 1
        if offsets.shape != (B, Ho, Wo, G, K, 2) or weights.shape != (B, Ho, Wo, G, K):
            raise ValueError("attn shapes do not match")
        out = np.empty((B, Ho, Wo, G, D), dtype=np.float64)
        rc = self._lib.oracle_attn_forward(self._ptr(value), self._ptr(offsets), self._ptr(weights),
                                           int(bool(softmax)), self._ptr(out), B, H, W, G, D, kh, kw,
                                           sh, sw, ph, pw, dh, dw, int(nthreads))
        if rc != 0:
            raise ValueError("oracle_attn_forward rejected its arguments")
        return out

    def attn_backward(self, value, offsets, weights, grad_out, kernel_size, stride=1, padding=0,
                      dilation=1, softmax=False, nthreads=0):
        """Gradients of attn_forward for the cotangent grad_out [B, Ho, Wo,
        G, D]: (grad_value [B, H, W, G, D], grad_offsets [B, Ho, Wo, G, K, 2]
        as (dy, dx), grad_weights [B, Ho, Wo, G, K]), fp64."""
        pair = lambda v: (int(v), int(v)) if np.isscalar(v) else (int(v[0]), int(v[1]))  # noqa: E731
        (kh, kw), (sh, sw), (ph, pw), (dh, dw) = (pair(v) for v in
                                                  (kernel_size, stride, padding, dilation))
        value, offsets, weights, grad_out = (self._f32(t) for t in
                                             (value, offsets, weights, grad_out))
        B, H, W, G, D = value.shape
        K = kh * kw
        Ho = (H + 2 * ph - dh * (kh - 1) - 1) // sh + 1
        Wo = (W + 2 * pw - dw * (kw - 1) - 1) // sw + 1
        if (offsets.shape != (B, Ho, Wo, G, K, 2) or weights.shape != (B, Ho, Wo, G, K)
                or grad_out.shape != (B, Ho, Wo, G, D)):
            raise ValueError("attn shapes do not match")
        gv = np.empty((B, H, W, G, D), dtype=np.float64)
        go_ = np.empty((B, Ho, Wo, G, K, 2), dtype=np.float64)
        gw = np.empty((B, Ho, Wo, G, K), dtype=np.float64)
        rc = self._lib.oracle_attn_backward(self._ptr(value), self._ptr(offsets), self._ptr(weights),
                                            int(bool(softmax)), self._ptr(grad_out), self._ptr(gv),
                                            self._ptr(go_), self._ptr(gw), B, H, W, G, D, kh, kw,
                                            sh, sw, ph, pw, dh, dw, int(nthreads))
        if rc != 0:
            raise ValueError("oracle_attn_backward rejected its arguments")
        return gv, go_, gw

    def msda_backward(self, value, shapes, starts, locations, weights, grad_out, softmax=False,
                      nthreads=0):
        """Gradients of msda_forward for the cotangent grad_out [B, Q, G, D]:
        (grad_value [B, S, G, D], grad_locations [B, Q, G, L, K, 2],
        grad_weights [B, Q, G, L*K]), fp64."""
        value, locations, weights, grad_out = (self._f32(t) for t in
                                               (value, locations, weights, grad_out))
        shapes = np.ascontiguousarray(np.asarray(shapes), dtype=np.int32).reshape(-1, 2)
        starts = np.ascontiguousarray(np.asarray(starts), dtype=np.int32).reshape(-1)
        B, S, G, D = value.shape
        L = shapes.shape[0]
        Bq, Q, G2, L2, K, two = locations.shape
        if ((Bq, G2, L2, two) != (B, G, L, 2) or weights.shape != (B, Q, G, L * K)
                or starts.shape != (L,) or grad_out.shape != (B, Q, G, D)):
            raise ValueError("msda shapes do not match")
        gv = np.empty((B, S, G, D), dtype=np.float64)
        gl = np.empty((B, Q, G, L, K, 2), dtype=np.float64)
        gw = np.empty((B, Q, G, L * K), dtype=np.float64)
        rc = self._lib.oracle_msda_backward(self._ptr(value), self._ptr(shapes), self._ptr(starts), L,
                                            self._ptr(locations), self._ptr(weights),
                                            int(bool(softmax)), self._ptr(grad_out), self._ptr(gv),
                                            self._ptr(gl), self._ptr(gw), B, S, G, D, Q, K,
                                            int(nthreads))
        if rc != 0:
            raise ValueError("oracle_msda_backward rejected its arguments")
        return gv, gl, gw


class ConvDesc:
    """Convolution parameters of the general problem: stride, padding and
    dilation as (h, w) pairs (an int means both), weight groups and offset
    (deformable) groups."""

    def __init__(self, stride=1, padding=0, dilation=1, groups=1, offset_groups=1):
        pair = lambda v: (int(v), int(v)) if np.isscalar(v) else (int(v[0]), int(v[1]))  # noqa: E731
        self.stride, self.padding, self.dilation = pair(stride), pair(padding), pair(dilation)
        self.groups, self.offset_groups = int(groups), int(offset_groups)

    def out_size(self, H, W, kh, kw):
        def one(n, k, s, p, d):
            span = n + 2 * p - d * (k - 1) - 1
            return span // s + 1 if span >= 0 else 0
        return (one(H, kh, self.stride[0], self.padding[0], self.dilation[0]),
                one(W, kw, self.stride[1], self.padding[1], self.dilation[1]))

    def __repr__(self):
        return (f"ConvDesc(stride={self.stride}, padding={self.padding}, dilation={self.dilation}, "
                f"groups={self.groups}, offset_groups={self.offset_groups})")


_default = None


def get():
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def forward(*args, **kwargs):
    return get().forward(*args, **kwargs)


def forward_points(*args, **kwargs):
    return get().forward_points(*args, **kwargs)


def forward_ex(*args, **kwargs):
    return get().forward_ex(*args, **kwargs)


def forward_points_ex(*args, **kwargs):
    return get().forward_points_ex(*args, **kwargs)


def backward(*args, **kwargs):
    return get().backward(*args, **kwargs)


def backward_ex(*args, **kwargs):
    return get().backward_ex(*args, **kwargs)


def backward_points_ex(*args, **kwargs):
    return get().backward_points_ex(*args, **kwargs)


def msda_forward(*args, **kwargs):
    return get().msda_forward(*args, **kwargs)


def msda_backward(*args, **kwargs):
    return get().msda_backward(*args, **kwargs)


def attn_forward(*args, **kwargs):
    return get().attn_forward(*args, **kwargs)


def attn_backward(*args, **kwargs):
    return get().attn_backward(*args, **kwargs)
