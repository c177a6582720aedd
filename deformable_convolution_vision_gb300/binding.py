"""ctypes binding of ``libdcn.so`` with the C ABI's names.

Argument marshalling only: tensors become device (or host) pointers, the
stream becomes a ``cudaStream_t``; every step of the forward pass runs in
the library's CUDA kernels.  There is no fallback: if the library is not
built, every call raises.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libdcn.so")

DCN_F32, DCN_BF16, DCN_F16 = 0, 1, 2
DCN_PATH_AUTO, DCN_PATH_SIMT, DCN_PATH_TC = 0, 1, 2
DCN_SAMPLE_INPUT_DTYPE, DCN_SAMPLE_F32 = 0, 1
STATUS = {0: "DCN_OK", 1: "DCN_ERR_INVALID_ARG", 2: "DCN_ERR_UNSUPPORTED", 3: "DCN_ERR_CUDA",
          4: "DCN_ERR_NO_DEVICE", 5: "DCN_ERR_OOM", 6: "DCN_ERR_TIMEOUT", 7: "DCN_ERR_BOUNDS"}
STATUS_CODE = {v: k for k, v in STATUS.items()}

EXPORTS = ["dcn_create", "dcn_destroy", "dcn_forward", "dcn_pack_weight", "dcn_forward_packed",
           "dcn_forward_host", "dcn_set_path", "dcn_last_path", "dcn_sync_status",
           "dcn_selftest_timeout", "dcn_status_string", "dcn_forward_noalloc",
           "dcn_set_sample_precision", "dcn_out_size", "dcn_forward_ex", "dcn_pack_weight_ex",
           "dcn_forward_packed_ex", "dcn_backward", "dcn_backward_ex", "dcn_msda_forward",
           "dcn_msda_backward", "dcn_attn_forward", "dcn_attn_backward", "dcn_nchw_to_nhwc",
           "dcn_nhwc_to_nchw"]


class ConvDesc(ctypes.Structure):
    """``dcn_conv_desc_t``: the general problem (stride, per-axis padding,
    dilation, weight groups, offset groups)."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "C", "H", "W", "O", "kh", "kw", "stride_h", "stride_w", "pad_h", "pad_w",
        "dil_h", "dil_w", "groups", "offset_groups")]


class DcnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None


def load():
    """Load libdcn.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY):
        raise RuntimeError(f"{LIBRARY} is not built; run deformable_convolution_vision_gb300.build.build()")
    lib = ctypes.CDLL(LIBRARY)
    P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    fwd = [P, P, P, P, P, P, P] + [I] * 9 + [P]
    sig = {
        "dcn_create": ([ctypes.POINTER(P)], I),
        "dcn_destroy": ([P], I),
        "dcn_forward": (fwd, I),
        "dcn_pack_weight": ([P, P, I, I, I, I, I, P], I),
        "dcn_forward_packed": ([P, P, P, P, P, P] + [I] * 9 + [P], I),
        "dcn_forward_host": (fwd, I),
        "dcn_set_path": ([P, I], I),
        "dcn_set_sample_precision": ([P, I], I),
        "dcn_last_path": ([P], I),
        "dcn_sync_status": ([P, P], I),
        "dcn_selftest_timeout": ([P, LL, P], I),
        "dcn_status_string": ([I], ctypes.c_char_p),
        "dcn_forward_noalloc": ([P, P, P, P, P, P] + [I] * 9 + [P], I),
        "dcn_out_size": ([I] * 5, I),
        "dcn_forward_ex": ([P, P, P, P, P, P, P, ctypes.POINTER(ConvDesc), I, P], I),
        "dcn_pack_weight_ex": ([P, P, ctypes.POINTER(ConvDesc), I, P], I),
        "dcn_forward_packed_ex": ([P, P, P, P, P, P, ctypes.POINTER(ConvDesc), I, P], I),
        "dcn_backward": ([P] * 11 + [I] * 9 + [P], I),
        "dcn_backward_ex": ([P] * 11 + [ctypes.POINTER(ConvDesc), I, P], I),
        "dcn_msda_forward": ([P, P, P, I, P, P, P] + [I] * 8 + [P], I),
        "dcn_msda_backward": ([P, P, P, I, P, P, P, P, P, P] + [I] * 8 + [P], I),
        "dcn_attn_forward": ([P, P, P, P] + [I] * 15 + [P], I),
        "dcn_attn_backward": ([P] * 7 + [I] * 15 + [P], I),
        "dcn_nchw_to_nhwc": ([P, P] + [I] * 5 + [P], I),
        "dcn_nhwc_to_nchw": ([P, P] + [I] * 5 + [P], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _ptr(t):
    """Pointer of a tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != 0:
        raise DcnError(status, where)


def dcn_status_string(status):
    return load().dcn_status_string(status).decode()


def dcn_create():
    h = ctypes.c_void_p()
    _check(load().dcn_create(ctypes.byref(h)), "dcn_create")
    return h


def dcn_destroy(h):
    _check(load().dcn_destroy(h), "dcn_destroy")


def dcn_forward(h, x, offset, mask, weight, bias, out, B, C, H, W, O, kh, kw, pad, dtype,
                stream=None):
    _check(load().dcn_forward(h, _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight), _ptr(bias),
                              _ptr(out), B, C, H, W, O, kh, kw, pad, dtype, _stream(stream)),
           "dcn_forward")


def dcn_pack_weight(h, weight, O, C, kh, kw, dtype, stream=None):
    _check(load().dcn_pack_weight(h, _ptr(weight), O, C, kh, kw, dtype, _stream(stream)),
           "dcn_pack_weight")


def dcn_forward_packed(h, x, offset, mask, bias, out, B, C, H, W, O, kh, kw, pad, dtype,
                       stream=None):
    _check(load().dcn_forward_packed(h, _ptr(x), _ptr(offset), _ptr(mask), _ptr(bias), _ptr(out),
                                     B, C, H, W, O, kh, kw, pad, dtype, _stream(stream)),
           "dcn_forward_packed")


def dcn_forward_host(h, x, offset, mask, weight, bias, out, B, C, H, W, O, kh, kw, pad, dtype,
                     stream=None):
    _check(load().dcn_forward_host(h, _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight), _ptr(bias),
                                   _ptr(out), B, C, H, W, O, kh, kw, pad, dtype, _stream(stream)),
           "dcn_forward_host")


def dcn_set_path(h, path):
    _check(load().dcn_set_path(h, path), "dcn_set_path")


def dcn_set_sample_precision(h, mode):
    _check(load().dcn_set_sample_precision(h, mode), "dcn_set_sample_precision")


def dcn_last_path(h):
    return load().dcn_last_path(h)


def dcn_sync_status(h, stream=None):
    """Returns the status code (0 = OK) instead of raising, so callers can
    inspect DCN_ERR_TIMEOUT."""
    return load().dcn_sync_status(h, _stream(stream))


def dcn_selftest_timeout(h, timeout_ns, stream=None):
    _check(load().dcn_selftest_timeout(h, int(timeout_ns), _stream(stream)), "dcn_selftest_timeout")


def dcn_forward_noalloc(x, offset, mask, weight, bias, out, B, C, H, W, O, kh, kw, pad, dtype,
                        stream=None):
    """The allocation-free forward pass (no handle; fixed scratch)."""
    _check(load().dcn_forward_noalloc(_ptr(x), _ptr(offset), _ptr(mask), _ptr(weight), _ptr(bias),
                                      _ptr(out), B, C, H, W, O, kh, kw, pad, dtype,
                                      _stream(stream)),
           "dcn_forward_noalloc")


def dcn_out_size(n, k, stride, pad, dil):
    return load().dcn_out_size(n, k, stride, pad, dil)


def dcn_forward_ex(h, x, offset, mask, weight, bias, out, desc, dtype, stream=None):
    _check(load().dcn_forward_ex(h, _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight), _ptr(bias),
                                 _ptr(out), ctypes.byref(desc), dtype, _stream(stream)),
           "dcn_forward_ex")


def dcn_pack_weight_ex(h, weight, desc, dtype, stream=None):
    _check(load().dcn_pack_weight_ex(h, _ptr(weight), ctypes.byref(desc), dtype, _stream(stream)),
           "dcn_pack_weight_ex")


def dcn_forward_packed_ex(h, x, offset, mask, bias, out, desc, dtype, stream=None):
    _check(load().dcn_forward_packed_ex(h, _ptr(x), _ptr(offset), _ptr(mask), _ptr(bias),
                                        _ptr(out), ctypes.byref(desc), dtype, _stream(stream)),
           "dcn_forward_packed_ex")


def dcn_backward(h, x, offset, mask, weight, grad_out, grad_x, grad_offset, grad_mask,
                 grad_weight, grad_bias, B, C, H, W, O, kh, kw, pad, dtype, stream=None):
    _check(load().dcn_backward(h, _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight), _ptr(grad_out),
                               _ptr(grad_x), _ptr(grad_offset), _ptr(grad_mask), _ptr(grad_weight),
                               _ptr(grad_bias), B, C, H, W, O, kh, kw, pad, dtype,
                               _stream(stream)),
           "dcn_backward")


def dcn_backward_ex(h, x, offset, mask, weight, grad_out, grad_x, grad_offset, grad_mask,
                    grad_weight, grad_bias, desc, dtype, stream=None):
    _check(load().dcn_backward_ex(h, _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight),
                                  _ptr(grad_out), _ptr(grad_x), _ptr(grad_offset), _ptr(grad_mask),
                                  _ptr(grad_weight), _ptr(grad_bias), ctypes.byref(desc), dtype,
                                  _stream(stream)),
           "dcn_backward_ex")


def dcn_msda_forward(value, shapes, starts, locations, weights, out, B, S, G, D, Q, K, softmax,
                     dtype, stream=None):
    """shapes: host sequence of (H, W) pairs; starts: host sequence of row offsets."""
    L = len(starts)
    sh = (ctypes.c_int * (2 * L))(*[int(v) for hw in shapes for v in hw])
    st = (ctypes.c_int * L)(*[int(v) for v in starts])
    _check(load().dcn_msda_forward(_ptr(value), sh, st, L, _ptr(locations), _ptr(weights), _ptr(out),
                                   B, S, G, D, Q, K, int(bool(softmax)), dtype, _stream(stream)),
           "dcn_msda_forward")


def dcn_msda_backward(value, shapes, starts, locations, weights, grad_out, grad_value,
                      grad_locations, grad_weights, B, S, G, D, Q, K, softmax, dtype, stream=None):
    """shapes: host sequence of (H, W) pairs; starts: host sequence of row offsets."""
    L = len(starts)
    sh = (ctypes.c_int * (2 * L))(*[int(v) for hw in shapes for v in hw])
    st = (ctypes.c_int * L)(*[int(v) for v in starts])
    _check(load().dcn_msda_backward(_ptr(value), sh, st, L, _ptr(locations), _ptr(weights),
                                    _ptr(grad_out), _ptr(grad_value), _ptr(grad_locations),
                                    _ptr(grad_weights), B, S, G, D, Q, K, int(bool(softmax)),
                                    dtype, _stream(stream)),
           "dcn_msda_backward")


def dcn_attn_forward(value, offsets, weights, out, B, H, W, G, D, kh, kw, stride_h, stride_w,
                     pad_h, pad_w, dil_h, dil_w, softmax, dtype, stream=None):
    _check(load().dcn_attn_forward(_ptr(value), _ptr(offsets), _ptr(weights), _ptr(out), B, H, W,
                                   G, D, kh, kw, stride_h, stride_w, pad_h, pad_w, dil_h, dil_w,
                                   int(bool(softmax)), dtype, _stream(stream)),
           "dcn_attn_forward")


def dcn_attn_backward(value, offsets, weights, grad_out, grad_value, grad_offsets, grad_weights,
                      B, H, W, G, D, kh, kw, stride_h, stride_w, pad_h, pad_w, dil_h, dil_w,
                      softmax, dtype, stream=None):
    _check(load().dcn_attn_backward(_ptr(value), _ptr(offsets), _ptr(weights), _ptr(grad_out),
                                    _ptr(grad_value), _ptr(grad_offsets), _ptr(grad_weights), B, H,
                                    W, G, D, kh, kw, stride_h, stride_w, pad_h, pad_w, dil_h,
                                    dil_w, int(bool(softmax)), dtype, _stream(stream)),
           "dcn_attn_backward")


def dcn_nchw_to_nhwc(src, dst, B, C, H, W, dtype, stream=None):
    _check(load().dcn_nchw_to_nhwc(_ptr(src), _ptr(dst), B, C, H, W, dtype, _stream(stream)),
           "dcn_nchw_to_nhwc")


def dcn_nhwc_to_nchw(src, dst, B, C, H, W, dtype, stream=None):
    _check(load().dcn_nhwc_to_nchw(_ptr(src), _ptr(dst), B, C, H, W, dtype, _stream(stream)),
           "dcn_nhwc_to_nchw")
