"""The C-ABI library loads and exports every symbol the header declares
(no GPU needed; no compute is launched)."""

import ctypes
import os
import re

import pytest
import torch

from deformable_convolution_vision_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dcn.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIBRARY):
        from deformable_convolution_vision_gb300 import build
        build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DCN_API\s+[\w\s\*]+?\b(dcn_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(binding.EXPORTS) == set(names), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert binding.dcn_status_string(code) == name
    assert binding.dcn_status_string(99) == "DCN_ERR_UNKNOWN"


def test_null_handle_is_rejected_before_any_launch(lib):
    assert lib.dcn_set_path(None, 0) == binding.STATUS_CODE["DCN_ERR_INVALID_ARG"]
    assert lib.dcn_last_path(None) == -1
    assert lib.dcn_destroy(None) == 0
    args = [None] * 7 + [1, 64, 8, 8, 64, 3, 3, 1, 1, None]
    assert lib.dcn_forward(*args) == binding.STATUS_CODE["DCN_ERR_INVALID_ARG"]
    assert lib.dcn_sync_status(None, None) == binding.STATUS_CODE["DCN_ERR_INVALID_ARG"]
    assert lib.dcn_selftest_timeout(None, 1000, None) == binding.STATUS_CODE["DCN_ERR_INVALID_ARG"]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_device_reports_no_device(lib):
    h = ctypes.c_void_p()
    assert lib.dcn_create(ctypes.byref(h)) == binding.STATUS_CODE["DCN_ERR_NO_DEVICE"]
    assert h.value is None


def test_python_wrappers_marshal_every_argument(lib):
    """Each binding wrapper passes exactly the arguments its C function
    takes; NULL pointers come back as DCN_ERR_INVALID_ARG before any launch
    (no device is touched)."""
    bad = binding.STATUS_CODE["DCN_ERR_INVALID_ARG"]
    h = ctypes.c_void_p()   # NULL handle
    desc = binding.ConvDesc(1, 64, 8, 8, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1, 1)
    calls = [
        lambda: binding.dcn_forward(h, None, None, None, None, None, None, 1, 64, 8, 8, 64, 3, 3, 1,
                                    1, 0),
        lambda: binding.dcn_forward_packed(h, None, None, None, None, None, 1, 64, 8, 8, 64, 3, 3, 1,
                                           1, 0),
        lambda: binding.dcn_pack_weight(h, None, 64, 64, 3, 3, 1, 0),
        lambda: binding.dcn_forward_host(h, None, None, None, None, None, None, 1, 64, 8, 8, 64, 3, 3,
                                         1, 1, 0),
        lambda: binding.dcn_forward_ex(h, None, None, None, None, None, None, desc, 1, 0),
        lambda: binding.dcn_pack_weight_ex(h, None, desc, 1, 0),
        lambda: binding.dcn_forward_packed_ex(h, None, None, None, None, None, desc, 1, 0),
        lambda: binding.dcn_forward_noalloc(None, None, None, None, None, None, 1, 64, 8, 8, 64, 3,
                                            3, 1, 1, 0),
        lambda: binding.dcn_backward(h, None, None, None, None, None, None, None, None, None, None,
                                     1, 64, 8, 8, 64, 3, 3, 1, 1, 0),
        lambda: binding.dcn_backward_ex(h, None, None, None, None, None, None, None, None, None,
                                        None, desc, 1, 0),
        lambda: binding.dcn_msda_forward(None, [(8, 8)], [0], None, None, None, 1, 64, 8, 32, 10,
                                         4, True, 1, 0),
        lambda: binding.dcn_msda_backward(None, [(8, 8)], [0], None, None, None, None, None, None,
                                          1, 64, 8, 32, 10, 4, True, 1, 0),
        lambda: binding.dcn_attn_forward(None, None, None, None, 1, 8, 8, 4, 16, 3, 3, 1, 1, 1, 1,
                                         1, 1, True, 1, 0),
        lambda: binding.dcn_attn_backward(None, None, None, None, None, None, None, 1, 8, 8, 4, 16,
                                          3, 3, 1, 1, 1, 1, 1, 1, True, 1, 0),
        lambda: binding.dcn_nchw_to_nhwc(None, None, 1, 64, 8, 8, 1, 0),
        lambda: binding.dcn_nhwc_to_nchw(None, None, 1, 64, 8, 8, 1, 0),
    ]
    for call in calls:
        with pytest.raises(binding.DcnError) as e:
            call()
        assert e.value.status == bad


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers: only where nothing can launch")
def test_sizes_whose_product_wraps_are_rejected(lib):
    """Every indexed tensor must hold fewer than 2^31 elements.  Dimensions
    whose element count overflows a 64-bit product (and would wrap round
    to a small one) must still be refused, before any launch.  The pointers
    are fake and never dereferenced."""
    bad = binding.STATUS_CODE["DCN_ERR_INVALID_ARG"]
    src, dst, f32a, f32b, f32c = (ctypes.c_void_p(0x100000 * k) for k in range(1, 6))
    # value 2^30 x 2^30 pixels of 16 channels: 2^64 elements; a 2^30 stride
    # leaves a 1 x 1 output, so every other count is small
    big, stride = 1 << 30, 1 << 30
    assert lib.dcn_attn_forward(src, f32a, f32b, dst, 1, big, big, 1, 16, 1, 1, stride, stride,
                                0, 0, 1, 1, 1, 1, None) == bad
    assert lib.dcn_attn_backward(src, f32a, f32b, dst, f32a, f32b, f32c, 1, big, big, 1, 16, 1, 1,
                                 stride, stride, 0, 0, 1, 1, 1, 1, None) == bad
    # layout copies: 2^15 images of 2^20 channels x 2^14 x 2^15 pixels = 2^64
    assert lib.dcn_nchw_to_nhwc(src, dst, 1 << 15, 1 << 20, 1 << 14, 1 << 15, 1, None) == bad
    assert lib.dcn_nhwc_to_nchw(src, dst, 1 << 15, 1 << 20, 1 << 14, 1 << 15, 1, None) == bad
    # plainly oversized problems on the other handle-free entries
    shapes = (ctypes.c_int * 2)(8, 8)
    starts = (ctypes.c_int * 1)(0)
    assert lib.dcn_msda_forward(src, shapes, starts, 1, f32a, f32b, dst, 2, 1 << 30, 1, 2, 1, 1,
                                1, 1, None) == bad
    assert lib.dcn_msda_backward(src, shapes, starts, 1, f32a, f32b, dst, f32a, f32b, f32c, 2,
                                 1 << 30, 1, 2, 1, 1, 1, 1, None) == bad
    assert lib.dcn_forward_noalloc(src, f32a, f32b, dst, f32c, dst, 1, 1 << 16, 1 << 16, 1 << 16,
                                   16, 1, 1, 0, 1, None) == bad
    assert lib.dcn_out_size(1 << 30, 1, 1, 1 << 30, 1) == 0
