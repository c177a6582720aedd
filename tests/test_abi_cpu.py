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
