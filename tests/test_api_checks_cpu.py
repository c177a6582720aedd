"""The Python entry points' buffer checks, on the CPU.

The kernels take raw pointers: a tensor on another device, or a caller's
``out`` of the wrong size, dtype or layout, would be read or written out of
bounds.  The helpers that refuse them are checked here with host and
``meta`` tensors; nothing reaches the library.
"""

import pytest
import torch

import deformable_convolution_vision_gb300 as dcn

CPU = torch.device("cpu")


def test_devices_must_match():
    a = torch.zeros(4)
    dcn._check_devices(CPU, offset=a, mask=None, weight=a)
    with pytest.raises(ValueError, match="mask must be on cpu"):
        dcn._check_devices(CPU, offset=a, mask=torch.zeros(4, device="meta"))


def test_out_must_be_exactly_what_the_kernel_writes():
    shape = (2, 8, 5, 3)
    good = torch.empty(shape, memory_format=torch.channels_last)
    dcn._check_out(good, shape, torch.float32, CPU, channels_last=True)
    dcn._check_out(torch.empty(shape), shape, torch.float32, CPU)
    bad = {
        "short": torch.empty((2, 8, 5, 2), memory_format=torch.channels_last),
        "dtype": torch.empty(shape, dtype=torch.bfloat16, memory_format=torch.channels_last),
        "layout": torch.empty(shape),                                   # NCHW, not channels-last
        "strided": torch.empty((2, 8, 5, 6), memory_format=torch.channels_last)[..., ::2],
        "device": torch.empty(shape, device="meta", memory_format=torch.channels_last),
    }
    for name, t in bad.items():
        with pytest.raises(ValueError, match="out must be"):
            dcn._check_out(t, shape, torch.float32, CPU, channels_last=True)
    with pytest.raises(ValueError):
        dcn._check_out(torch.empty(shape, memory_format=torch.channels_last), shape,
                       torch.float32, CPU)                               # contiguous wanted


def test_host_tensors_are_refused_before_the_library():
    x = torch.zeros(1, 4, 8, 8).contiguous(memory_format=torch.channels_last)
    with pytest.raises(ValueError, match="CUDA"):
        dcn.deform_conv2d(x, torch.zeros(1, 18, 8, 8), torch.zeros(4, 4, 3, 3), padding=1)
    v = torch.zeros(1, 64, 2, 16)
    with pytest.raises(ValueError, match="CUDA"):
        dcn.msda(v, [(8, 8)], [0], torch.zeros(1, 3, 2, 1, 4, 2), torch.zeros(1, 3, 2, 4))
    with pytest.raises(ValueError, match="CUDA"):
        dcn.attn(torch.zeros(1, 8, 8, 2, 16), torch.zeros(1, 8, 8, 2, 9, 2),
                 torch.zeros(1, 8, 8, 2, 9), 3, padding=1)
