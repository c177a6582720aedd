"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is the oracle's C source with one plausible slip (a swapped
offset channel, truncation instead of floor, a swapped corner weight, a
transposed tap order, a wrong padding sign, the mask or bias dropped, an
off-by-one border test; for the general form swapped stride or padding
axes, a dropped dilation, a wrong offset-group or weight-group index).
Every mutant stays inside its arrays.  It is compiled into a temporary library and run
against every pin; a mutant that passes all of them would mean the pins
cannot see that class of error.  The mistakes are planted on the CPU only.
"""

import os
import subprocess

import pytest

import oracle
from tests import pins

MUTANTS = {
    "swap_dy_dx": [("+ j * p->dw) + dx;", "+ j * p->dw) + dy;"), ("+ i * p->dh) + dy;", "+ i * p->dh) + dx;")],
    "trunc_not_floor": [("floorf(py)", "truncf(py)"), ("floorf(px)", "truncf(px)")],
    "swap_x_weights": [("wx[2] = {1.0 - lx, lx}", "wx[2] = {lx, 1.0 - lx}")],
    "swap_y_weights": [("wy[2] = {1.0 - ly, ly}", "wy[2] = {ly, 1.0 - ly}")],
    "tap_order_column_major": [("const int k = i * p->kw + j;", "const int k = j * p->kh + i;")],
    "pad_sign": [("(float)(h * p->sh - p->ph + i * p->dh)", "(float)(h * p->sh + p->ph + i * p->dh)")],
    "mask_dropped": [("acc += wt * m * s;", "acc += wt * s;")],
    "bias_dropped": [("out[o * out_stride] = acc + (p->bias ? (double)p->bias[o] : 0.0);",
                      "out[o * out_stride] = acc;")],
    "border_off_by_one": [("yy <= p->H - 1", "yy <= p->H - 2")],
    "corner_step_wrong": [("const double xx = (double)fx0 + e;", "const double xx = (double)fx0 + 2 * e;")],
    # the general parameters
    "stride_axes_swapped": [("h * p->sh - p->ph", "h * p->sw - p->ph"), ("w * p->sw - p->pw", "w * p->sh - p->pw")],
    "dilation_dropped": [("+ i * p->dh) + dy", "+ i) + dy"), ("+ j * p->dw) + dx", "+ j) + dx")],
    "pad_axes_swapped": [("h * p->sh - p->ph", "h * p->sh - p->pw"), ("w * p->sw - p->pw", "w * p->sw - p->ph")],
    "offset_group_by_weight_group": [("const size_t oq = (size_t)b * p->ogroups + q;",
                                      "const size_t oq = (size_t)b * p->ogroups + (c / Cg) % p->ogroups;")],
    "weight_group_modulo": [("const int g = o / Og;", "const int g = o % p->groups;")],
    "weight_channel_rotated": [("(c - g * Cg)) * p->kh", "((c - g * Cg + 1) % Cg)) * p->kh")],
    "offset_group_ignored": [("const size_t oq = (size_t)b * p->ogroups + q;",
                              "const size_t oq = (size_t)b * p->ogroups;")],
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as fh:
        return fh.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, source, name):
    text = source
    for old, new in MUTANTS[name]:
        assert old in text, f"mutation anchor not found: {old!r}"
        text = text.replace(old, new, 1)   # the first occurrence: the forward's code
    src = os.path.join(tmp_path, f"{name}.c")
    lib = os.path.join(tmp_path, f"{name}.so")
    with open(src, "w") as fh:
        fh.write(text)
    oracle.compile_oracle(src, lib)
    mutant = oracle.Oracle(lib, src)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
