"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is the oracle's C source with one plausible slip (a swapped
offset channel, truncation instead of floor, a swapped corner weight, a
transposed tap order, a wrong padding sign, the mask or bias dropped, an
off-by-one border test).  It is compiled into a temporary library and run
against every pin; a mutant that passes all of them would mean the pins
cannot see that class of error.  The mistakes are planted on the CPU only.
"""

import os
import subprocess

import pytest

import oracle
from tests import pins

MUTANTS = {
    "swap_dy_dx": [("+ j) + dx;", "+ j) + dy;"), ("+ i) + dy;", "+ i) + dx;")],
    "trunc_not_floor": [("floorf(py)", "truncf(py)"), ("floorf(px)", "truncf(px)")],
    "swap_x_weights": [("wx[2] = {1.0 - lx, lx}", "wx[2] = {lx, 1.0 - lx}")],
    "swap_y_weights": [("wy[2] = {1.0 - ly, ly}", "wy[2] = {ly, 1.0 - ly}")],
    "tap_order_column_major": [("const int k = i * p->kw + j;", "const int k = j * p->kh + i;")],
    "pad_sign": [("(float)(h - p->pad + i)", "(float)(h + p->pad + i)")],
    "mask_dropped": [("acc += wt * m * s;", "acc += wt * s;")],
    "bias_dropped": [("out[o * out_stride] = acc + (p->bias ? (double)p->bias[o] : 0.0);",
                      "out[o * out_stride] = acc;")],
    "border_off_by_one": [("yy <= p->H - 1", "yy <= p->H - 2")],
    "corner_step_wrong": [("const double xx = (double)fx0 + e;", "const double xx = (double)fx0 + 2 * e;")],
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
        text = text.replace(old, new)
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
