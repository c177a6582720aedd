"""The MSDA oracle against its pins, and planted mistakes in a copy of its
source against the same pins (CPU only)."""

import os

import pytest

import oracle
from tests import pins_msda


@pytest.mark.parametrize("pin", pins_msda.ALL_MSDA_PINS, ids=lambda p: p.__name__)
def test_msda_pin(pin):
    pin(oracle.get())


MUTANTS = {
    "xy_swapped": [("loc[0] * (float)W - 0.5f", "loc[1] * (float)W - 0.5f"),
                   ("loc[1] * (float)H - 0.5f", "loc[0] * (float)H - 0.5f")],
    "no_half_pixel": [("loc[0] * (float)W - 0.5f", "loc[0] * (float)W"),
                      ("loc[1] * (float)H - 0.5f", "loc[1] * (float)H")],
    "align_corners_scale": [("loc[0] * (float)W - 0.5f", "loc[0] * (float)(W - 1)"),
                            ("loc[1] * (float)H - 0.5f", "loc[1] * (float)(H - 1)")],
    "softmax_unnormalised": [("for (int t = 0; t < LK; ++t) a[t] /= wsum;", "")],
    "level_start_ignored": [("(size_t)starts[l] + (size_t)yy * W", "(size_t)yy * W")],
    "level_shape_swapped": [("const int H = shapes[2 * l], W = shapes[2 * l + 1];\n                for",
                             "const int W = shapes[2 * l], H = shapes[2 * l + 1];\n                for")],
    "x_weights_swapped": [("const double wx[2] = {1.0 - lx, lx};", "const double wx[2] = {lx, 1.0 - lx};")],
    "head_ignored": [("* G + g) * D;", "* G) * D;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_msda_mutant_is_caught(tmp_path, name):
    with open(oracle.MSDA_SOURCE) as fh:
        text = fh.read()
    for old, new in MUTANTS[name]:
        assert old in text, f"mutation anchor not found: {old!r}"
        text = text.replace(old, new)
    src = os.path.join(tmp_path, f"{name}.c")
    lib = os.path.join(tmp_path, f"{name}.so")
    with open(src, "w") as fh:
        fh.write(text)
    oracle.compile_oracle(oracle.SOURCE, lib, extra=(src,))
    mutant = oracle.Oracle(lib, oracle.SOURCE)
    caught = []
    for pin in pins_msda.ALL_MSDA_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every MSDA pin"
