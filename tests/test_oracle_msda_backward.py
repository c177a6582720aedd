"""The MSDA backward oracle against its pins, and planted mistakes in a
copy of its source against the same pins (CPU only)."""

import os

import pytest

import oracle
from tests import pins_msda_backward as pins


@pytest.mark.parametrize("pin", pins.ALL_MSDA_BACKWARD_PINS, ids=lambda p: p.__name__)
def test_msda_backward_pin(pin):
    pin(oracle.get())


# each edit is applied once, inside oracle_msda_backward
MUTANTS = {
    "dx_sign_flipped": [("const double sgn[2] = {-1.0, 1.0};", "const double sgn[2] = {1.0, -1.0};")],
    "loc_unscaled": [("gl[0] = a[t] * g_px * (double)W;", "gl[0] = a[t] * g_px;")],
    "loc_axes_swapped": [("gl[0] = a[t] * g_px * (double)W;", "gl[0] = a[t] * g_py * (double)H;"),
                         ("gl[1] = a[t] * g_py * (double)H;", "gl[1] = a[t] * g_px * (double)W;")],
    "loc_without_attention": [("gl[0] = a[t] * g_px * (double)W;", "gl[0] = g_px * (double)W;")],
    "softmax_not_centred": [("gw[t] = a[t] * (ga[t] - s_ag);", "gw[t] = a[t] * ga[t];")],
    "softmax_ignored": [("gw[t] = a[t] * (ga[t] - s_ag);", "gw[t] = ga[t];")],
    "value_without_attention": [("const double cw = a[t] * wy[ay] * wx[ex];",
                                 "const double cw = wy[ay] * wx[ex];")],
    "dpx_with_x_weight": [("g_px += wy[ay] * sgn[ex] * dot;", "g_px += wx[ex] * sgn[ex] * dot;")],
    "grad_a_without_row_weight": [("g_a += wy[ay] * wx[ex] * dot;", "g_a += wx[ex] * dot;")],
    "value_to_wrong_head": [("double *gv = grad_value + (((size_t)b * S + s) * G + g) * D;",
                             "double *gv = grad_value + (((size_t)b * S + s) * G + (G - 1 - g)) * D;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_msda_backward_mutant_is_caught(tmp_path, name):
    with open(oracle.MSDA_SOURCE) as fh:
        text = fh.read()
    start = text.index("int oracle_msda_backward(")
    head, body = text[:start], text[start:]
    for old, new in MUTANTS[name]:
        assert body.count(old) == 1, f"mutation anchor not unique in the backward: {old!r}"
        body = body.replace(old, new, 1)
    src = os.path.join(tmp_path, f"{name}.c")
    lib = os.path.join(tmp_path, f"{name}.so")
    with open(src, "w") as fh:
        fh.write(head + body)
    oracle.compile_oracle(oracle.SOURCE, lib, extra=(src,))
    mutant = oracle.Oracle(lib, oracle.SOURCE)
    caught = []
    for pin in pins.ALL_MSDA_BACKWARD_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every MSDA backward pin"
