"""The single-scale sampling backward oracle against its pins, and planted
mistakes in a copy of its source against the same pins (CPU only)."""

import os

import pytest

import oracle
from tests import pins_attn_backward as pins


@pytest.mark.parametrize("pin", pins.ALL_ATTN_BACKWARD_PINS, ids=lambda p: p.__name__)
def test_attn_backward_pin(pin):
    pin(oracle.get())


# each edit is applied once, inside oracle_attn_backward
MUTANTS = {
    "derivative_sign_flipped": [("const double dsgn[2] = {-1.0, 1.0};", "const double dsgn[2] = {1.0, -1.0};")],
    "offset_axes_swapped": [("gofs[0] = a[k] * g_y;", "gofs[0] = a[k] * g_x;"),
                            ("gofs[1] = a[k] * g_x;", "gofs[1] = a[k] * g_y;")],
    "offset_without_weight": [("gofs[0] = a[k] * g_y;", "gofs[0] = g_y;")],
    "softmax_not_centred": [("gw[k] = a[k] * (ga[k] - s_ag);", "gw[k] = a[k] * ga[k];")],
    "value_without_weight": [("const double s = a[k] * rw[ay] * cwx[ex];", "const double s = rw[ay] * cwx[ex];")],
    "dy_with_row_weight": [("g_y += dsgn[ay] * cwx[ex] * dot;", "g_y += dsgn[ay] * rw[ay] * dot;")],
    "grad_a_without_column_weight": [("g_a += rw[ay] * cwx[ex] * dot;", "g_a += rw[ay] * dot;")],
    "value_to_wrong_group": [("(((size_t)b * H + (size_t)yy) * W + (size_t)xx) * G + g;",
                              "(((size_t)b * H + (size_t)yy) * W + (size_t)xx) * G + (G - 1 - g);")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_attn_backward_mutant_is_caught(tmp_path, name):
    with open(oracle.ATTN_SOURCE) as fh:
        text = fh.read()
    cut = text.index("int oracle_attn_backward(")
    head, body = text[:cut], text[cut:]
    for old, new in MUTANTS[name]:
        assert body.count(old) == 1, f"mutation anchor not unique in the backward: {old!r}"
        body = body.replace(old, new, 1)
    src = os.path.join(tmp_path, f"{name}.c")
    lib = os.path.join(tmp_path, f"{name}.so")
    with open(src, "w") as fh:
        fh.write(head + body)
    oracle.compile_oracle(oracle.SOURCE, lib, extra=(oracle.MSDA_SOURCE, src))
    mutant = oracle.Oracle(lib, oracle.SOURCE)
    caught = []
    for pin in pins.ALL_ATTN_BACKWARD_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every single-scale backward pin"
