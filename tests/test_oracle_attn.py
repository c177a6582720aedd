"""The single-scale deformable sampling oracle against its pins, and
planted mistakes in a copy of its source against the same pins (CPU only)."""

import os

import pytest

import oracle
from tests import pins_attn


@pytest.mark.parametrize("pin", pins_attn.ALL_ATTN_PINS, ids=lambda p: p.__name__)
def test_attn_pin(pin):
    pin(oracle.get())


MUTANTS = {
    "dy_dx_swapped": [("i * dh) + orow[2 * k];", "i * dh) + orow[2 * k + 1];"),
                      ("j * dw) + orow[2 * k + 1];", "j * dw) + orow[2 * k];")],
    "stride_ignored": [("(float)(ho * sh - ph + i * dh)", "(float)(ho - ph + i * dh)")],
    "dilation_ignored": [("(float)(wo * sw - pw + j * dw)", "(float)(wo * sw - pw + j)")],
    "padding_sign": [("(float)(ho * sh - ph + i * dh)", "(float)(ho * sh + ph + i * dh)")],
    "taps_column_major": [("const int i = k / kw, j = k % kw;", "const int i = k % kh, j = k / kh;")],
    "softmax_unnormalised": [("for (int k = 0; k < K; ++k) a[k] /= wsum;", "")],
    "x_weights_swapped": [("const double wx[2] = {1.0 - lx, lx};", "const double wx[2] = {lx, 1.0 - lx};")],
    "group_ignored": [("* W + (size_t)xx) * G + g) * D;", "* W + (size_t)xx) * G) * D;")],
    "border_off_by_one": [("xx <= W - 1)) continue;", "xx < W - 1)) continue;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_attn_mutant_is_caught(tmp_path, name):
    with open(oracle.ATTN_SOURCE) as fh:
        text = fh.read()
    # the edits apply to the forward only (the backward repeats some lines)
    cut = text.index("int oracle_attn_backward(")
    fwd, rest = text[:cut], text[cut:]
    for old, new in MUTANTS[name]:
        assert fwd.count(old) == 1, f"mutation anchor not unique: {old!r}"
        fwd = fwd.replace(old, new, 1)
    text = fwd + rest
    src = os.path.join(tmp_path, f"{name}.c")
    lib = os.path.join(tmp_path, f"{name}.so")
    with open(src, "w") as fh:
        fh.write(text)
    oracle.compile_oracle(oracle.SOURCE, lib, extra=(oracle.MSDA_SOURCE, src))
    mutant = oracle.Oracle(lib, oracle.SOURCE)
    caught = []
    for pin in pins_attn.ALL_ATTN_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every single-scale sampling pin"
