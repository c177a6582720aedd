"""Planted mistakes in a copy of the oracle's backward pass must each fail
at least one backward pin (a flipped or transposed derivative, the mask
dropped from one gradient or added to another, the offset channels
swapped, the column gradient summed over the wrong outputs, a transposed
corner in the scatter, images dropped from the weight and bias sums).
Every mutant stays inside its arrays; they run on the CPU only."""

import os

import pytest

import oracle
from tests import pins_backward

MUTANTS = {
    "dsdy_sign": [("s_y += (a ? 1.0 : -1.0) * wx[e] * v;", "s_y += (a ? -1.0 : 1.0) * wx[e] * v;")],
    "dsdy_uses_wy": [("s_y += (a ? 1.0 : -1.0) * wx[e] * v;", "s_y += (a ? 1.0 : -1.0) * wy[a] * v;")],
    "dsdx_uses_wx": [("s_x += (e ? 1.0 : -1.0) * wy[a] * v;", "s_x += (e ? 1.0 : -1.0) * wx[e] * v;")],
    "offset_channels_swapped": [
        ("goff[(ptrdiff_t)(q * 2 * k_total + 2 * k) * stride] = g_dy;",
         "goff[(ptrdiff_t)(q * 2 * k_total + 2 * k) * stride] = g_dx;"),
        ("goff[(ptrdiff_t)(q * 2 * k_total + 2 * k + 1) * stride] = g_dx;",
         "goff[(ptrdiff_t)(q * 2 * k_total + 2 * k + 1) * stride] = g_dy;")],
    "grad_x_mask_dropped": [("+= ga * m * wy[a] * wx[e];", "+= ga * wy[a] * wx[e];")],
    "grad_weight_mask_dropped": [("gw[wi] += gov * m * s;", "gw[wi] += gov * s;")],
    "grad_mask_times_mask": [("g_m += ga * s;", "g_m += ga * m * s;")],
    "grad_offset_mask_dropped": [("g_dy += ga * m * s_y;", "g_dy += ga * s_y;"),
                                 ("g_dx += ga * m * s_x;", "g_dx += ga * s_x;")],
    "column_grad_wrong_outputs": [("for (int o = g * Og; o < (g + 1) * Og; ++o) {\n"
                                   "                        const double gov",
                                   "for (int o = 0; o < Og; ++o) {\n"
                                   "                        const double gov")],
    "grad_x_corner_transposed": [("+= ga * m * wy[a] * wx[e];", "+= ga * m * wy[e] * wx[a];")],
    "weight_sum_last_image": [("for (int b = 0; b < p.B; ++b) acc += part[(size_t)b * per_image + t];",
                               "acc = part[(size_t)(p.B - 1) * per_image + t];")],
    "bias_sum_first_image": [("for (int b = 0; b < p.B; ++b) acc += part[(size_t)b * per_image + n_w + o];",
                              "acc = part[n_w + o];")],
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as fh:
        return fh.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_backward_mutant_is_caught(tmp_path, source, name):
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
    for pin in pins_backward.ALL_BACKWARD_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every backward pin"
