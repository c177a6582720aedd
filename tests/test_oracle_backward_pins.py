"""The oracle's backward pass against its pins (CPU only)."""

import pytest

import oracle
from tests import pins_backward


@pytest.mark.parametrize("pin", pins_backward.ALL_BACKWARD_PINS, ids=lambda p: p.__name__)
def test_backward_pin(pin):
    pin(oracle.get())


def test_points_variant_matches_full():
    pins_backward.check_points_match_full(oracle.get())
