"""The oracle checked against what the pages and mathematics fix (CPU only)."""

import numpy as np
import pytest
import torch

import oracle
from tests import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_points_match_full(orc):
    x, off, m, w, b = pins._rand_problem(80, B=2, C=3, H=7, W=6, O=4, kh=3, kw=3, pad=1, off_std=2.0)
    full = orc.forward(x, off, m, w, b, 1)
    pts = np.array([[0, 0, 0], [1, 6, 5], [0, 3, 2], [1, 0, 5], [1, 6, 0]])
    got = orc.forward_points(x, off, m, w, b, 1, pts)
    for t, (bb, h, ww) in enumerate(pts):
        assert np.array_equal(got[t], full[bb, :, h, ww])


def test_thread_count_does_not_change_bits(orc):
    x, off, m, w, b = pins._rand_problem(81, B=2, C=5, H=9, W=8, O=3, kh=3, kw=3, pad=1, off_std=3.0)
    one = orc.forward(x, off, m, w, b, 1, nthreads=1)
    many = orc.forward(x, off, m, w, b, 1, nthreads=4)
    assert np.array_equal(one, many)


def test_rejects_bad_shapes(orc):
    x, off, m, w, b = pins._rand_problem(82, B=1, C=2, H=5, W=5, O=2, kh=3, kw=3, pad=1, off_std=1.0)
    with pytest.raises(ValueError):
        orc.forward(x, off[:, :4], m, w, b, 1)
    with pytest.raises(ValueError):
        orc.forward_points(x, off, m, w, b, 1, np.array([[0, 5, 0]]))
