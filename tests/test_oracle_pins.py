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


def test_general_points_match_full(orc):
    s = pins.GEN_SHAPES[0]
    x, off, m, w, b = pins._rand_problem_ex(83, s, off_std=2.0)
    desc = pins._conv_desc(s)
    full = orc.forward_ex(x, off, m, w, b, desc)
    B, O, Ho, Wo = full.shape
    pts = np.array([[0, 0, 0], [1, Ho - 1, Wo - 1], [0, Ho // 2, 1], [1, 0, Wo - 1]])
    got = orc.forward_points_ex(x, off, m, w, b, desc, pts)
    for t, (bb, h, ww) in enumerate(pts):
        assert np.array_equal(got[t], full[bb, :, h, ww])


def test_general_form_reduces_to_page_form(orc):
    """Stride 1, dilation 1, one group and one offset group: the general
    entry point gives the page-1 entry point's bits."""
    x, off, m, w, b = pins._rand_problem(84, B=2, C=3, H=8, W=7, O=4, kh=3, kw=5, pad=2, off_std=2.0)
    page = orc.forward(x, off, m, w, b, 2)
    general = orc.forward_ex(x, off, m, w, b, oracle.ConvDesc(padding=2))
    assert np.array_equal(page, general)


def test_general_rejects_bad_shapes(orc):
    s = pins.GEN_SHAPES[0]
    x, off, m, w, b = pins._rand_problem_ex(85, s, off_std=1.0)
    desc = pins._conv_desc(s)
    with pytest.raises(ValueError):          # offsets of one offset group only
        orc.forward_ex(x, off[:, :off.shape[1] // 2], m, w, b, desc)
    with pytest.raises(ValueError):          # groups that do not divide C
        orc.forward_ex(x, off, m, w, b, oracle.ConvDesc(stride=2, padding=(1, 2), dilation=(1, 2),
                                                        groups=3, offset_groups=2))
