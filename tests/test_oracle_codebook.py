"""Pins for oracle/codebook.py: Lloyd-Max and uniform codebooks for N(0,1).

The Lloyd-Max solver integrates with the trapezoidal rule (VeloxQuant-MLX page,
"Stage 2"); here its result is checked against the two optimality conditions
evaluated in closed form with the error function, against the required 16-level
values, and against J. Max's 1960 tables."""
import functools
import math

import numpy as np
import pytest
from scipy.integrate import quad
from scipy.special import ndtr

from oracle import codebook
from tests.conftest import read_golden

GOLD = read_golden("lloyd_max_16.txt")


@functools.lru_cache(maxsize=None)
def lm(bits):
    return codebook.lloyd_max(bits)


def pdf(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)


def closed_form_conditional_means(bounds):
    """E[X | a < X < b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a)); outer cells end at the
    support +-8 used by the solver."""
    e = np.concatenate([[codebook.SUPPORT[0]], bounds, [codebook.SUPPORT[1]]])
    num = np.array([pdf(a) - pdf(b) for a, b in zip(e[:-1], e[1:])])
    den = ndtr(e[1:]) - ndtr(e[:-1])
    return num / den


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_lloyd_max_optimality_conditions(bits):
    c, b, _ = lm(bits)
    assert len(c) == 2 ** bits and np.all(np.diff(c) > 0)
    np.testing.assert_allclose(b, (c[:-1] + c[1:]) / 2, atol=1e-15)  # condition 1
    np.testing.assert_allclose(c, closed_form_conditional_means(b), rtol=0, atol=1e-9)  # condition 2
    np.testing.assert_allclose(c, -c[::-1], atol=1e-12)  # symmetric


def test_two_levels_closed_form():
    c, _, _ = lm(1)
    np.testing.assert_allclose(c, [-math.sqrt(2 / math.pi), math.sqrt(2 / math.pi)], atol=1e-9)


def test_sixteen_levels_required_values():
    c, _, _ = lm(4)
    assert round(c[8], 4) == float(GOLD["inner16"][0]) and round(-c[7], 4) == float(GOLD["inner16"][0])
    assert round(c[15], 4) == float(GOLD["outer16"][0]) and round(-c[0], 4) == float(GOLD["outer16"][0])


def test_textbook_levels():
    c2, _, _ = lm(2)
    c3, _, _ = lm(3)
    for got, want in zip(list(c2[2:]) + list(c3[4:]), GOLD["levels4"] + GOLD["levels8"]):
        assert abs(got - float(want)) <= _half_ulp(want)


def _half_ulp(text):
    """Half a unit of the last printed decimal of a table entry."""
    decimals = len(text.split(".")[1]) if "." in text else 0
    return 0.5 * 10.0 ** -decimals + 1e-12


def _mse_by_quad(c, b):
    e = np.concatenate([[-np.inf], b, [np.inf]])
    return sum(quad(lambda x, ci=ci: (x - ci) ** 2 * pdf(x), lo, hi, limit=200)[0]
               for ci, lo, hi in zip(c, e[:-1], e[1:]))


def test_textbook_distortion():
    for bits, want in zip((2, 3, 4), GOLD["mse"]):
        c, b, _ = lm(bits)
        assert abs(_mse_by_quad(c, b) - float(want)) <= _half_ulp(want)


def test_uniform_codebook_textbook():
    for bits, step, mse in zip((2, 3, 4), GOLD["uniform_step"], GOLD["uniform_mse"]):
        c, b, delta = codebook.uniform_codebook(bits)
        assert abs(delta - float(step)) <= _half_ulp(step)
        assert abs(_mse_by_quad(c, b) - float(mse)) <= _half_ulp(mse)
        np.testing.assert_allclose(np.diff(c), delta, rtol=1e-12)
        np.testing.assert_allclose(c, -c[::-1], atol=1e-12)


def test_uniform_two_levels_equals_lloyd_max():
    c_u, _, _ = codebook.uniform_codebook(1)
    c_l, _, _ = lm(1)
    np.testing.assert_allclose(c_u, c_l, atol=1e-6)


def test_uniform_mse_closed_form_matches_quadrature():
    for n, delta in ((4, 0.7), (8, 0.5), (16, 0.41)):
        c = (np.arange(n) - (n - 1) / 2) * delta
        b = (c[:-1] + c[1:]) / 2
        assert abs(codebook.uniform_mse(delta, n) - _mse_by_quad(c, b)) < 1e-10


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_float32_tables(bits):
    c, _, _ = lm(bits)
    c32, b32 = codebook.float32_tables(c)
    assert c32.dtype == np.float32 and b32.dtype == np.float32
    assert np.array_equal(c32, c.astype(np.float32))
    assert np.all(c32[:-1] < b32) and np.all(b32 < c32[1:])
    assert b32[len(b32) // 2] == 0.0  # symmetric table: the middle boundary is exactly 0
    # every value is assigned to its nearest centroid by counting boundaries below it
    u = np.random.default_rng(0).standard_normal(20000).astype(np.float32)
    idx = np.sum(u[:, None] > b32[None, :], axis=1)
    nearest = np.argmin(np.abs(u[:, None].astype(np.float64) - c32[None, :]), axis=1)
    assert np.array_equal(idx, nearest)
