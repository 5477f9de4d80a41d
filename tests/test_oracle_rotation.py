"""Pins for oracle/rotation.py: the randomised Hadamard rotation.

Checked against facts that do not come from the oracle: scipy's Hadamard
matrix, the Sylvester doubling H H = d I, closed forms for basis vectors, and
the orthogonality the AdapTQ and VeloxQuant-MLX pages rely on."""
import math

import numpy as np
import pytest
import scipy.linalg

from oracle import rotation

DIMS = [1, 2, 4, 8, 16, 32, 64, 128, 256]


@pytest.mark.parametrize("d", DIMS)
def test_sylvester_is_hadamard(d):
    h = rotation.sylvester(d)
    assert np.array_equal(h @ h, d * np.eye(d, dtype=np.int64))  # exact, integers
    assert np.array_equal(h, h.T)
    assert np.array_equal(h, scipy.linalg.hadamard(d))


@pytest.mark.parametrize("d", DIMS)
def test_fwht_matches_library_matrix(d):
    x = np.random.default_rng(d).standard_normal((5, d))
    ref = x @ scipy.linalg.hadamard(d).T
    np.testing.assert_allclose(rotation.fwht(x), ref, rtol=0, atol=1e-12 * d)


@pytest.mark.parametrize("d", [8, 128, 256])
def test_fwht_closed_forms(d):
    e0 = np.zeros(d); e0[0] = 1
    assert np.array_equal(rotation.fwht(e0), np.ones(d))
    assert np.array_equal(rotation.fwht(np.ones(d)), d * e0)
    k = d // 2 + 3 if d > 4 else 1
    ek = np.zeros(d); ek[k] = 1
    col = np.array([(-1) ** bin(i & k).count("1") for i in range(d)], dtype=float)
    assert np.array_equal(rotation.fwht(ek), col)


@pytest.mark.parametrize("d", [128, 256])
def test_rotation_is_orthogonal(d):
    rng = np.random.default_rng(7)
    s = np.where(rng.integers(0, 2, d) == 0, 1, -1)
    x = rng.standard_normal((64, d))
    y = rng.standard_normal((64, d))
    rx, ry = rotation.rotate(x, s), rotation.rotate(y, s)
    np.testing.assert_allclose(np.linalg.norm(rx, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    np.testing.assert_allclose(np.sum(rx * ry, axis=1), np.sum(x * y, axis=1), rtol=0, atol=1e-10)
    np.testing.assert_allclose(rotation.unrotate(rx, s), x, rtol=0, atol=1e-12)
    # fp32 norms preserved to 1e-6 relative as well
    rx32 = rotation.rotate(x.astype(np.float32), s).astype(np.float32)
    rel = np.abs(np.linalg.norm(rx32, axis=1) / np.linalg.norm(x.astype(np.float32), axis=1) - 1)
    assert rel.max() < 1e-6


@pytest.mark.parametrize("d", [128, 256])
def test_signs_applied_before_transform(d):
    """R e_j = s_j H e_j / sqrt(d): the sign of coordinate j multiplies column j.  (If the
    transform came first the signs would multiply the rows instead.)"""
    rng = np.random.default_rng(3)
    s = np.where(rng.integers(0, 2, d) == 0, 1, -1)
    h = scipy.linalg.hadamard(d)
    for j in (0, 5, d - 1):
        e = np.zeros(d); e[j] = 1
        np.testing.assert_allclose(rotation.rotate(e, s), s[j] * h[:, j] / math.sqrt(d), atol=1e-15)


def test_outlier_is_spread_evenly():
    """AdapTQ page, "The Math Fix": the rotation smears one large coordinate over all of
    them -- a one-hot vector of size A becomes d coordinates of magnitude A / sqrt(d)."""
    d, amp = 128, 50.0
    s = np.where(np.random.default_rng(1).integers(0, 2, d) == 0, 1, -1)
    x = np.zeros(d); x[17] = amp
    np.testing.assert_allclose(np.abs(rotation.rotate(x, s)), amp / math.sqrt(d), rtol=1e-14)
