"""Randomised Hadamard rotation (oracle; test infrastructure only).

Sources:
  * AdapTQ page ("Shrinking the LLM KV Cache by 8x on CPU"), section "The Math
    Fix: Hadamard Accelerated Rotation (HAR)": a random sign flip followed by a
    Fast Walsh-Hadamard Transform spreads an outlier's energy over all
    dimensions; the transform uses additions and subtractions only.
  * VeloxQuant-MLX page ("I Ported a Google Research Paper to Apple Silicon"),
    section "Stage 1: Random Rotation": the preconditioner multiplies by a
    Rademacher (+1/-1) diagonal, applies the Walsh-Hadamard transform and divides
    by sqrt(d); it is selected for power-of-two head dimensions.

Reading taken: signs first, then the transform, then 1/sqrt(d), i.e.
    R = H diag(s) / sqrt(d),
which is what the VeloxQuant code listing computes (the prose formula on that
page puts the transform first; either order is orthogonal).  H is the Sylvester
Hadamard matrix, H[i, j] = (-1)^popcount(i & j); it is symmetric and H H = d I,
so R^T = diag(s) H / sqrt(d) undoes the rotation.
"""
from __future__ import annotations

import math

import numpy as np


def fwht(x: np.ndarray) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform along the last axis, float64.

    Butterfly form: at stride h, each pair (a, b) = (x[i], x[i+h]) with bit h of i
    clear becomes (a + b, a - b).  This is H x for the Sylvester H."""
    y = np.array(x, dtype=np.float64, copy=True)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("length must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(*lead, d // (2 * h), 2, h)
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(*lead, d)
        h *= 2
    return y


def sylvester(d: int) -> np.ndarray:
    """Dense Sylvester Hadamard matrix of order d (int64), by the doubling
    H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]].  Used by tests only."""
    h = np.ones((1, 1), dtype=np.int64)
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate(x: np.ndarray, s: np.ndarray) -> np.ndarray:
    """x~ = H (s * x) / sqrt(d), float64, along the last axis."""
    d = np.shape(x)[-1]
    return fwht(np.asarray(s, dtype=np.float64) * np.asarray(x, dtype=np.float64)) / math.sqrt(d)


def unrotate(y: np.ndarray, s: np.ndarray) -> np.ndarray:
    """x = s * (H y) / sqrt(d), the inverse (= transpose) of ``rotate``."""
    d = np.shape(y)[-1]
    return np.asarray(s, dtype=np.float64) * fwht(y) / math.sqrt(d)
