"""Scalar codebooks for the rotated, unit-norm coordinates (oracle; test infrastructure).

Source: VeloxQuant-MLX page ("I Ported a Google Research Paper to Apple
Silicon"), sections "The Core Idea: Why KV Vectors Can Be Compressed" and
"Stage 2: Lloyd-Max Scalar Quantization":
  1. optimal boundaries sit at the midpoints of neighbouring centroids;
  2. each centroid is the conditional mean of the density over its cell,
     c_i = int x f(x) dx / int f(x) dx over [b_{i-1}, b_i];
  the solver starts from evenly spaced centroids over the support, alternates
  the two conditions and integrates numerically with the trapezoidal rule until
  the centroids stop moving.

Readings taken (the page leaves them open):
  * density f = standard normal, support [-8, 8] (the outer cells end there);
  * "b-bit" means 2^b levels (the page's MSE variant), as the 16 centroids
    +-0.1284 .. +-2.7326 of a 4-bit table require;
  * iterate until max |change| < 1e-13 instead of the page's 100-iteration /
    1e-8 default, which stops before the 16-level table is settled to 4 decimals;
  * quadrature: composite trapezoid on a fixed grid of step 2^-17 over the support;
    each cell uses the grid nodes strictly inside it plus its two end points.
  * "uniform b-bit codes": symmetric levels c_i = (i - (n-1)/2) * delta, the step
    delta minimising the N(0,1) mean squared error (the root of its derivative),
    boundaries at midpoints.

Tables handed to the quantiser are float32: C32 = fp32(c) and the decision
boundaries Bd32_i = fp32((C32_i + C32_{i+1}) / 2), computed from the float32
centroids so that "nearest centroid" and "count of boundaries below" agree.
"""
from __future__ import annotations

import math
from typing import Tuple

import numpy as np
from scipy.special import ndtr

SUPPORT = (-8.0, 8.0)
GRID_STEP = 2.0 ** -17


def normal_pdf(x):
    return np.exp(-0.5 * np.asarray(x, dtype=np.float64) ** 2) / math.sqrt(2.0 * math.pi)


def _cell_trapezoid(g, gnode, x, edges, step):
    """Composite trapezoid of g over each cell [edges[i], edges[i+1]] using the fixed grid
    nodes x strictly inside the cell plus the two edge points.  gnode = g(x)."""
    n_nodes = len(x)
    lo = x[0]
    # first node strictly greater than each inner edge
    k = np.floor((edges[1:-1] - lo) / step).astype(np.int64) + 1
    first = np.concatenate([[0], k])  # first node of each cell
    last = np.concatenate([k - 1, [n_nodes - 1]])  # last node of each cell
    inner_sum = np.add.reduceat(gnode, first)
    # nodes first..last: trapezoid over equal panels = h * (sum - (g_first + g_last)/2)
    inner = step * inner_sum - 0.5 * step * (gnode[first] + gnode[last])
    left = (x[first] - edges[:-1]) * (g(edges[:-1]) + gnode[first]) / 2.0
    right = (edges[1:] - x[last]) * (gnode[last] + g(edges[1:])) / 2.0
    return inner + left + right


def lloyd_max(bits: int, tol: float = 1e-13, max_iter: int = 100000) -> Tuple[np.ndarray, np.ndarray, int]:
    """Lloyd-Max centroids and boundaries (float64) for N(0,1) with 2^bits levels.
    Returns (centroids, boundaries, iterations)."""
    lo, hi = SUPPORT
    n = 2 ** bits
    n_panels = int(round((hi - lo) / GRID_STEP))
    x = lo + GRID_STEP * np.arange(n_panels + 1, dtype=np.float64)
    f = normal_pdf(x)
    xf = x * f

    def g0(t):
        return normal_pdf(t)

    def g1(t):
        return np.asarray(t) * normal_pdf(t)

    c = np.linspace(lo, hi, n)  # evenly spaced start over the support
    for it in range(1, max_iter + 1):
        b = (c[:-1] + c[1:]) / 2.0  # condition 1: boundaries at midpoints
        edges = np.concatenate([[lo], b, [hi]])
        mass = _cell_trapezoid(g0, f, x, edges, GRID_STEP)
        moment = _cell_trapezoid(g1, xf, x, edges, GRID_STEP)
        new = moment / mass  # condition 2: conditional mean over each cell
        moved = np.max(np.abs(new - c))
        c = new
        if moved < tol:
            return c, (c[:-1] + c[1:]) / 2.0, it
    raise RuntimeError("Lloyd-Max did not converge")


def uniform_mse(delta: float, n: int) -> float:
    """Mean squared error of the symmetric uniform quantiser with n levels and step delta
    on N(0,1), in closed form: per cell [a, b] with level c,
    int (x - c)^2 phi = (1 + c^2)(Phi(b) - Phi(a)) + (a - 2c) phi(a) - (b - 2c) phi(b)."""
    c = (np.arange(n) - (n - 1) / 2.0) * delta
    edges = np.concatenate([[-np.inf], (c[:-1] + c[1:]) / 2.0, [np.inf]])
    a, b = edges[:-1], edges[1:]
    pa = np.where(np.isfinite(a), normal_pdf(np.where(np.isfinite(a), a, 0.0)), 0.0)
    pb = np.where(np.isfinite(b), normal_pdf(np.where(np.isfinite(b), b, 0.0)), 0.0)
    at = np.where(np.isfinite(a), a, 0.0)
    bt = np.where(np.isfinite(b), b, 0.0)
    cell = (1.0 + c * c) * (ndtr(b) - ndtr(a)) + (at - 2 * c) * pa - (bt - 2 * c) * pb
    return float(np.sum(cell))


def uniform_mse_slope(delta: float, n: int) -> float:
    """d MSE / d delta of the symmetric uniform quantiser, in closed form.  With level
    c_i = k_i delta (k_i = i - (n-1)/2) on cell [a_i, b_i], the boundary terms of the
    derivative cancel (midpoints are equidistant from both levels), leaving
    -2 sum_i k_i [ phi(a_i) - phi(b_i) - k_i delta (Phi(b_i) - Phi(a_i)) ]."""
    k = np.arange(n) - (n - 1) / 2.0
    a = np.where(np.arange(n) == 0, -np.inf, (k - 0.5) * delta)
    b = np.where(np.arange(n) == n - 1, np.inf, (k + 0.5) * delta)
    pa = np.where(np.isfinite(a), normal_pdf(np.where(np.isfinite(a), a, 0.0)), 0.0)
    pb = np.where(np.isfinite(b), normal_pdf(np.where(np.isfinite(b), b, 0.0)), 0.0)
    return float(-2.0 * np.sum(k * (pa - pb - k * delta * (ndtr(b) - ndtr(a)))))


def uniform_codebook(bits: int) -> Tuple[np.ndarray, np.ndarray, float]:
    """Symmetric uniform levels with the MSE-optimal step: the root of d MSE / d delta,
    found by bisection (the slope is negative below the optimum and positive above).
    Returns (centroids, boundaries, delta)."""
    n = 2 ** bits
    lo, hi = 1e-3, 2.0 * 8.0 / max(1, n - 1)
    assert uniform_mse_slope(lo, n) < 0 < uniform_mse_slope(hi, n)
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if uniform_mse_slope(mid, n) < 0:
            lo = mid
        else:
            hi = mid
    delta = 0.5 * (lo + hi)
    c = (np.arange(n) - (n - 1) / 2.0) * delta
    return c, (c[:-1] + c[1:]) / 2.0, delta


def float32_tables(centroids: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """(C32, Bd32): float32 centroids and float32 midpoints of neighbouring C32 values."""
    c32 = np.asarray(centroids, dtype=np.float64).astype(np.float32)
    mid = (c32[:-1].astype(np.float64) + c32[1:].astype(np.float64)) / 2.0
    return c32, mid.astype(np.float32)


def tables(kind: str, bits: int) -> Tuple[np.ndarray, np.ndarray]:
    """float32 (centroids, boundaries) of the named codebook ("lloyd_max" | "uniform")."""
    if kind == "lloyd_max":
        c, _, _ = lloyd_max(bits)
    elif kind == "uniform":
        c, _, _ = uniform_codebook(bits)
    else:
        raise ValueError(kind)
    return float32_tables(c)
