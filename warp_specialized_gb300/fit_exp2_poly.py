"""Fits the polynomial behind the forward kernel's optional FMA-pipe
exponential (`ATTN_OPT_EXP2_FMA`): p(f) ~ 2^f on [-1/2, 1/2], degree 3,
minimising the largest relative error |p(f) / 2^f - 1| by the Remez
exchange algorithm (Remez, 1934; as in Cheney, Introduction to Approximation
Theory, ch. 3).

The kernel splits x = n + f with n = round(x) (Cody and Waite's argument
reduction, done by adding and subtracting 1.5 * 2^23) and adds n to the
exponent field of p(f).  Run this file to print the coefficients (c0..c3,
lowest degree first) that `attn_fwd_kernel.cuh` carries, rounded to fp32,
and the error they reach.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def _solve(nodes: np.ndarray) -> tuple[np.ndarray, float]:
    """Coefficients c and level E with (p(x_i) - 2^x_i) / 2^x_i = (-1)^i E
    at the DEGREE + 2 nodes."""
    n = len(nodes)
    a = np.zeros((n, n))
    for i, x in enumerate(nodes):
        w = 2.0 ** x
        a[i, :DEGREE + 1] = [x ** k / w for k in range(DEGREE + 1)]
        a[i, DEGREE + 1] = -((-1.0) ** i)
    sol = np.linalg.solve(a, np.ones(n))
    return sol[:DEGREE + 1], float(sol[DEGREE + 1])


def rel_err(c: np.ndarray, x: np.ndarray) -> np.ndarray:
    p = np.polynomial.polynomial.polyval(x, c)
    return p / 2.0 ** x - 1.0


def fit(iters: int = 30) -> tuple[np.ndarray, float]:
    """Remez exchange: start from Chebyshev extrema, move each node to the
    local extremum of the error between sign changes, until the levels
    equalise."""
    k = np.arange(DEGREE + 2)
    nodes = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * (DEGREE + 1 - k) / (DEGREE + 1))
    grid = np.linspace(LO, HI, 200001)
    c = np.zeros(DEGREE + 1)
    for _ in range(iters):
        c, _ = _solve(nodes)
        e = rel_err(c, grid)
        # one extremum per run of equal sign
        sign = np.sign(e)
        bounds = np.flatnonzero(np.diff(sign) != 0) + 1
        runs = np.split(np.arange(len(grid)), bounds)
        ext = [r[np.argmax(np.abs(e[r]))] for r in runs if len(r)]
        if len(ext) < DEGREE + 2:
            break
        ext = np.array(ext)
        # keep DEGREE + 2 alternating extrema holding the largest errors
        while len(ext) > DEGREE + 2:
            drop = 0 if abs(e[ext[0]]) < abs(e[ext[-1]]) else len(ext) - 1
            ext = np.delete(ext, drop)
        nodes = grid[ext]
    return c, float(np.max(np.abs(rel_err(c, grid))))


def coefficients_f32() -> np.ndarray:
    c, _ = fit()
    return c.astype(np.float32)


if __name__ == "__main__":
    c, err = fit()
    c32 = c.astype(np.float32)
    grid = np.linspace(LO, HI, 200001)
    print("coefficients (c0..c3):", ", ".join(f"{float(v):.9g}f" for v in c32))
    print(f"max relative error: {err:.3e} (fp64 coefficients), "
          f"{np.max(np.abs(rel_err(c32.astype(np.float64), grid))):.3e} (fp32 coefficients)")
