"""Fit the polynomial of the forward kernel's FMA-pipe exponential, 2^f on [-1/2, 1/2].

Method: Remez exchange for the minimax *relative* error of a degree-3 polynomial p(f) ≈ 2^f
(equioscillation of (p(f) - 2^f) / 2^f at 5 points), in float64, then every coefficient
rounded to the nearest float32.  The kernel evaluates 2^x as 2^j · p(x - j) with j the
integer nearest x (Cody–Waite-style range reduction with one constant: j is exact, so the
reduced argument x - j is exact in float32 too).

    python fit_exp2_poly.py          # prints the coefficients and the error of both forms

The printed float32 coefficients are the ones in fwd_tc.cuh; tests/test_exp2_poly_cpu.py
re-runs this fit and checks that they agree and that the bound holds.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def _solve(nodes):
    """Coefficients c (c0..cD) and level E with (p(x) - 2^x) = (-1)^k E 2^x at the nodes."""
    n = DEGREE + 2
    a = np.zeros((n, n))
    b = np.exp2(nodes)
    for k, x in enumerate(nodes):
        a[k, : DEGREE + 1] = x ** np.arange(DEGREE + 1)
        a[k, DEGREE + 1] = -((-1) ** k) * np.exp2(x)
    sol = np.linalg.solve(a, b)
    return sol[: DEGREE + 1], sol[DEGREE + 1]


def rel_err(c, x):
    return np.polynomial.polynomial.polyval(x, c) / np.exp2(x) - 1.0


def remez(iters: int = 30):
    # start from Chebyshev extrema
    k = np.arange(DEGREE + 2)
    nodes = (LO + HI) / 2 + (HI - LO) / 2 * np.cos(np.pi * k[::-1] / (DEGREE + 1))
    grid = np.linspace(LO, HI, 200001)
    c = None
    for _ in range(iters):
        c, _level = _solve(nodes)
        e = rel_err(c, grid)
        # new nodes: the extrema of e on each interval between sign changes
        sign = np.sign(e)
        cuts = np.flatnonzero(np.diff(sign) != 0) + 1
        pieces = np.split(np.arange(grid.size), cuts)
        ext = [p[np.argmax(np.abs(e[p]))] for p in pieces]
        if len(ext) != DEGREE + 2:
            break
        new = grid[ext]
        if np.max(np.abs(new - nodes)) < 1e-12:
            nodes = new
            break
        nodes = new
    return c


def coefficients_f32():
    return np.asarray(remez(), dtype=np.float32)


def max_rel_err_f32(c32, samples: int = 1 << 20):
    """Largest relative error of the float32 polynomial (evaluated in float64) on the range."""
    x = np.linspace(LO, HI, samples)
    return float(np.max(np.abs(rel_err(c32.astype(np.float64), x))))


if __name__ == "__main__":
    c64 = remez()
    c32 = c64.astype(np.float32)
    print("float64 coefficients:", ", ".join(f"{v:.17g}" for v in c64))
    print("float32 coefficients:", ", ".join(f"{float(v):.9g}f" for v in c32))
    print("hex:", ", ".join(hex(int(np.float32(v).view(np.uint32))) for v in c32))
    print(f"max relative error, float64 coefficients: {np.max(np.abs(rel_err(c64, np.linspace(LO, HI, 1 << 20)))):.3e}")
    print(f"max relative error, float32 coefficients: {max_rel_err_f32(c32):.3e}")
