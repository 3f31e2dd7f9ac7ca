"""Derives the coefficients of the cubic in exp2_poly.cuh.

Remez exchange for the polynomial p of a given degree that minimises the
maximum RELATIVE error |p(f) / 2^f - 1| over f in [0, 1]:

  1. Start from the Chebyshev extrema mapped to [0, 1] (degree + 2 points).
  2. Solve the linear system p(x_i) - 2^x_i = (-1)^i E 2^x_i for the
     coefficients and the levelled error E.
  3. Move the reference to the extrema of the new error curve (found on a
     fine grid and refined by a parabola through three samples).
  4. Repeat until the reference stops moving.

float64 is ample for a cubic on [0, 1].  Run as a script to print the fp32
hex constants; tests/test_exp2_poly.py calls fit() to check the header.
"""
from __future__ import annotations

import numpy as np


def fit(degree: int = 3, iters: int = 40, grid: int = 200001):
    n = degree + 2
    xs = 0.5 * (1.0 - np.cos(np.pi * np.arange(n) / (n - 1)))
    g = np.linspace(0.0, 1.0, grid)
    coef = err = None
    for _ in range(iters):
        f = np.exp2(xs)
        a = np.zeros((n, n))
        a[:, :degree + 1] = xs[:, None] ** np.arange(degree + 1)
        a[:, degree + 1] = -((-1.0) ** np.arange(n)) * f
        sol = np.linalg.solve(a, f)
        coef, err = sol[:degree + 1], sol[degree + 1]
        e = np.polyval(coef[::-1], g) / np.exp2(g) - 1.0
        # interior extrema where the slope changes sign, plus both ends
        k = np.where(np.diff(np.sign(np.diff(e))) != 0)[0] + 1
        new = [0.0]
        for i in k:
            y0, y1, y2 = e[i - 1], e[i], e[i + 1]
            den = y0 - 2 * y1 + y2
            shift = 0.5 * (y0 - y2) / den if den != 0 else 0.0
            new.append(g[i] + shift * (g[1] - g[0]))
        new.append(1.0)
        if len(new) != n:
            break
        new = np.array(new)
        if np.max(np.abs(new - xs)) < 1e-12:
            xs = new
            break
        xs = new
    return coef, abs(err)


def fp32_hex(x: float) -> str:
    """C hex-float literal of x rounded to fp32."""
    h = float(np.float32(x)).hex()           # e.g. 0x1.fff6320000000p-1
    mant, exp = h.split("p")
    mant = mant.rstrip("0")
    if mant.endswith("."):
        mant = mant[:-1]
    return f"{mant}p{exp}f"


if __name__ == "__main__":
    for deg in (3, 4, 5):
        c, e = fit(deg)
        print(f"degree {deg}: max relative error {e:.3e} (2^{np.log2(e):.2f})")
        print("  " + ", ".join(fp32_hex(x) for x in c))
