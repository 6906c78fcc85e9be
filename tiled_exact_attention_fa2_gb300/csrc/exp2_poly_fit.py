"""Fit the polynomial used by the kernels' FMA-pipe exp2 (run: python exp2_poly_fit.py).

2^x is computed as 2^j * 2^f with j = round(x) and f = x - j in [-1/2, 1/2]
(Cody-Waite range reduction, Cody & Waite, "Software Manual for the
Elementary Functions", 1980).  2^f is approximated by a polynomial whose
coefficients minimise the maximum *relative* error on [-1/2, 1/2]; they are
found with the Remez exchange algorithm (Remez 1934) on the equioscillation
conditions  p(f_i) - 2^f_i = (-1)^i E 2^f_i.  The constant term is pinned
to 1 so that 2^0 is exact.

Prints the coefficients (c1..cn of 1 + c1 f + c2 f^2 + ...) and the maximum
relative error of the fp64 polynomial and of its fp32 Horner evaluation.
"""
import numpy as np


def remez_exp2(degree: int, lo: float = -0.5, hi: float = 0.5, iters: int = 30):
    n = degree  # unknowns c1..cn plus E
    # initial reference: Chebyshev extrema
    k = np.arange(n + 1)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * (n - k) / n)
    for _ in range(iters):
        # p(x) = 1 + sum c_k x^k ; require 1 + sum c_k x_i^k - 2^x_i = (-1)^i E 2^x_i
        A = np.zeros((n + 1, n + 1))
        for i, xi in enumerate(x):
            A[i, :n] = [xi ** (p + 1) for p in range(n)]
            A[i, n] = -((-1) ** i) * 2.0 ** xi
        b = 2.0 ** x - 1.0
        sol = np.linalg.solve(A, b)
        c = sol[:n]
        grid = np.linspace(lo, hi, 200001)
        err = (1 + sum(c[p] * grid ** (p + 1) for p in range(n))) / 2.0 ** grid - 1
        # new reference: extrema of the error between sign changes
        idx = [0]
        for i in range(1, len(grid) - 1):
            if (err[i] - err[i - 1]) * (err[i + 1] - err[i]) <= 0:
                idx.append(i)
        idx.append(len(grid) - 1)
        ext = grid[idx]
        vals = err[idx]
        # keep n+1 alternating extrema with the largest magnitudes
        sel = [0]
        for i in range(1, len(ext)):
            if np.sign(vals[i]) == np.sign(vals[sel[-1]]):
                if abs(vals[i]) > abs(vals[sel[-1]]):
                    sel[-1] = i
            else:
                sel.append(i)
        while len(sel) > n + 1:
            if abs(vals[sel[0]]) < abs(vals[sel[-1]]):
                sel.pop(0)
            else:
                sel.pop()
        if len(sel) == n + 1:
            x = ext[sel]
    return c, np.abs(err).max()


def fp32_horner(c, f):
    f = f.astype(np.float32)
    acc = np.float32(c[-1])
    for ck in reversed(c[:-1]):
        acc = (acc * f + np.float32(ck)).astype(np.float32)
    return (acc * f + np.float32(1.0)).astype(np.float32)


if __name__ == "__main__":
    for deg in (3, 4):
        c, e = remez_exp2(deg)
        f = np.linspace(-0.5, 0.5, 100001)
        e32 = np.abs(fp32_horner(c, f).astype(np.float64) / 2.0 ** f - 1).max()
        print(f"degree {deg}: coefficients {', '.join(repr(float(np.float32(v))) for v in c)}")
        print(f"   max rel error fp64 {e:.3e}, fp32 Horner {e32:.3e}")
