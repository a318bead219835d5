"""Fit the cubic used by the prefill kernel's software exp2.

2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]; 2^f is
approximated by c0 + c1 f + c2 f^2 + c3 f^3 with coefficients minimising the
maximum relative error on [-1/2, 1/2] (Remez exchange on the relative error,
started from Chebyshev nodes).  Run: python fit_exp2_poly.py
"""
import numpy as np


def fit(deg=3, iters=40):
    lo, hi = -0.5, 0.5
    k = np.arange(deg + 2)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * k[::-1] / (deg + 1))
    grid = np.linspace(lo, hi, 200001)
    for _ in range(iters):
        # solve p(x_i) - 2^x_i = (-1)^i E 2^x_i  (equioscillating relative error)
        A = np.zeros((deg + 2, deg + 2))
        for i, xi in enumerate(x):
            A[i, :deg + 1] = xi ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2.0 ** xi
        sol = np.linalg.solve(A, 2.0 ** x)
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        # new reference: extrema of the error in each sign-alternating segment
        idx = [np.argmax(np.abs(err[(grid >= a) & (grid <= b)])) + np.searchsorted(grid, a)
               for a, b in zip(np.r_[lo, (x[:-1] + x[1:]) / 2], np.r_[(x[:-1] + x[1:]) / 2, hi])]
        x = grid[idx]
    return c, np.abs(err).max()


if __name__ == "__main__":
    c, e = fit()
    print("coefficients c0..c3:", ", ".join("%.9ef" % v for v in c))
    print("max relative error: %.3e" % e)
