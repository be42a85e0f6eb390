"""Coefficients of the cubic that the paired extend kernel uses for 2^f, f in [-1/2, 1/2].

Part of the kernel's exponentials run on the FMA pipe instead of the exponential unit: with
x = n + f, n = round(x) (Cody and Waite's argument reduction), 2^x = 2^n * p(f), where 2^n is
built from its exponent bits and p is the cubic below.  The coefficients minimise the largest
*relative* error |p(f) / 2^f - 1| over the interval (the minimax polynomial), found here with the
Remez exchange algorithm: solve for the coefficients and the levelled error E at five reference
points, move the references to the extrema of the error, and repeat until the extrema are level.
The error bound is about 7.5e-5, well inside bf16's half-ulp of 2^-9 = 1.95e-3, the precision P
is stored in.

Run ``python -m prefix_shared_kv_gb300.fit_exp2`` to print the coefficients as they appear in
csrc/extend_pair.cu; a CPU test checks that the two agree.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def remez(degree: int = DEGREE, lo: float = LO, hi: float = HI, iters: int = 30):
    """Minimax coefficients c[0..degree] (lowest first) of p(f) ~ 2^f in relative error, and the
    levelled error."""
    n = degree + 2
    # Chebyshev extrema as the first reference points
    ref = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    grid = np.linspace(lo, hi, 200001)
    coef, err = None, None
    for _ in range(iters):
        # p(f_i) - 2^f_i = (-1)^i E 2^f_i  (relative error levelled at the references)
        A = np.zeros((n, n))
        for i, f in enumerate(ref):
            A[i, :degree + 1] = f ** np.arange(degree + 1)
            A[i, degree + 1] = -((-1.0) ** i) * 2.0 ** f
        sol = np.linalg.solve(A, 2.0 ** ref)
        coef, err = sol[:degree + 1], abs(sol[degree + 1])
        rel = np.polyval(coef[::-1], grid) / 2.0 ** grid - 1.0
        # new references: the extremum of the error in each run of constant sign
        sign = np.sign(rel)
        cuts = np.flatnonzero(np.diff(sign) != 0) + 1
        runs = np.split(np.arange(grid.size), cuts)
        ext = [r[np.argmax(np.abs(rel[r]))] for r in runs]
        if len(ext) < n:
            break
        while len(ext) > n:  # keep the n largest, alternating by construction of the runs
            drop = 0 if abs(rel[ext[0]]) < abs(rel[ext[-1]]) else -1
            ext.pop(drop)
        new = grid[ext]
        if np.allclose(new, ref, atol=1e-12):
            break
        ref = new
    return coef, err


def max_rel_error(coef, lo: float = LO, hi: float = HI) -> float:
    f = np.linspace(lo, hi, 400001)
    return float(np.max(np.abs(np.polyval(np.asarray(coef)[::-1], f) / 2.0 ** f - 1.0)))


def float32_coefficients():
    coef, _ = remez()
    return [float(np.float32(c)) for c in coef]


if __name__ == "__main__":
    c = float32_coefficients()
    for i, v in enumerate(c):
        print(f"c{i} = {v!r}f")
    print(f"max relative error {max_rel_error(c):.3e}")
