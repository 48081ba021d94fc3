"""Fit the cubic used by the kernels' software exp2 (run once; prints C constants).

The FlashAttention-4 pages (key contribution #2) compute part of the softmax
exponentials as a degree-3 polynomial on the FMA units, next to the hardware
exp2, and state that degree 3 is accurate enough for bf16; they give no
coefficients and no range reduction.  This script supplies both from standard
numerical analysis:

* range reduction: x = n + f with n = round-to-nearest(x), f in [-1/2, 1/2],
  2^x = 2^n * 2^f, where 2^n is applied by an integer add on the exponent bits;
* p(f) ~= 2^f is the degree-3 polynomial minimising the maximum RELATIVE error
  on [-1/2, 1/2], found with the Remez exchange algorithm (weight 2^-f),
  then rounded to fp32 and re-checked in fp32 Horner arithmetic.

Usage: python fit_exp2_poly.py
"""
from __future__ import annotations

import numpy as np

A, B = -0.5, 0.5
DEG = 3


def _solve(ref):
    n = DEG + 2
    M = np.zeros((n, n))
    rhs = np.exp2(ref)
    for i, x in enumerate(ref):
        M[i, :DEG + 1] = [x ** k for k in range(DEG + 1)]
        M[i, DEG + 1] = (-1) ** i * np.exp2(x)  # relative error level E * 2^x
    sol = np.linalg.solve(M, rhs)
    return sol[:DEG + 1], sol[DEG + 1]


def _rel_err(c, x):
    p = np.polyval(c[::-1], x)
    return p / np.exp2(x) - 1.0


def remez(iters=50):
    k = np.arange(DEG + 2)
    ref = (A + B) / 2 + (B - A) / 2 * np.cos(np.pi * k[::-1] / (DEG + 1))
    grid = np.linspace(A, B, 200001)
    c = None
    for _ in range(iters):
        c, E = _solve(ref)
        e = _rel_err(c, grid)
        # split the grid into sign runs and take each run's extremum
        sgn = np.sign(e)
        idx = np.flatnonzero(np.diff(sgn) != 0)
        bounds = np.concatenate(([0], idx + 1, [len(grid)]))
        ext = [lo + int(np.argmax(np.abs(e[lo:hi]))) for lo, hi in zip(bounds[:-1], bounds[1:])]
        if len(ext) < DEG + 2:
            break
        # keep DEG+2 alternating extrema with the largest magnitude window
        while len(ext) > DEG + 2:
            if abs(e[ext[0]]) < abs(e[ext[-1]]):
                ext.pop(0)
            else:
                ext.pop()
        new_ref = grid[ext]
        if np.max(np.abs(new_ref - ref)) < 1e-12:
            ref = new_ref
            break
        ref = new_ref
    return c


def fp32_check(c32):
    x = np.linspace(A, B, 1000001).astype(np.float32)
    p = np.float32(c32[3])
    for k in (2, 1, 0):
        p = (p * x + np.float32(c32[k])).astype(np.float32)
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)))


if __name__ == "__main__":
    c = remez()
    c32 = [np.float32(v) for v in c]
    print("max relative error (exact coefficients):",
          float(np.max(np.abs(_rel_err(c, np.linspace(A, B, 1000001))))))
    print("max relative error (fp32 Horner):", fp32_check(c32))
    for k, v in enumerate(c32):
        print(f"constexpr float kExp2C{k} = {float(v).hex()}f;  // {float(v):.9g}")
