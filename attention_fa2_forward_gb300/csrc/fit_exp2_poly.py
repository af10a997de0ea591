"""Fit the degree-3 polynomial used for 2^f, f in [-1/2, 1/2], in sm103_ptx.cuh.

Remez exchange on the relative error |p(f) / 2^f - 1| (equioscillation on
deg + 2 points), then rounding of the coefficients to fp32 and a dense check
of the fp32 Horner evaluation. Prints the coefficients and their fp32 bit
patterns (the constants in exp2_poly3_pair) and the maximum relative error.

    python fit_exp2_poly.py [degree]
"""
import struct
import sys

import numpy as np


def remez_relative(deg, a=-0.5, b=0.5, iters=40):
    n = deg + 2
    x = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    grid = np.linspace(a, b, 200001)
    coef = None
    for _ in range(iters):
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = (-1) ** i * np.exp2(x[i])
        sol = np.linalg.solve(A, np.exp2(x))
        coef = sol[:deg + 1]
        err = (np.polyval(coef[::-1], grid) - np.exp2(grid)) / np.exp2(grid)
        segments = np.split(np.arange(grid.size), np.where(np.diff(np.sign(err)) != 0)[0] + 1)
        extrema = [seg[np.argmax(np.abs(err[seg]))] for seg in segments]
        if len(extrema) != n:
            break
        x = grid[extrema]
    return coef


def fp32_horner_error(c32, a=-0.5, b=0.5):
    f = np.linspace(a, b, 400001).astype(np.float32)
    p = np.full_like(f, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        p = (p * f + c32[k]).astype(np.float32)
    return float(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1).max())


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c32 = remez_relative(deg).astype(np.float32)
    for k, c in enumerate(c32):
        bits = struct.unpack("<I", struct.pack("<f", float(c)))[0]
        print(f"c{k} = {float(c):.8f}  (0x{bits:08X})")
    print(f"max relative error (fp32 Horner on [-1/2, 1/2]): {fp32_horner_error(c32):.3e}")
