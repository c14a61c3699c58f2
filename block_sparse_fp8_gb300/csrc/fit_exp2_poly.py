#!/usr/bin/env python3
"""Fits the polynomial the attention kernel uses for part of its exp2 evaluations.

Range reduction (Cody & Waite, "Software Manual for the Elementary Functions", 1980): for
x >= -126, n = round(x) and f = x - n lie in [-1/2, 1/2], and 2^x = 2^n * 2^f.  The rounding
uses the fp32 "magic number" 1.5 * 2^23: j = x + 1.5*2^23 rounds x to an integer held in j's
low mantissa bits, n = j - 1.5*2^23, and 2^n is applied by adding n << 23 (the low bits of
j << 23) to the bit pattern of the polynomial value.

2^f on [-1/2, 1/2] is approximated by the degree-d polynomial minimising the maximum
RELATIVE error, found with the Remez exchange algorithm (Remez, 1934) on a dense grid and
then rounded to fp32.  The script prints the coefficients (c0 .. cd) and the maximum relative
error of fp32 Horner evaluation; it is the source of the constants in ptx_sm103.cuh.

    python fit_exp2_poly.py [degree]
"""
import sys

import numpy as np


def remez_relative(deg, iters=30, grid=200001):
    xs = np.linspace(-0.5, 0.5, grid)
    f = np.exp2(xs)
    k = np.arange(deg + 2)
    nodes = 0.5 * np.cos(np.pi * k / (deg + 1))[::-1]  # Chebyshev start
    coef = None
    for _ in range(iters):
        # p(x_j) - 2^x_j = (-1)^j E 2^x_j at the nodes (equioscillating relative error)
        A = np.zeros((deg + 2, deg + 2))
        for j, x in enumerate(nodes):
            A[j, :deg + 1] = x ** np.arange(deg + 1)
            A[j, deg + 1] = -((-1) ** j) * np.exp2(x)
        sol = np.linalg.solve(A, np.exp2(nodes))
        coef = sol[:deg + 1]
        err = (np.polyval(coef[::-1], xs) - f) / f
        # new nodes: the largest error between consecutive sign changes
        sign = np.sign(err)
        idx = [0]
        for i in range(1, grid):
            if sign[i] != sign[idx[-1]]:
                idx.append(i)
            elif abs(err[i]) > abs(err[idx[-1]]):
                idx[-1] = i
        if len(idx) < deg + 2:
            break
        while len(idx) > deg + 2:
            if abs(err[idx[0]]) < abs(err[idx[-1]]):
                idx.pop(0)
            else:
                idx.pop()
        nodes = xs[idx]
    return coef


def fp32_horner_error(coef32):
    xs = np.linspace(-0.5, 0.5, 400001).astype(np.float32)
    acc = np.full_like(xs, coef32[-1])
    for c in coef32[-2::-1]:
        acc = (acc * xs + c).astype(np.float32)
    ref = np.exp2(xs.astype(np.float64))
    return float(np.max(np.abs(acc.astype(np.float64) - ref) / ref))


def main():
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 4
    coef = remez_relative(deg)
    c32 = coef.astype(np.float32)
    print(f"degree {deg}: max relative error (fp32 Horner) = {fp32_horner_error(c32):.3e}")
    for i, c in enumerate(c32):
        print(f"  c{i} = {float(c).hex()}f  // {float(c):.9e}")


if __name__ == "__main__":
    main()
