"""Coefficients of the polynomial p(f) ~ 2^f, f in [-1/2, 1/2], that the
prefill softmax uses for part of its exponentials (csrc/prefill.cu,
exp2_poly).

Minimax fit of the RELATIVE error by the Remez exchange algorithm (E. Ya.
Remez, 1934; see W. J. Cody and W. Waite, "Software Manual for the
Elementary Functions", 1980, ch. 2): solve for the coefficients and a
levelled error E such that (p(x_i) - 2^x_i) / 2^x_i = (-1)^i E at n + 2
reference points, move the points to the extrema of the error, repeat.  The
coefficients are then rounded to float32 and the maximum relative error of
that float32 polynomial, evaluated by Horner's rule in float64 on a dense
grid, is printed.

    python gqa_attention_kv_decode_gb300/csrc/exp2_poly_fit.py [degree]
"""

from __future__ import annotations

import sys

import numpy as np


def remez_rel(n: int, lo: float = -0.5, hi: float = 0.5, iters: int = 30) -> np.ndarray:
    """Coefficients c[0..n] (c[k] multiplies x^k) of the degree-n minimax
    approximation of 2^x on [lo, hi] in relative error."""
    m = n + 2
    x = 0.5 * (lo + hi) - 0.5 * (hi - lo) * np.cos(np.pi * np.arange(m) / (m - 1))
    grid = np.linspace(lo, hi, 200001)
    coef = None
    for _ in range(iters):
        f = np.exp2(x)
        A = np.stack([x ** k / f for k in range(n + 1)] + [(-1.0) ** np.arange(m)], axis=1)
        coef = np.linalg.solve(A, np.ones(m))[:-1]
        err = np.polyval(coef[::-1], grid) / np.exp2(grid) - 1.0
        # one extremum of the error per run of equal sign
        idx, start = [], 0
        sign = np.sign(err)
        for i in range(1, len(grid) + 1):
            if i == len(grid) or sign[i] != sign[start]:
                idx.append(start + int(np.argmax(np.abs(err[start:i]))))
                start = i
        while len(idx) > m:  # drop the smaller end extremum
            idx.pop(0 if abs(err[idx[0]]) < abs(err[idx[-1]]) else -1)
        if len(idx) < m:
            break
        x = grid[idx]
    return coef


def main():
    n = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c32 = remez_rel(n).astype(np.float32)
    grid = np.linspace(-0.5, 0.5, 2000001)
    p = np.zeros_like(grid)
    for c in c32[::-1].astype(np.float64):  # Horner, as the kernel evaluates it
        p = p * grid + c
    rel = np.abs(p / np.exp2(grid) - 1.0).max()
    print("degree", n)
    for i, c in enumerate(c32):
        print(f"  c{i} = {float(c):.9g}f  ({int(np.float32(c).view(np.uint32)):#010x})")
    print(f"  max relative error on [-1/2, 1/2]: {rel:.3e} (2^{np.log2(rel):.2f})")


if __name__ == "__main__":
    main()
