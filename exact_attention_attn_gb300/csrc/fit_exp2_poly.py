"""Fit the polynomial behind the FMA-pipe exp2 of the tensor-core kernels.

Method: Cody-Waite style range reduction 2^y = 2^j * 2^f with j = round(y)
and f = y - j in [-1/2, 1/2]; 2^f is approximated by the degree-3 polynomial
minimising the maximum relative error on [-1/2, 1/2], found with the Remez
exchange algorithm on the relative-error functional.  Run it to reproduce the
coefficients written into sm100_ptx.cuh:

    python exact_attention_attn_gb300/csrc/fit_exp2_poly.py
"""
import numpy as np


def remez_exp2(deg: int, iters: int = 40):
    n = deg + 2
    xs = 0.5 * np.cos(np.pi * np.arange(n) / (n - 1))[::-1]
    grid = np.linspace(-0.5, 0.5, 40001)
    for _ in range(iters):
        A = np.zeros((n, n))
        for i, x in enumerate(xs):
            A[i, :deg + 1] = x ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2.0 ** x
        sol = np.linalg.solve(A, 2.0 ** xs)
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        turn = [0] + [i for i in range(1, len(grid) - 1)
                      if (err[i] - err[i - 1]) * (err[i + 1] - err[i]) <= 0] + [len(grid) - 1]
        if len(turn) >= n:
            keep = np.argsort(-np.abs(err[turn]))[:n]
            xs = np.sort(grid[np.array(turn)[keep]])
    c32 = c.astype(np.float32)
    err32 = np.abs((np.polyval(c32.astype(np.float64)[::-1], grid) - 2.0 ** grid) / 2.0 ** grid).max()
    return c32, err32


if __name__ == "__main__":
    c, e = remez_exp2(3)
    print("coefficients c0..c3 (float32):", [float(x) for x in c])
    print("max relative error on [-1/2, 1/2]: %.3e" % e)
