"""Fits the polynomial the forward kernel uses to evaluate 2^f on the FMA
pipe for f in [-1/2, 1/2] (after Cody-Waite range reduction x = n + f with
n = round(x), so 2^x = 2^n * 2^f and 2^n is an exponent-field add).

Method: Remez exchange for the minimax *relative* error of a degree-3
polynomial; coefficients are rounded to float32 and the float32 Horner
evaluation is checked on a dense grid.  Run: python fit_exp2_poly.py
"""

import numpy as np


def remez_rel(deg=3, lo=-0.5, hi=0.5, iters=30):
    n = deg + 2
    k = np.arange(n)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * k[::-1] / (n - 1))
    grid = np.linspace(lo, hi, 200001)
    for _ in range(iters):
        f = np.exp2(x)
        # p(x_i) - f(x_i) = (-1)^i E f(x_i)  -> relative equioscillation
        A = np.zeros((n, n))
        for j in range(deg + 1):
            A[:, j] = x ** j
        A[:, deg + 1] = -((-1.0) ** k) * f
        sol = np.linalg.solve(A, f)
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], grid) - np.exp2(grid)) / np.exp2(grid)
        # new extrema: one per sign-alternating segment
        s = np.sign(err)
        idx = [0]
        for i in range(1, len(grid)):
            if s[i] != s[idx[-1]]:
                idx.append(i)
            elif abs(err[i]) > abs(err[idx[-1]]):
                idx[-1] = i
        if len(idx) >= n:
            # keep n alternating extrema with the largest magnitudes, in order
            while len(idx) > n:
                m = np.argmin(np.abs(err[idx]))
                idx.pop(m)
            x = grid[idx]
    return c, np.max(np.abs(err))


if __name__ == "__main__":
    c, e = remez_rel()
    c32 = c.astype(np.float32)
    g = np.linspace(-0.5, 0.5, 1000001).astype(np.float32)
    p = np.float32(c32[3])
    for j in (2, 1, 0):
        p = (p * g + c32[j]).astype(np.float32)
    rel = np.abs(p.astype(np.float64) - np.exp2(g.astype(np.float64))) / np.exp2(g.astype(np.float64))
    print("coefficients c0..c3 (float32):", [float(v) for v in c32])
    print("hex:", [hex(np.float32(v).view(np.uint32)) for v in c32])
    print(f"minimax relative error {e:.3e}; float32 Horner max relative error {rel.max():.3e}")
