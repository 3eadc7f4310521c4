"""Fit the polynomial the prefill softmax uses for part of its exp2 evaluations.

2^t is split (Cody-Waite range reduction) into 2^n * 2^f with n = round(t) and
f = t - n in [-1/2, 1/2]; 2^f is a degree-3 polynomial whose maximum relative
error on [-1/2, 1/2] is minimised by the Remez exchange algorithm. Run this
script to reproduce the constants in prefill.cu (printed as float32).
"""
import numpy as np


def remez_exp2(deg=3, lo=-0.5, hi=0.5, iters=30):
    n = deg + 2
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    g = np.linspace(lo, hi, 200001)
    for _ in range(iters):
        a = np.zeros((n, n))
        for i in range(n):
            a[i, : deg + 1] = x[i] ** np.arange(deg + 1)
            a[i, deg + 1] = (-1) ** i * np.exp2(x[i])
        c = np.linalg.solve(a, np.exp2(x))[: deg + 1]
        err = np.polyval(c[::-1], g) / np.exp2(g) - 1
        d = np.diff(err)
        ext = np.where(np.sign(d[:-1]) != np.sign(d[1:]))[0] + 1
        sel = []
        for p in np.concatenate([[0], ext, [len(g) - 1]]):
            if sel and np.sign(err[p]) == np.sign(err[sel[-1]]):
                if abs(err[p]) > abs(err[sel[-1]]):
                    sel[-1] = p
            else:
                sel.append(p)
        while len(sel) > n:
            sel.pop(0) if abs(err[sel[0]]) < abs(err[sel[-1]]) else sel.pop()
        x = g[sel]
    return c, float(np.max(np.abs(err)))


if __name__ == "__main__":
    coeffs, max_rel = remez_exp2()
    print("coefficients c0..c3:", [repr(float(np.float32(v))) for v in coeffs], "max relative error", max_rel)
