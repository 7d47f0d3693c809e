"""Fits the polynomial the kernel uses for part of its exp2 evaluations.

The kernel computes 2^x for x <= 8 either with the hardware approximation
(ex2.approx) or, for a fixed subset of the columns of each score tile, on the
FMA pipe: x is split into an integer j = round(x) and a remainder
f = x - j in [-1/2, 1/2]; 2^f is a polynomial p(f); 2^j is added to the
exponent field with an integer shift and add (Cody and Waite's range
reduction).  This script finds p: the degree-3 polynomial minimising the
maximum RELATIVE error |p(f) / 2^f - 1| over [-1/2, 1/2], posed as a linear
program on a dense grid (scipy.optimize.linprog), then rounds the coefficients
to float32 and reports the error of the float32 Horner evaluation.

Run: python fit_exp2_poly.py  -> prints the coefficients c0..c3 (p = c0 + f(c1 + f(c2 + f c3))).
"""

import numpy as np
from scipy.optimize import linprog


def fit(degree=3, n=20001):
    f = np.linspace(-0.5, 0.5, n)
    y = np.exp2(f)
    V = np.stack([f ** i for i in range(degree + 1)], axis=1) / y[:, None]  # p(f)/2^f
    # variables: c_0..c_d, e ; minimise e subject to |V c - 1| <= e
    nv = degree + 2
    cost = np.zeros(nv)
    cost[-1] = 1.0
    A = np.vstack([np.hstack([V, -np.ones((n, 1))]), np.hstack([-V, -np.ones((n, 1))])])
    b = np.concatenate([np.ones(n), -np.ones(n)])
    res = linprog(cost, A_ub=A, b_ub=b, bounds=[(None, None)] * nv, method="highs")
    assert res.success
    return res.x[:-1], res.x[-1]


def horner_f32(c, f):
    c = [np.float32(x) for x in c]
    f = np.asarray(f, dtype=np.float32)
    r = np.full_like(f, c[-1])
    for ci in c[-2::-1]:
        r = (r * f + ci).astype(np.float32)  # one fma per step in the kernel
    return r


if __name__ == "__main__":
    c, e = fit()
    c32 = np.asarray(c, dtype=np.float32)
    f = np.linspace(-0.5, 0.5, 200001)
    rel = np.abs(horner_f32(c32, f).astype(np.float64) / np.exp2(f) - 1)
    print("minimax relative error (exact arithmetic): %.3e" % e)
    print("float32 Horner max relative error: %.3e" % rel.max())
    for i, x in enumerate(c32):
        print("c%d = %.9ef  (0x%08x)" % (i, x, np.float32(x).view(np.uint32)))
