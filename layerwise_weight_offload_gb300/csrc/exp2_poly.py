"""Coefficients of the cubic that attention.cu uses for 2^f, f in [-1/2, 1/2].

The kernel splits x = n + f with n = round(x) and f in [-1/2, 1/2], takes
2^f from a cubic c0 + c1 f + c2 f^2 + c3 f^3 and adds n to the exponent
field.  The cubic minimises the largest relative error |p(f) / 2^f - 1| over
a dense grid of the interval (a Chebyshev approximation problem, solved as a
linear program).  Run this file to print the coefficients as fp32 literals
and the error they reach.
"""
import numpy as np
from scipy.optimize import linprog


def fit(degree=3, points=4001):
    f = np.linspace(-0.5, 0.5, points)
    y = np.exp2(f)
    # variables: c_0..c_degree, t; minimise t subject to
    # +-(sum_k c_k f^k / y - 1) <= t
    V = np.stack([f ** k for k in range(degree + 1)], axis=1) / y[:, None]
    ones = np.ones((points, 1))
    A = np.vstack([np.hstack([V, -ones]), np.hstack([-V, -ones])])
    b = np.concatenate([np.ones(points), -np.ones(points)])
    cost = np.zeros(degree + 2)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=A, b_ub=b, bounds=[(None, None)] * (degree + 2), method="highs")
    assert res.success, res.message
    return res.x[:-1]


def max_rel_error_fp32(c, points=200001):
    f = np.linspace(-0.5, 0.5, points).astype(np.float32)
    c32 = np.asarray(c, dtype=np.float32)
    p = np.float32(c32[3])
    for k in (2, 1, 0):
        p = (p * f + c32[k]).astype(np.float32)
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)))


if __name__ == "__main__":
    c = fit()
    for k, v in enumerate(c):
        print("c%d = %.9ef" % (k, np.float32(v)))
    print("max relative error in fp32 Horner evaluation: %.3e" % max_rel_error_fp32(c))
