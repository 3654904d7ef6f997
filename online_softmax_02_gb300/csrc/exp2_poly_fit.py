"""Fit of the degree-3 polynomial for 2^f, f in [-1/2, 1/2], used by the
software exponential in common.cuh (soft_exp2x2).

p(f) = 1 + c1 f + c2 f^2 + c3 f^3 (p(0) = 1, so integer arguments are exact)
with (c1, c2, c3) minimising max |p(f) / 2^f - 1| over a dense grid: a
linear program in (c1, c2, c3, t), minimise t subject to
|p(f_i) - 2^f_i| <= t 2^f_i. Run: python exp2_poly_fit.py (needs scipy);
prints the coefficients rounded to FP32 and the relative error they reach.
"""
import numpy as np
from scipy.optimize import linprog


def fit(degree=3, points=4001):
    f = np.linspace(-0.5, 0.5, points)
    y = np.exp2(f)
    A = np.stack([f ** k for k in range(1, degree + 1)], 1)
    a_ub = np.vstack([np.hstack([A, -y[:, None]]), np.hstack([-A, -y[:, None]])])
    b_ub = np.concatenate([y - 1, 1 - y])
    res = linprog(np.r_[np.zeros(degree), 1.0], A_ub=a_ub, b_ub=b_ub,
                  bounds=[(None, None)] * degree + [(0, None)], method="highs")
    c = res.x[:degree].astype(np.float32)
    rel = np.abs((1 + A @ c.astype(np.float64)) / y - 1).max()
    return c, rel


if __name__ == "__main__":
    c, rel = fit()
    for k, v in enumerate(c, 1):
        print("c%d = %r" % (k, float(v)))
    print("max relative error %.4e" % rel)
