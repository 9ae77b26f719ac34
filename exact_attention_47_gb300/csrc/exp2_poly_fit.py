"""Fit of the polynomial behind ex2_poly2 (ptx.cuh): 2^f on [-1/2, 1/2].

2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]; 2^f is
approximated by a degree-4 polynomial whose relative error is made nearly
equal-ripple by iteratively reweighted least squares on Chebyshev points
(weights grow where the error is largest).  Run to print the coefficients
(fp32, lowest degree first) and the fp32 Horner evaluation's worst relative
error on a dense grid.
"""

import numpy as np

DEGREE = 4


def fit(degree=DEGREE, iters=30, points=4001):
    f = np.cos(np.linspace(0.0, np.pi, points)) * 0.5
    y = np.exp2(f)
    w = 1.0 / y
    for _ in range(iters):
        a = np.vander(f, degree + 1, increasing=True) * w[:, None]
        c, *_ = np.linalg.lstsq(a, y * w, rcond=None)
        err = np.abs(np.polyval(c[::-1], f) / y - 1.0)
        w = w * (1.0 + 50.0 * err / err.max())
    return c.astype(np.float32)


def horner_f32(c, f):
    """fp32 Horner evaluation of the polynomial with fp32 coefficients c."""
    f = np.asarray(f, dtype=np.float32)
    acc = np.full_like(f, c[-1])
    for k in range(len(c) - 2, -1, -1):
        acc = (acc * f + c[k]).astype(np.float32)
    return acc


if __name__ == "__main__":
    c = fit()
    f = np.linspace(-0.5, 0.5, 200001, dtype=np.float32)
    rel = np.abs(horner_f32(c, f).astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)
    print("coefficients:", ", ".join("%.9e" % v for v in c))
    print("max relative error %.3e (2^%.2f)" % (rel.max(), np.log2(rel.max())))
