"""Derive the polynomial the pair kernel uses to turn a squared chord into a squared angle.

For two unit vectors at angle theta' <= 90 degrees, the squared chord is q = |u - v|^2 =
4 sin^2(theta'/2), so theta'^2 = 4 asin^2(sqrt(q)/2) = q * f(q) with f analytic on [0, 2]
(f(0) = 1). We fit P(q) ~ f(q), minimising the largest ABSOLUTE error in theta' (relative error
of f times theta'/2), by Lawson's iteratively reweighted least squares on a Chebyshev grid, with
f evaluated in 40-digit arithmetic. Prints the coefficients (highest degree last) and the worst
theta' error before and after rounding them to fp32.

The kernel uses two fits: degree 7 on theta' <= 90 degrees (any chord), and degree 5 on
theta' <= 72.4 degrees (for groups whose caps keep every theta' below 72 degrees).

Run: python fit_arcsin2.py [degree [theta_max_deg]]   (defaults: 7 90)
"""
import sys

import mpmath as mp
import numpy as np

mp.mp.dps = 40
DEG = int(sys.argv[1]) if len(sys.argv) > 1 else 7
THETA_MAX_DEG = float(sys.argv[2]) if len(sys.argv) > 2 else 90.0
N = 6000


def f_exact(q):
    q = mp.mpf(q)
    if q == 0:
        return mp.mpf(1)
    th = 2 * mp.asin(mp.sqrt(q) / 2)
    return th * th / q


def main():
    qmax = 4 * mp.sin(mp.radians(THETA_MAX_DEG) / 2) ** 2
    xs = [qmax * (1 - mp.cos(mp.pi * (k + mp.mpf("0.5")) / N)) / 2 for k in range(N)]
    fx = np.array([float(f_exact(x)) for x in xs])
    th = np.array([float(2 * mp.asin(mp.sqrt(x) / 2)) for x in xs])
    xf = np.array([float(x) for x in xs])
    V = np.vander(xf, DEG + 1, increasing=True)
    w = np.ones(N) / N
    for _ in range(2000):
        W = np.sqrt(w) * th / fx
        c, *_ = np.linalg.lstsq(V * W[:, None], fx * W, rcond=None)
        err = np.abs(V @ c - fx) / fx * th / 2
        w = w * (err / err.max()) ** 0.5
        w /= w.sum()
    print("degree", DEG, "on theta' <= %g deg: max |d theta'| (rad) %.3e" % (THETA_MAX_DEG, err.max()))
    c32 = c.astype(np.float32).astype(np.float64)
    err32 = np.abs(V @ c32 - fx) / fx * th / 2
    print("after fp32 rounding of the coefficients: %.3e" % err32.max())
    for k, v in enumerate(c):
        print("  c%d = %.17g" % (k, v))


if __name__ == "__main__":
    main()
