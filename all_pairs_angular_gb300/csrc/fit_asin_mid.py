"""Derive the polynomial the pair kernel uses for separations between 55 and 125 degrees.

There the dot product d = u.v of two unit vectors determines theta without loss: theta =
pi/2 - asin(d), and asin(d) = d * R(d^2) with R(t) = asin(sqrt t)/sqrt t analytic on [0, 1).
The kernel only uses this form when the caps of both groups prove |d| < cos(55 deg), so R is
fitted on t in [0, cos^2(54.5 deg)] (half a degree of margin, far above the fp32 error of d), with
degree 4 (error 1.5e-7 rad, also after rounding the coefficients to fp32, inside the kernel's
precision budget; degree 5 gives about 1e-8 for one more instruction per pair). We minimise the largest ABSOLUTE error
of d * R(d^2) (= the error in theta, radians) by Lawson's iteratively reweighted least squares on a
Chebyshev grid, with R evaluated in 40-digit arithmetic. Prints the coefficients (lowest degree
first) and the worst theta error before and after rounding them to fp32.

Run: python fit_asin_mid.py [degree [theta_fit_deg]]   (defaults: 4 54.5)
"""
import sys

import mpmath as mp
import numpy as np

mp.mp.dps = 40
DEG = int(sys.argv[1]) if len(sys.argv) > 1 else 4
N = 6000
THETA_FIT_DEG = float(sys.argv[2]) if len(sys.argv) > 2 else 54.5


def r_exact(t):
    t = mp.mpf(t)
    if t == 0:
        return mp.mpf(1)
    s = mp.sqrt(t)
    return mp.asin(s) / s


def main():
    tmax = mp.cos(mp.radians(THETA_FIT_DEG)) ** 2
    ts = [tmax * (1 - mp.cos(mp.pi * (k + mp.mpf("0.5")) / N)) / 2 for k in range(N)]
    rx = np.array([float(r_exact(t)) for t in ts])
    dx = np.array([float(mp.sqrt(t)) for t in ts])
    tf = np.array([float(t) for t in ts])
    V = np.vander(tf, DEG + 1, increasing=True)
    w = np.ones(N) / N
    for _ in range(2000):
        W = np.sqrt(w) * dx
        c, *_ = np.linalg.lstsq(V * W[:, None], rx * W, rcond=None)
        err = np.abs(V @ c - rx) * dx
        w = w * (err / err.max() + 1e-30) ** 0.5
        w /= w.sum()
    print("degree", DEG, "on t <= cos^2(%g deg): max |d theta| (rad) %.3e" % (THETA_FIT_DEG, err.max()))
    c32 = c.astype(np.float32).astype(np.float64)
    err32 = np.abs(V @ c32 - rx) * dx
    print("after fp32 rounding of the coefficients: %.3e" % err32.max())
    for k, v in enumerate(c):
        print("  r%d = %.17g" % (k, v))


if __name__ == "__main__":
    main()
