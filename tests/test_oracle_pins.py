"""Pins for the fp64 oracle: it is checked against things other than itself.

Source: "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080", section "The problem" (separation
formula, 0.25-degree bins, every ordered pair counted, histogram sums of exactly N^2, the
Landy-Szalay omega) and Appendix A (clamp of the cosine, truncation of the index, clamp to the
last bin, omega only where RR > 0).

What pins what:
  * closed forms: two galaxies on the equator are |delta RA| apart (wrapped to <= 180 deg); two on
    one meridian are |delta Dec| apart; two on opposite meridians are 180 - |Dec1 + Dec2| apart.
    These fix the formula, the arcminute conversion and the truncating bin rule;
  * an independent fp64 formula: atan2(|u x v|, u . v) on unit vectors, written here with the
    ``math`` module, agrees with the oracle's arccos form on random and tightly clustered pairs;
  * invariants: totals n1*n2, bitwise symmetry theta(i,j) = theta(j,i), self-pairs in bin 0,
    antipodes in the last bin (and the clamp when the bins stop short of 180 degrees);
  * statistics: for a uniform sphere the fraction of pairs in [a, b) converges to
    (cos a - cos b)/2 with standard deviation about sqrt(2 f (1 - f))/n;
  * edge windows, by construction: equator pairs placed just inside / outside 1e-6 rad of an edge;
  * omega closed forms: D = R gives omega = 0; DD scaled by (1 + a) against DR = RR gives a;
    unequal catalog sizes normalise by pair totals; RR = 0 gives NaN.
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

W = 0.25
NB = 720


def _vec(ra_arcmin: float, dec_arcmin: float):
    a = ra_arcmin * math.pi / 10800
    d = dec_arcmin * math.pi / 10800
    return (math.cos(d) * math.cos(a), math.cos(d) * math.sin(a), math.sin(d))


def _theta_atan2(p, q) -> float:
    """Independent fp64 separation: atan2(|u x v|, u . v)."""
    u, v = _vec(*p), _vec(*q)
    cx = u[1] * v[2] - u[2] * v[1]
    cy = u[2] * v[0] - u[0] * v[2]
    cz = u[0] * v[1] - u[1] * v[0]
    return math.atan2(math.sqrt(cx * cx + cy * cy + cz * cz), u[0] * v[0] + u[1] * v[1] + u[2] * v[2])


def _f32(x) -> float:
    return float(np.float32(x))


# ------------------------------------------------------------------ closed forms

def test_equator_pairs_follow_delta_ra_closed_form():
    rnd = random.Random(5)
    # RA on a 1/64 arcmin grid: exact in fp32, so delta RA is known exactly
    ra = np.array([rnd.randrange(0, 21600 * 64) / 64.0 for _ in range(400)], np.float32)
    dec = np.zeros_like(ra)
    i = np.repeat(np.arange(len(ra)), len(ra))
    j = np.tile(np.arange(len(ra)), len(ra))
    bins = oracle.pair_bin(ra[i], dec[i], ra[j], dec[j], W, NB)
    theta = oracle.pair_theta(ra[i], dec[i], ra[j], dec[j])
    for a, b, k, th in zip(i, j, bins, theta):
        dra = abs(Fraction(float(ra[a])) - Fraction(float(ra[b])))
        sep = min(dra, 21600 - dra)                    # arcmin, exact
        assert abs(th - float(sep) * math.pi / 10800) < 3e-8
        exact = sep / 15                                # bins of 15 arcmin
        if exact.denominator == 1 and exact > 0:        # exactly on an edge: either side is allowed
            assert k in (int(exact) - 1, min(int(exact), NB - 1))
        else:
            assert k == min(math.floor(exact), NB - 1)


def test_meridian_and_opposite_meridian_closed_forms():
    rnd = random.Random(6)
    for _ in range(3000):
        ra0 = rnd.randrange(0, 10800 * 16) / 16.0
        d1 = rnd.randrange(-5400 * 16, 5400 * 16 + 1) / 16.0
        d2 = rnd.randrange(-5400 * 16, 5400 * 16 + 1) / 16.0
        same = oracle.pair_theta([ra0], [d1], [ra0], [d2])[0]
        assert abs(same - abs(d1 - d2) * math.pi / 10800) < 3e-8
        opp = oracle.pair_theta([ra0], [d1], [ra0 + 10800], [d2])[0]
        assert abs(opp - (10800 - abs(d1 + d2)) * math.pi / 10800) < 3e-8
    # a pole and any point on the equator are 90 degrees apart: bin 360 of 0.25-degree bins
    # sits exactly on an edge, so the pair must be in bin 359 or 360
    k = oracle.pair_bin([1234.5], [5400.0], [77.25], [0.0], W, NB)[0]
    assert k in (359, 360)
    th = oracle.pair_theta([1234.5], [5400.0], [77.25], [0.0])[0]
    assert abs(th - math.pi / 2) < 1e-12


# --------------------------------------------------------- independent formula

@pytest.mark.parametrize("clustered", [False, True])
def test_matches_independent_atan2_formula(clustered):
    rnd = random.Random(8 if clustered else 9)
    n = 48
    if clustered:
        base = (rnd.uniform(0, 21600), rnd.uniform(-5000, 5000))
        pts = [(_f32(base[0] + rnd.gauss(0, 0.05)), _f32(base[1] + rnd.gauss(0, 0.05))) for _ in range(n)]
    else:
        ra, dec = synth.uniform_sphere(n, seed=31)
        pts = list(zip(ra.tolist(), dec.tolist()))
    ra = np.array([p[0] for p in pts], np.float32)
    dec = np.array([p[1] for p in pts], np.float32)
    i = np.repeat(np.arange(n), n)
    j = np.tile(np.arange(n), n)
    th = oracle.pair_theta(ra[i], dec[i], ra[j], dec[j])
    bins = oracle.pair_bin(ra[i], dec[i], ra[j], dec[j], W, NB)
    w_rad = W * math.pi / 180
    for a, b, t, k in zip(i, j, th, bins):
        ref = _theta_atan2(pts[a], pts[b])
        # the arccos form loses about sqrt(2 eps) ~ 1.5e-8 rad at tiny separations
        assert abs(t - ref) < 2.5e-8
        kr = min(math.floor(ref / w_rad), NB - 1)
        if k != kr:
            edge = max(k, kr) * w_rad
            assert abs(ref - edge) < 5e-8 and abs(k - kr) == 1
    # the histogram of all ordered pairs equals the per-pair bins counted here
    h = oracle.histogram(ra, dec, bin_width_deg=W, nbins=NB, threads=2)
    assert np.array_equal(h.hist, np.bincount(bins, minlength=NB).astype(np.uint64))


# ------------------------------------------------------------------ invariants

def test_sums_symmetry_self_pairs():
    c = synth.catalogs(300, 257, 3, 30.0, seed=41)
    dd = oracle.histogram(c.ra_d, c.dec_d, bin_width_deg=W, nbins=NB)
    dr = oracle.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, W, NB)
    assert int(dd.hist.sum()) == 300 * 300
    assert int(dr.hist.sum()) == 300 * 257
    i = np.repeat(np.arange(300), 300)
    j = np.tile(np.arange(300), 300)
    a = oracle.pair_theta(c.ra_d[i], c.dec_d[i], c.ra_d[j], c.dec_d[j])
    b = oracle.pair_theta(c.ra_d[j], c.dec_d[j], c.ra_d[i], c.dec_d[i])
    assert np.array_equal(a, b)                       # bitwise symmetric
    self_bins = oracle.pair_bin(c.ra_d, c.dec_d, c.ra_d, c.dec_d, W, NB)
    assert np.all(self_bins == 0)
    # DR against the reversed-role RD gives the same histogram
    rd = oracle.histogram(c.ra_r, c.dec_r, c.ra_d, c.dec_d, W, NB)
    assert np.array_equal(dr.hist, rd.hist)


def test_antipodes_land_in_last_bin_and_clamp():
    ra, dec = synth.uniform_sphere(500, seed=51)
    ra2 = np.where(ra < 10800, ra + 10800, ra - 10800).astype(np.float32)
    dec2 = (-dec).astype(np.float32)
    assert np.all(oracle.pair_bin(ra, dec, ra2, dec2, W, NB) == NB - 1)
    # bins covering only 25 degrees: everything beyond lands in the last bin
    b = oracle.pair_bin(ra, dec, ra2, dec2, W, 100)
    assert np.all(b == 99)
    h = oracle.histogram(ra, dec, bin_width_deg=W, nbins=100)
    th = oracle.pair_theta(np.repeat(ra, 500), np.repeat(dec, 500), np.tile(ra, 500), np.tile(dec, 500))
    assert int(h.hist[99]) >= int(np.sum(th >= 25 * math.pi / 180))


def test_empty_catalogs_and_bad_arguments():
    h = oracle.histogram(np.zeros(0, np.float32), np.zeros(0, np.float32), bin_width_deg=W, nbins=NB)
    assert int(h.hist.sum()) == 0
    with pytest.raises(ValueError):
        oracle.histogram([0.0], [0.0], bin_width_deg=0.0, nbins=10)
    with pytest.raises(ValueError):
        oracle.histogram([0.0], [0.0], bin_width_deg=0.25, nbins=0)


# ------------------------------------------------------------------ statistics

@pytest.mark.parametrize("w,nb", [(10.0, 18), (0.25, 720)])
def test_uniform_sphere_bin_fractions_converge_to_closed_form(w, nb):
    n = 2000
    ra, dec = synth.uniform_sphere(n, seed=61)
    h = oracle.histogram(ra, dec, bin_width_deg=w, nbins=nb)
    counts = h.hist.astype(np.float64)
    counts[0] -= n                                    # remove the self-pairs
    frac = counts / (n * (n - 1))
    lo = np.radians(np.arange(nb) * w)
    hi = np.radians(np.minimum((np.arange(nb) + 1) * w, 180.0))
    f = (np.cos(lo) - np.cos(hi)) / 2
    sd = np.sqrt(2 * f * (1 - f)) / n
    assert np.all(np.abs(frac - f) <= 5 * sd + 1e-12), np.max(np.abs(frac - f) / (sd + 1e-30))


# ------------------------------------------------------------------ edge windows

def test_edge_windows_by_construction():
    # equator pairs at 15 arcmin (the 0.25-degree edge) +- offsets; 1e-6 rad = 0.0034377 arcmin
    base = 100.0
    offsets = [-0.006, -0.002, 0.002, 0.006, -0.0005, 0.0005]
    ra1 = np.array([base], np.float32)                # one anchor: 1 x 6 ordered pairs
    ra2 = np.array([base + 15 + o for o in offsets], np.float32)
    h = oracle.histogram(ra1, np.zeros(1, np.float32), ra2, np.zeros(len(offsets), np.float32), W, NB)
    below = above = 0
    for r in ra2:
        sep_rad = (float(r) - base) * math.pi / 10800
        e = 0.25 * math.pi / 180
        if e - 1e-6 <= sep_rad < e:
            below += 1
        elif e <= sep_rad < e + 1e-6:
            above += 1
    assert (below, above) == (2, 2)
    assert int(h.near_below[1]) == below and int(h.near_above[1]) == above
    assert int(h.near_below.sum()) == below and int(h.near_above.sum()) == above
    assert int(h.hist[0]) == 3 and int(h.hist[1]) == 3


# ------------------------------------------------------------------ omega

def test_omega_closed_forms():
    c = synth.catalogs(400, 0, 4, 30.0, seed=71)
    hh = oracle.histogram(c.ra_d, c.dec_d, bin_width_deg=1.0, nbins=180).hist
    om = oracle.omega(hh, hh, hh, 400, 400)
    assert np.all(np.isnan(om[hh == 0]))
    assert np.all(om[hh > 0] == 0.0)
    rr = np.array([1000, 2000, 0, 5], np.uint64)
    dr = rr.copy()
    dd = np.array([1500, 1000, 3, 5], np.uint64)
    om = oracle.omega(dd, dr, rr, 10, 10)
    assert om[0] == 0.5 and om[1] == -0.5 and math.isnan(om[2]) and om[3] == 0.0
    # unequal sizes: DD = RR (n_d/n_r)^2 and DR = RR (n_d/n_r) describe an unclustered D
    n_d, n_r = 300, 1200
    rr = np.array([16000, 32000, 48], np.uint64)
    dd = rr // 16
    dr = rr // 4
    assert np.allclose(oracle.omega(dd, dr, rr, n_d, n_r), 0.0, atol=1e-15)
    # the page's expression, term by term, when the sizes are equal
    rnd = np.random.default_rng(3)
    rr = rnd.integers(1, 10**9, 50).astype(np.uint64)
    dr = rnd.integers(0, 10**9, 50).astype(np.uint64)
    dd = rnd.integers(0, 10**9, 50).astype(np.uint64)
    om = oracle.omega(dd, dr, rr, 7, 7)
    ref = (dd.astype(object) - 2 * dr.astype(object) + rr.astype(object))
    for k in range(50):
        assert om[k] == float(Fraction(int(ref[k]), int(rr[k])))
