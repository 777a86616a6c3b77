"""The seeded generator: portable elementary functions, workload shapes, determinism."""
import math
import random

import numpy as np
import pytest

import synth


def test_elementary_functions_match_libm_to_two_ulp():
    rnd = random.Random(7)
    for _ in range(5000):
        x = rnd.uniform(-7.5, 7.5)
        for name, ref in (("sin", math.sin), ("cos", math.cos)):
            got, want = synth.elementary(name, x), ref(x)
            assert abs(got - want) <= 2 * math.ulp(max(abs(want), 1e-300)) + 1e-300 or abs(got - want) < 4e-16
        y, z = rnd.uniform(-1, 1), rnd.uniform(-1, 1)
        assert abs(synth.elementary("atan2", y, z) - math.atan2(y, z)) < 5e-16
        assert abs(synth.elementary("asin", y) - math.asin(y)) < 5e-16
        p = 10 ** rnd.uniform(-300, 300)
        assert abs(synth.elementary("log", p) - math.log(p)) <= 4 * math.ulp(abs(math.log(p)))


def test_same_seed_same_catalog_and_different_seed_differs():
    a = synth.catalogs(500, 400, 5, 30.0, seed=11)
    b = synth.catalogs(500, 400, 5, 30.0, seed=11)
    c = synth.catalogs(500, 400, 5, 30.0, seed=12)
    assert a.digest() == b.digest()
    assert a.digest() != c.digest()


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_workload_shapes(idx):
    c = synth.config(idx)
    spec = synth.CONFIGS[idx]
    assert c.n_d == spec["n_d"] and c.n_r == spec["n_r"]
    for ra, dec in ((c.ra_d, c.dec_d), (c.ra_r, c.dec_r)):
        assert ra.dtype == np.float32 and dec.dtype == np.float32
        assert np.all(np.isfinite(ra)) and np.all(np.isfinite(dec))
        if spec["patch_arcmin"] > 0:
            assert ra.min() >= 0 and ra.max() < 300 and dec.min() >= 0 and dec.max() < 300
        else:
            assert ra.min() >= 0 and ra.max() < 21600
            assert dec.min() >= -5400 and dec.max() <= 5400


def test_uniform_sphere_declination_distribution():
    # sin(dec) of a uniform sphere is uniform on [-1, 1]
    ra, dec = synth.uniform_sphere(200_000, seed=3)
    s = np.sin(dec.astype(np.float64) * math.pi / 10800)
    hist, _ = np.histogram(s, bins=20, range=(-1, 1))
    expect = len(s) / 20
    assert np.all(np.abs(hist - expect) < 6 * math.sqrt(expect))
    hist_ra, _ = np.histogram(ra, bins=24, range=(0, 21600))
    assert np.all(np.abs(hist_ra - len(ra) / 24) < 6 * math.sqrt(len(ra) / 24))


def test_clump_members_spread_like_sigma():
    n_clumps, sigma = 4, 30.0
    c = synth.catalogs(8000, 0, n_clumps, sigma, seed=21)
    half = c.n_d // 2
    ra = c.ra_d[half:].astype(np.float64) * math.pi / 10800
    dec = c.dec_d[half:].astype(np.float64) * math.pi / 10800
    v = np.stack([np.cos(dec) * np.cos(ra), np.cos(dec) * np.sin(ra), np.sin(dec)], 1)
    for k in range(n_clumps):
        m = v[k::n_clumps]
        centre = m.mean(0)
        centre /= np.linalg.norm(centre)
        ang = np.arccos(np.clip(m @ centre, -1, 1)) * 10800 / math.pi  # arcmin
        # two Gaussian tangent components: mean square separation = 2 sigma^2
        rms = math.sqrt(np.mean(ang ** 2))
        assert abs(rms - math.sqrt(2) * sigma) < 0.1 * math.sqrt(2) * sigma


def test_sample_rows_distinct_sorted_and_seeded():
    a = synth.sample_rows(10_000, 2000, seed=4)
    b = synth.sample_rows(10_000, 2000, seed=4)
    assert np.array_equal(a, b)
    assert len(np.unique(a)) == 2000 and np.all(np.diff(a) > 0) and a[0] >= 0 and a[-1] < 10_000
