"""GPU parity: the CUDA library through its C ABI against the fp64 oracle.

The rule (from the fp64 definition of "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080", section
"The problem"): every histogram sums to exactly n1*n2; every bin equals the oracle's except that
pairs whose fp64 theta is within 1e-6 rad of a bin edge may sit in the bin on the other side of
that edge (checked through cumulative counts by oracle.check.edge_flux); omega computed on the GPU
from the GPU counts equals the oracle's omega of the same counts to 1e-12 relative.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import check

pytestmark = pytest.mark.gpu

TOL = oracle.EDGE_TOL_RAD
DEFAULT_EXACT = 2


@pytest.fixture(scope="module")
def ctx(acf):
    c = acf.Context(0)
    yield c
    c.close()


def _compare(acf, ctx, ra1, dec1, ra2, dec2, w, nb, threads=0):
    g = ctx.histogram(ra1, dec1, ra2, dec2, bin_width_deg=w, nbins=nb)
    torch.cuda.synchronize()
    gh = acf.as_uint64(g)
    o = oracle.histogram(ra1, dec1, ra2, dec2, w, nb, threads=threads)
    rep = check.edge_flux(gh, o.hist, o.near_below, o.near_above)
    n1 = len(ra1)
    n2 = n1 if ra2 is None else len(ra2)
    assert int(gh.sum()) == n1 * n2
    assert rep.ok, str(rep)
    return gh, o, rep


def test_tiny_workload_full_parity_and_omega(acf, ctx):
    c = synth.config(0)
    w, nb = c.bin_width_deg, c.nbins
    dd, _, r1 = _compare(acf, ctx, c.ra_d, c.dec_d, None, None, w, nb)
    dr, _, r2 = _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, w, nb)
    rr, _, r3 = _compare(acf, ctx, c.ra_r, c.dec_r, None, None, w, nb)
    tdd, tdr, trr = (torch.from_numpy(x.view(np.int64)).cuda() for x in (dd, dr, rr))
    om = ctx.omega(tdd, tdr, trr, c.n_d, c.n_r).cpu().numpy()
    assert check.omega_close(om, oracle.omega(dd, dr, rr, c.n_d, c.n_r), rel=1e-12)


# sizes spanning several i-rows (2048 per row) and j-chunks (128) with ragged tails
@pytest.mark.parametrize("n1,n2", [(1, 1), (1, 5), (7, 1), (129, 127), (2047, 2049), (4097, 300), (5000, 4099)])
def test_ragged_cross_and_auto(acf, ctx, n1, n2):
    c = synth.catalogs(n1, n2, 3 if n1 >= 6 else 0, 30.0, seed=1000 + n1 + n2)
    _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)
    _compare(acf, ctx, c.ra_d, c.dec_d, None, None, 0.25, 720)
    _compare(acf, ctx, c.ra_r, c.dec_r, None, None, 0.25, 720)


@pytest.mark.parametrize("w,nb,layout", [
    (0.25, 720, 0),     # direct map, lane-private copies
    (0.25, 720, 2),     # direct map, forced block-shared histogram
    (0.25, 1440, 0),    # the page's 1440 bins: bins beyond 180 degrees stay empty
    (0.25, 100, 0),     # bins stop at 25 degrees: the rest is clamped into bin 99
    (0.35, 515, 0),     # 180/w not an integer: clamp map
    (0.35, 40, 0),      # clamp map with heavy clamping
    (1.0, 180, 0),
    (10.0, 18, 0),
    (45.0, 4, 0),       # tiny P: still the direct map (P odd: no dot form)
    (60.0, 3, 0),       # P = 3 < 4: clamp map
    (0.01, 18000, 0),   # fine binning: block-shared layout
    (0.03, 2000, 0),    # 6000 half-turn bins, 2000 used: direct map, block layout
    (7.0, 1, 0),        # one bin
])
def test_binnings(acf, ctx, w, nb, layout):
    c = synth.catalogs(1500, 1200, 8, 60.0, seed=77)
    ctx.set_option("layout", layout)
    try:
        _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, w, nb)
        _compare(acf, ctx, c.ra_d, c.dec_d, None, None, w, nb)
    finally:
        ctx.set_option("layout", 0)


@pytest.mark.parametrize("threads", [512, 1024])
def test_thread_counts(acf, ctx, threads):
    c = synth.catalogs(3000, 2500, 10, 30.0, seed=5)
    ctx.set_option("threads", threads)
    try:
        _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)
        _compare(acf, ctx, c.ra_d, c.dec_d, None, None, 0.25, 720)
        assert ctx.info("threads") == threads
    finally:
        ctx.set_option("threads", 0)


def test_small_field_contention(acf, ctx):
    c = synth.catalogs(3000, 3000, 40, 3.0, seed=3, patch_arcmin=300.0)
    dd, _, _ = _compare(acf, ctx, c.ra_d, c.dec_d, None, None, 0.25, 720)
    assert dd[40:].sum() == 0  # a 5x5 degree patch has no pair beyond ~7.1 degrees
    _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)


def test_special_pairs(acf, ctx):
    # duplicates, exact antipodes, poles, equator, RA wrap: all land where the oracle puts them
    ra = np.array([0.0, 0.0, 10800.0, 21599.99, 5.0, 1234.5, 1234.5, 77.25, 300.0, 300.0], np.float32)
    dec = np.array([0.0, 0.0, 0.0, 0.0, 5400.0, -5400.0, 5400.0, 0.0, 100.0, -100.0], np.float32)
    _compare(acf, ctx, ra, dec, None, None, 0.25, 720)
    ra2 = np.where(ra < 10800, ra + 10800, ra - 10800).astype(np.float32)
    g = acf.as_uint64(ctx.histogram(ra, dec, ra2, -dec, bin_width_deg=0.25, nbins=720))
    torch.cuda.synchronize()
    o = oracle.histogram(ra, dec, ra2, -dec, 0.25, 720)
    assert check.edge_flux(g, o.hist, o.near_below, o.near_above).ok
    pb = ctx.pair_bins(ra, dec, ra2, -dec, 0.25, 720).cpu().numpy()
    assert np.all(pb == 719)  # exact antipodes: the last bin


def test_empty_inputs_give_zero_histograms(acf, ctx):
    e = np.zeros(0, np.float32)
    one = np.ones(3, np.float32)
    for args in ((e, e, None, None), (e, e, one, one), (one, one, e, e)):
        g = ctx.histogram(*args, bin_width_deg=0.25, nbins=720)
        torch.cuda.synchronize()
        assert int(acf.as_uint64(g).sum()) == 0


def test_argument_errors_return_codes(acf, ctx):
    d = torch.zeros(4, device="cuda")
    out = torch.empty(720, dtype=torch.int64, device="cuda")
    h = ctx.handle
    lib = acf.load()
    P = lambda t: t.data_ptr()
    assert lib.acf_histogram(h, P(d), P(d), -1, None, None, 0, 0.25, 720, P(out)) == acf.ACF_ERR_ARG
    assert lib.acf_histogram(h, P(d), P(d), 4, None, None, 0, 0.0, 720, P(out)) == acf.ACF_ERR_ARG
    assert lib.acf_histogram(h, P(d), P(d), 4, None, None, 0, float("nan"), 720, P(out)) == acf.ACF_ERR_ARG
    assert lib.acf_histogram(h, P(d), P(d), 4, None, None, 0, 0.25, 0, P(out)) == acf.ACF_ERR_ARG
    assert lib.acf_histogram(h, P(d), P(d), 4, None, None, 0, 0.25, 720, None) == acf.ACF_ERR_ARG
    assert lib.acf_histogram(h, P(d), P(d), 4, P(d), None, 4, 0.25, 720, P(out)) == acf.ACF_ERR_ARG
    assert lib.acf_histogram(h, P(d), P(d), 4, None, None, 0, 1e-4, 10**6, P(out)) == acf.ACF_ERR_UNSUPPORTED
    assert "exceeds" in acf.acf_last_error(h)
    assert lib.acf_omega(h, P(out), P(out), P(out), 0, 1, 1, P(out)) == acf.ACF_ERR_ARG
    assert lib.acf_set_option(h, b"no_such_option", 1) == acf.ACF_ERR_ARG
    assert lib.acf_set_option(h, b"threads", 256) == acf.ACF_ERR_ARG
    # the context still works afterwards
    c = synth.catalogs(100, 100, 0, 0.0, seed=1)
    _compare(acf, ctx, c.ra_d, c.dec_d, None, None, 0.25, 720)


def test_correlate_host_matches_device_path(acf, ctx):
    c = synth.catalogs(2500, 2200, 10, 30.0, seed=9)
    dd, dr, rr, om = ctx.correlate_host(c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)
    tdd = ctx.histogram(c.ra_d, c.dec_d, bin_width_deg=0.25, nbins=720)
    tdr = ctx.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, bin_width_deg=0.25, nbins=720)
    trr = ctx.histogram(c.ra_r, c.dec_r, bin_width_deg=0.25, nbins=720)
    tom = ctx.omega(tdd, tdr, trr, c.n_d, c.n_r)
    torch.cuda.synchronize()
    assert np.array_equal(dd, acf.as_uint64(tdd))
    assert np.array_equal(dr, acf.as_uint64(tdr))
    assert np.array_equal(rr, acf.as_uint64(trr))
    assert check.omega_close(om, tom.cpu().numpy(), rel=0.0)
    assert check.omega_close(om, oracle.omega(dd, dr, rr, c.n_d, c.n_r), rel=1e-12)


def test_correlate_equals_separate_histograms(acf, ctx):
    # one call, each catalog prepared once: the same counts as three histogram calls, and the
    # same omega as acf_omega on them
    c = synth.catalogs(5000, 6100, 12, 30.0, seed=19)
    dd, dr, rr, om = ctx.correlate(c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)
    tdd = ctx.histogram(c.ra_d, c.dec_d, bin_width_deg=0.25, nbins=720)
    tdr = ctx.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, bin_width_deg=0.25, nbins=720)
    trr = ctx.histogram(c.ra_r, c.dec_r, bin_width_deg=0.25, nbins=720)
    tom = ctx.omega(tdd, tdr, trr, c.n_d, c.n_r)
    torch.cuda.synchronize()
    for a, b in ((dd, tdd), (dr, tdr), (rr, trr)):
        assert torch.equal(a, b)
    assert check.omega_close(om.cpu().numpy(), tom.cpu().numpy(), rel=0.0)
    o = oracle.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)
    assert check.edge_flux(acf.as_uint64(dr), o.hist, o.near_below, o.near_above).ok


def _pair_sets(n, seed):
    """Random pairs over the whole sphere, tight pairs (< 1 deg), near-antipodal pairs, pairs near
    90 degrees, where the kernel switches between the difference and the sum chord, pairs near 55
    and 125 degrees, the edges of the dot form's range, and near 72 and 108, the short chord's."""
    rng = np.random.default_rng(seed)
    ra1, dec1 = synth.uniform_sphere(n, seed)
    ra2, dec2 = synth.uniform_sphere(n, seed + 1)
    sets = [(ra1, dec1, ra2, dec2)]
    # tight: offsets up to 1 degree
    sets.append((ra1, dec1, (ra1 + rng.uniform(-60, 60, n)).astype(np.float32) % np.float32(21600),
                 np.clip(dec1 + rng.uniform(-60, 60, n), -5400, 5400).astype(np.float32)))
    # near antipodal
    ra_a = np.where(ra1 < 10800, ra1 + 10800, ra1 - 10800) + rng.uniform(-60, 60, n)
    sets.append((ra1, dec1, (ra_a % 21600).astype(np.float32),
                 np.clip(-dec1 + rng.uniform(-60, 60, n), -5400, 5400).astype(np.float32)))
    # near 90 degrees: the pole against the equator band, plus equator pairs 90 degrees apart
    sets.append((ra1, np.full(n, 5400.0, np.float32) - rng.uniform(0, 30, n).astype(np.float32), ra2,
                 rng.uniform(-30, 30, n).astype(np.float32)))
    sets.append((ra1, np.zeros(n, np.float32), ((ra1 + 5400 + rng.uniform(-30, 30, n)) % 21600).astype(np.float32),
                 rng.uniform(-30, 30, n).astype(np.float32)))
    # near the edges of the dot form (55, 125 degrees) and of the short chord (72, 108 degrees)
    for lo in (53.0, 123.0, 70.0, 106.0):
        dra = rng.uniform(lo * 60, (lo + 4) * 60, n)
        sets.append((ra1, rng.uniform(-30, 30, n).astype(np.float32), ((ra1 + dra) % 21600).astype(np.float32),
                     rng.uniform(-30, 30, n).astype(np.float32)))
    return sets


@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("w,nb", [(0.25, 720), (0.01, 18000), (0.35, 515)])
def test_per_pair_bins_only_move_within_tolerance_of_an_edge(acf, ctx, w, nb, form):
    # form 0: the full-range chord form for every pair; form 1: the form a tightly bounded group
    # computes: the dot form wherever |u.v| < cos 55 deg, the short chord where |u.v| > cos 72 deg
    w_rad = math.radians(w)
    worst = 0.0
    ctx.set_option("pair_bins_form", form)
    try:
        for s in _pair_sets(400_000, seed=123):
            ra1, dec1, ra2, dec2 = (np.ascontiguousarray(a, dtype=np.float32) for a in s)
            gb = ctx.pair_bins(ra1, dec1, ra2, dec2, w, nb).cpu().numpy()
            ob = oracle.pair_bin(ra1, dec1, ra2, dec2, w, nb)
            th = oracle.pair_theta(ra1, dec1, ra2, dec2)
            bad = np.nonzero(gb != ob)[0]
            if len(bad):
                assert np.all(np.abs(gb[bad] - ob[bad]) == 1)
                edge = np.maximum(gb[bad], ob[bad]) * w_rad
                dist = np.abs(th[bad] - edge)
                worst = max(worst, float(dist.max()))
                assert np.all(dist < TOL), f"moved pair {float(dist.max()):.3e} rad from its edge"
    finally:
        ctx.set_option("pair_bins_form", 0)
    print(f"w={w} form={form}: largest distance from the edge of a moved pair {worst:.3e} rad")


@pytest.mark.parametrize("forms,exact", [(0, 1), (0, 0), (1, 2)])
def test_auto_correlation_decomposes_into_parts(acf, ctx, forms, exact):
    # DD(A u B) = DD(A) + DD(B) + 2 X(A, B) exactly. With the full-range chord form alone
    # (range_forms 0) the symmetric and the cross path bin every pair identically whatever its
    # grouping; with the range forms a pair near an edge may bin differently in another grouping,
    # unless exact mode 2 re-decides every near-edge pair in fp64.
    c = synth.catalogs(9000, 0, 20, 30.0, seed=8)
    a, b = slice(0, 4100), slice(4100, 9000)
    ctx.set_option("range_forms", forms)
    ctx.set_option("exact", exact)
    try:
        full = acf.as_uint64(ctx.histogram(c.ra_d, c.dec_d, bin_width_deg=0.25, nbins=720)).astype(object)
        da = acf.as_uint64(ctx.histogram(c.ra_d[a], c.dec_d[a], bin_width_deg=0.25, nbins=720)).astype(object)
        db = acf.as_uint64(ctx.histogram(c.ra_d[b], c.dec_d[b], bin_width_deg=0.25, nbins=720)).astype(object)
        x = acf.as_uint64(ctx.histogram(c.ra_d[a], c.dec_d[a], c.ra_d[b], c.dec_d[b], bin_width_deg=0.25,
                                        nbins=720)).astype(object)
        torch.cuda.synchronize()
    finally:
        ctx.set_option("range_forms", 1)
        ctx.set_option("exact", DEFAULT_EXACT)
    assert list(full) == list(da + db + 2 * x)


def test_acos_method_keeps_totals(acf, ctx):
    # the page's dot + acos route: a measured alternative. Its totals are exact; its bins are
    # not held to the 1e-6 rad rule (fp32 arccos near 0 and 180 degrees is too coarse).
    c = synth.catalogs(3000, 2000, 10, 30.0, seed=10)
    ctx.set_option("bin_method", 1)
    try:
        g = acf.as_uint64(ctx.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, bin_width_deg=0.25, nbins=720))
        s = acf.as_uint64(ctx.histogram(c.ra_d, c.dec_d, bin_width_deg=0.25, nbins=720))
        torch.cuda.synchronize()
        assert int(g.sum()) == 3000 * 2000 and int(s.sum()) == 3000 * 3000
        o = oracle.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)
        assert np.abs(g.astype(np.int64) - o.hist.astype(np.int64)).sum() < 0.01 * g.sum()
    finally:
        ctx.set_option("bin_method", 0)


def test_kernel_timing_records_launches(acf, ctx):
    c = synth.catalogs(2000, 2000, 0, 0.0, seed=2)
    try:
        # 1: the pair kernels; 2: the exact-mode fix-ups (one after each pair launch), for the
        # per-j records (720 bins) and the group records (18,000 bins, 3 launches forced)
        for mode in (1, 2):
            ctx.set_option("kernel_timing", mode)
            ctx.histogram(c.ra_d, c.dec_d, bin_width_deg=0.25, nbins=720)
            ctx.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, bin_width_deg=0.25, nbins=720)
            t = ctx.kernel_times()
            assert len(t) == 2 and all(x > 0 for x in t), (mode, t)
        ctx.set_option("units_per_launch", 50)
        ctx.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, bin_width_deg=0.01, nbins=18000)
        assert ctx.info("layout") == 2
        launches = ctx.info("launches")
        t = ctx.kernel_times()
        assert launches >= 3 and len(t) == launches and all(x > 0 for x in t), (launches, t)
        with pytest.raises(acf.AcfError):
            ctx.set_option("kernel_timing", 3)
    finally:
        ctx.set_option("units_per_launch", 0)
        ctx.set_option("kernel_timing", 0)


@pytest.mark.parametrize("layout", [1, 2])
def test_split_launches_accumulate(acf, ctx, layout):
    # a few work units per launch: later launches add into the block rows of earlier ones
    c = synth.catalogs(3000, 2600, 10, 30.0, seed=12)
    ctx.set_option("units_per_launch", 7)
    ctx.set_option("layout", layout)
    try:
        _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)
        assert ctx.info("launches") == -(-ctx.info("units") // 7)
        _compare(acf, ctx, c.ra_d, c.dec_d, None, None, 0.25, 720)
        assert ctx.info("launches") > 1
    finally:
        ctx.set_option("units_per_launch", 0)
        ctx.set_option("layout", 0)


# widths chosen so the edge windows are tight for a form: 180/2556 deg leaves the dot form a
# window only 0.02% wider than its worst-case error of 6e-7 rad (S = 11), 0.1478 deg the full-range
# chord (clamp map, S = 11) 0.4% wider
@pytest.mark.parametrize("w,nb", [(0.25, 720), (0.35, 515), (0.01, 18000), (0.25, 1440), (180.0 / 2556, 2556),
                                  (0.1478, 1218)])
def test_exact_mode_2_equals_oracle_bin_for_bin(acf, ctx, w, nb):
    c = synth.catalogs(4000, 3100, 12, 30.0, seed=14)
    ctx.set_option("exact", 2)
    try:
        for args in ((c.ra_d, c.dec_d, None, None), (c.ra_d, c.dec_d, c.ra_r, c.dec_r)):
            g, o, rep = _compare(acf, ctx, *args, w, nb)
            assert np.array_equal(g, o.hist), rep
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)


def test_pairs_exactly_on_edges_take_the_fp64_fallback(acf, ctx):
    # Equator galaxies 15 arcmin apart and meridian galaxies 15 arcmin apart: every separation is a
    # whole number of 0.25-degree bins, so every pair lies exactly on an edge. The fp32 code flags
    # them, the double-single pass cannot settle them (q equals the edge value to far below its
    # error bound), and the fp64 re-decision decides. A pair exactly on an edge may land on either
    # side within the rounding of the fp64 formula, which the edge rule allows.
    ra_eq = (7.5 + 15.0 * np.arange(200)).astype(np.float32)
    dec_eq = np.zeros(200, np.float32)
    dec_mer = (-2970.0 + 15.0 * np.arange(396)).astype(np.float32)
    ra_mer = np.full(396, 1000.0, np.float32)
    ctx.set_option("exact", 2)
    try:
        for ra, dec in ((ra_eq, dec_eq), (ra_mer, dec_mer)):
            _compare(acf, ctx, ra, dec, None, None, 0.25, 720)
            flagged, redone = ctx.info("exact_flagged"), ctx.info("exact_redone_fp64")
            n = len(ra)
            assert redone > 0 and redone <= flagged
            assert flagged >= n * (n - 1) // 2 // 2  # most of the off-diagonal pairs are on an edge
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)


def test_largest_histogram_that_fits_and_the_next_is_refused(acf, ctx):
    # The block-shared histogram (512 threads, 16 warps' 4 KB j-tiles) fills the shared memory at
    # 41,216 entries. Direct map (180/w integral): P + 2 entries, so P = 41214 is the largest; clamp
    # map: nbins entries when nbins <= floor(P) + 1. Both must still equal the oracle bin for bin
    # (exact mode 2); one entry more must be refused, and the context must keep working.
    c = synth.catalogs(1500, 1200, 6, 60.0, seed=71)
    lib = acf.load()
    ctx.set_option("exact", 2)
    try:
        for w, nb in ((180.0 / 41214, 41214), (180.0 / 41189.9, 41190)):
            for args in ((c.ra_d, c.dec_d, None, None), (c.ra_d, c.dec_d, c.ra_r, c.dec_r)):
                g, o, rep = _compare(acf, ctx, *args, w, nb)
                assert np.array_equal(g, o.hist), (w, nb, rep)
            assert ctx.info("hist_entries") in (41216, 41190) and ctx.info("threads") == 512
        ra, dec = torch.from_numpy(c.ra_d).cuda(), torch.from_numpy(c.dec_d).cuda()
        for w, nb in ((180.0 / 41216, 41216), (180.0 / 41300.5, 41217)):
            out = torch.empty(nb, dtype=torch.int64, device="cuda")
            rc = lib.acf_histogram(ctx.handle, ra.data_ptr(), dec.data_ptr(), c.n_d, None, None, 0, w, nb,
                                   out.data_ptr())
            assert rc == acf.ACF_ERR_UNSUPPORTED, (w, nb, rc)
            assert "shared memory" in acf.acf_last_error(ctx.handle)
        _compare(acf, ctx, c.ra_d, c.dec_d, None, None, 0.25, 720)
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)


def test_coincident_galaxies_overflow_the_queue_and_stay_exact(acf, ctx):
    # 2000 copies of one galaxy and 2000 of another 10.3 degrees away: 8M ordered pairs at
    # separation 0 and 8M at 10.3 degrees (bin 41 of 0.25). Every pair at separation 0 lies within
    # one fine unit above the edge at 0 and is flagged: 4M unordered pairs, in flag records of up to
    # 128 pairs each. With the automatic queue they all fit; with a queue of 1000 records most
    # overflow. An overflowed pair keeps its fp32 bin, which is exact here, and the overflow is
    # reported.
    ra = np.concatenate([np.full(2000, 600.0), np.full(2000, 600.0)]).astype(np.float32)
    dec = np.concatenate([np.full(2000, 100.0), np.full(2000, 100.0 + 618.0)]).astype(np.float32)
    expect = np.zeros(720, np.uint64)
    expect[0] = 2 * 2000 * 2000
    expect[int(618.0 / 15.0)] = 2 * 2000 * 2000
    ctx.set_option("exact", 2)
    try:
        for cap in (0, 1000):
            ctx.set_option("exact_queue", cap)
            g = acf.as_uint64(ctx.histogram(ra, dec, bin_width_deg=0.25, nbins=720))
            torch.cuda.synchronize()
            assert np.array_equal(g, expect), cap
            assert ctx.info("exact_flagged") >= 2 * 1999 * 1000
            assert (ctx.info("exact_overflow") > 0) == (cap > 0), cap
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)
        ctx.set_option("exact_queue", 0)


@pytest.mark.parametrize("line", ["equator", "meridian"])
@pytest.mark.parametrize("w,nb", [(0.25, 720), (0.01, 18000)])
def test_dense_sweep_across_every_edge(acf, ctx, w, nb, line):
    # equator: 128 copies of the point (0, 0) against 172,800 equator points every 1/8 arcmin around
    # the circle, separations min(ra, 21600 - ra); meridian: 128 copies of the south pole against
    # 86,401 points every 1/8 arcmin from pole to pole on one meridian, separations dec + 5400.
    # Every separation is exact, a dense sweep over every edge, with the i-set a single point so the
    # caps put whole j-groups on each form (dot form, short and full chords, both sides of 90
    # degrees). The only pairs within 1e-6 rad of an edge are those exactly on it (the grid step is
    # 3.6e-5 rad), so the edge-flux check leaves room for nothing else. That holds in exact mode 2
    # and, given its error bounds, in mode 0 too.
    if line == "equator":
        ra_a, dec_a = np.zeros(128, np.float32), np.zeros(128, np.float32)
        ra_b = (np.arange(172_800) / 8.0).astype(np.float32)
        dec_b = np.zeros(172_800, np.float32)
    else:
        ra_a, dec_a = np.zeros(128, np.float32), np.full(128, -5400.0, np.float32)
        dec_b = (-5400.0 + np.arange(86_401) / 8.0).astype(np.float32)
        ra_b = np.zeros(86_401, np.float32)
    o = oracle.histogram(ra_a, dec_a, ra_b, dec_b, w, nb)
    on_edge = o.near_below.sum() + o.near_above.sum()
    assert on_edge <= 2 * 128 * (2 * nb)  # only pairs exactly on an edge lie within 1e-6 rad of one
    for exact in (2, 0):
        ctx.set_option("exact", exact)
        try:
            g = acf.as_uint64(ctx.histogram(ra_a, dec_a, ra_b, dec_b, bin_width_deg=w, nbins=nb))
            torch.cuda.synchronize()
        finally:
            ctx.set_option("exact", DEFAULT_EXACT)
        rep = check.edge_flux(g, o.hist, o.near_below, o.near_above)
        assert int(g.sum()) == 128 * len(ra_b)
        assert rep.ok, (exact, str(rep))


def test_exact_mode_off_still_meets_edge_rule(acf, ctx):
    c = synth.catalogs(4000, 3100, 12, 30.0, seed=15)
    ctx.set_option("exact", 0)
    try:
        _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)
        _compare(acf, ctx, c.ra_d, c.dec_d, None, None, 0.25, 720)
        assert ctx.info("exact_flagged") == 0
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)


PATH_KEYS = ("pairs_fixed", "pairs_general", "pairs_fixed_exact", "pairs_general_exact", "pairs_masked",
             "pairs_mid", "pairs_mid_exact", "pairs_small", "pairs_small_exact")


@pytest.mark.parametrize("exact", [1, 2])
def test_path_counters_cover_every_computed_pair(acf, ctx, exact):
    c = synth.catalogs(5000, 4100, 12, 30.0, seed=16)
    ctx.set_option("exact", exact)
    try:
        ctx.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, bin_width_deg=0.25, nbins=720)
        got = {k: ctx.info(k) for k in PATH_KEYS}
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)
    rows = -(-5000 // 128)
    # every unit computes its whole 128-wide i-set against the j-chunk's real length
    assert sum(got.values()) == rows * 128 * 4100, got
    assert got["pairs_masked"] > 0
    if exact == 1:
        assert got["pairs_mid"] > 0 and got["pairs_small"] > 0
        assert got["pairs_small_exact"] > 0  # groups near 0 and 180 degrees: short chord with flags
        assert got["pairs_mid_exact"] == 0  # exact mode 1 never sends a group to the dot form
    else:
        # exact mode 2: every group flags near-edge pairs
        assert got["pairs_mid"] == got["pairs_small"] == got["pairs_fixed"] == got["pairs_general"] == 0
        assert got["pairs_mid_exact"] > 0 and got["pairs_small_exact"] > 0


@pytest.mark.parametrize("w,nb,mid_expected", [(0.25, 720, True), (4.0, 45, False), (0.35, 515, False)])
def test_range_forms_on_off_and_where_they_apply(acf, ctx, w, nb, mid_expected):
    # the dot form needs the direct map with P = 180 / w even (0.25 deg: P = 720; 4 deg: P = 45 is
    # odd; 0.35 deg: P is not an integer, clamp map); the short chord applies to every binning.
    # With the range forms on or off the edge rule holds.
    c = synth.catalogs(6000, 5000, 12, 30.0, seed=18)
    for forms in (1, 0):
        ctx.set_option("range_forms", forms)
        ctx.set_option("exact", 1)
        try:
            _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, w, nb)
            got = {k: ctx.info(k) for k in PATH_KEYS}
        finally:
            ctx.set_option("range_forms", 1)
            ctx.set_option("exact", DEFAULT_EXACT)
        assert (got["pairs_mid"] > 0) == (forms == 1 and mid_expected), got
        assert (got["pairs_small"] + got["pairs_small_exact"] > 0) == (forms == 1), got
    ctx.set_option("exact", 2)
    try:
        g, o, _ = _compare(acf, ctx, c.ra_d, c.dec_d, c.ra_r, c.dec_r, w, nb)
        assert np.array_equal(g, o.hist)
        if mid_expected:
            assert ctx.info("pairs_mid_exact") > 0 and ctx.info("pairs_mid") == 0
        assert ctx.info("pairs_small_exact") > 0 and ctx.info("pairs_small") == 0
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)


def test_kernel_launch_counter(acf, ctx):
    """kernel_launches counts every kernel of a call: eight catalog-preparation kernels (two radix-sort
    passes of count, scan and scatter, the vectors, the caps), which prepare both catalogs of a
    cross-correlation at once, the pair kernel and the merge, plus the edge tables and the fix-up in
    exact mode."""
    c = synth.catalogs(3000, 2500, 12, 30.0, seed=17)

    def launched(fn):
        before = ctx.info("kernel_launches")
        fn()
        return ctx.info("kernel_launches") - before

    assert launched(lambda: ctx.histogram(c.ra_d, c.dec_d, bin_width_deg=0.25, nbins=720)) == 8 + 2 + 2
    assert launched(lambda: ctx.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, bin_width_deg=0.25,
                                          nbins=720)) == 8 + 2 + 2
    # the whole job: both catalogs prepared once, one edge table, three histograms, omega
    assert launched(lambda: ctx.correlate(c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720)) == 8 + 1 + 3 * 3 + 1
    ctx.set_option("exact", 0)
    try:
        assert launched(lambda: ctx.histogram(c.ra_d, c.dec_d, bin_width_deg=0.25, nbins=720)) == 8 + 2
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)


def test_fp32_ceiling_probe_runs_the_arithmetic(acf, ctx):
    # the roofline's measured FP32 ceiling: a sane rate, and thread 0's chains replayed on the host
    # (fp32 fma emulated exactly in fp64: the product of two fp32 values and the sum with b = 1e-7
    # fit in 53 bits here, so one rounding to fp32 gives fmaf's result)
    iters = 1 << 14
    rate, t0 = acf.acf_fp32_peak(ctx.handle, iters)
    assert 5e12 < rate < 2e14, rate
    a, b = np.float64(np.float32(0.9999999)), np.float64(np.float32(1e-7))
    x = np.arange(8, dtype=np.float32)
    for _ in range(iters):
        x = (x.astype(np.float64) * a + b).astype(np.float32)
    s = np.float32(0.0)
    for c in range(8):
        s = np.float32(s + x[c])
    assert np.float32(t0) == s


def test_approximate_mode_keeps_totals_and_stays_near_the_edges(acf, ctx):
    # bin_method 2: dot product + the Abramowitz-Stegun 4.4.45 arccos polynomial (error <= 6.7e-5
    # rad plus fp32 dot-product error): totals exact, and every moved pair lies within 5e-4 rad of
    # an edge it crossed
    c = synth.catalogs(3000, 2500, 10, 30.0, seed=43)
    ctx.set_option("bin_method", 2)
    try:
        g = acf.as_uint64(ctx.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, bin_width_deg=0.25, nbins=720))
        ra1, dec1 = synth.uniform_sphere(200_000, 77)
        ra2, dec2 = synth.uniform_sphere(200_000, 78)
        gb = ctx.pair_bins(ra1, dec1, ra2, dec2, 0.25, 720).cpu().numpy()
        torch.cuda.synchronize()
    finally:
        ctx.set_option("bin_method", 0)
    assert int(g.sum()) == 3000 * 2500
    ob = oracle.pair_bin(ra1, dec1, ra2, dec2, 0.25, 720)
    th = oracle.pair_theta(ra1, dec1, ra2, dec2)
    bad = np.nonzero(gb != ob)[0]
    assert len(bad) > 0 and np.all(np.abs(gb[bad] - ob[bad]) == 1)
    edge = np.maximum(gb[bad], ob[bad]) * math.radians(0.25)
    assert float(np.abs(th[bad] - edge).max()) < 5e-4
