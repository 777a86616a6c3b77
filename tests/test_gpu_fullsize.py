"""Full-size workloads through the library in the launch configuration bench.py times.

- The pages' shape (two 100k catalogs) and the 5x5 degree field: every bin against the oracle's
  stored full histograms (tests/golden/, written by make_golden.py from oracle/ only), after
  proving the regenerated catalogs are the ones the golden files were computed from.
- The fine-binning workload (two 200k catalogs, 18,000 bins of 0.01 degrees): every bin against the
  oracle's stored full histograms too (the oracle needs minutes for it, so it ran once, offline).
- The 1M and the fine-binning workloads: 2000 seeded random rows of each family are checked
  against the oracle's edge rule (the GPU histogram of those rows against the full catalog vs the
  oracle's), and the full-size histograms are checked for their exact totals (n1*n2) and the DD
  split identity.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import check

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DEFAULT_EXACT = 2


@pytest.fixture(scope="module")
def ctx(acf):
    c = acf.Context(0)
    yield c
    c.close()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("exact", [2, 1, 0])
@pytest.mark.parametrize("idx", [1, 2])
def test_full_histograms_match_golden_oracle(acf, ctx, idx, exact):
    # the whole job through acf_correlate, in the launch configuration bench.py times (exact mode 2,
    # the default), and in the cheaper exact modes 1 and 0
    with open(os.path.join(GOLDEN, f"config{idx}_oracle.json")) as f:
        g = json.load(f)
    c = synth.config(idx)
    assert c.digest() == g["digest"], "regenerated catalogs differ from the ones the golden file was made from"
    w, nb = c.bin_width_deg, c.nbins
    ra_d, dec_d, ra_r, dec_r = map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r))
    ctx.set_option("exact", exact)
    try:
        dd, dr, rr, om = ctx.correlate(ra_d, dec_d, ra_r, dec_r, w, nb)
        torch.cuda.synchronize()
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)
    gpu = {"DD": acf.as_uint64(dd), "DR": acf.as_uint64(dr), "RR": acf.as_uint64(rr)}
    moved = {}
    for fam in ("DD", "DR", "RR"):
        ref = g[fam]
        rep = check.edge_flux(gpu[fam], np.array(ref["hist"], np.uint64), np.array(ref["near_below"], np.uint64),
                              np.array(ref["near_above"], np.uint64))
        assert rep.ok, f"{fam}: {rep}"
        assert int(gpu[fam].sum()) == 10**10
        moved[fam] = rep.moved_pairs
    # omega from the GPU counts equals the oracle's omega of the same counts
    om = om.cpu().numpy()
    assert check.omega_close(om, oracle.omega(gpu["DD"], gpu["DR"], gpu["RR"], c.n_d, c.n_r), rel=1e-12)
    # against the oracle's own counts: bins whose three counts agree give the same omega; report the rest
    ref_om = np.array([np.nan if x is None else x for x in g["omega"]])
    rr_ref = np.array(g["RR"]["hist"], np.float64)
    same = np.all([gpu[f] == np.array(g[f]["hist"], np.uint64) for f in ("DD", "DR", "RR")], axis=0)
    big = rr_ref >= 1000
    assert np.allclose(om[same & big], ref_om[same & big], rtol=1e-12, atol=0)
    dev = np.abs(om[big] - ref_om[big])
    print(f"config {idx} exact {exact}: net moved pairs {moved}; bins with RR>=1000: {int(big.sum())}, of which "
          f"{int((big & ~same).sum())} hold a moved pair; max |d omega| = {float(dev.max()):.3e}")
    if exact == 2:
        # every near-edge pair re-decided in fp64: the oracle's histograms bin for bin, so the omega
        # rule (|d omega| <= 1e-5 on bins with RR >= 1000) holds with d omega = 0
        for fam in ("DD", "DR", "RR"):
            assert np.array_equal(gpu[fam], np.array(g[fam]["hist"], np.uint64)), fam
        assert float(dev.max()) == 0.0


def test_fine_binning_full_histograms_match_golden_oracle(acf, ctx):
    # two 200k catalogs in 18,000 bins of 0.01 degrees through acf_correlate, as bench.py --config 4
    # times it (exact mode 2, the default): every bin of DD, DR and RR equals the oracle's stored full
    # histograms. This is where the exact mode works hardest: about 1.2% of the pairs lie within
    # their form's window of an edge and are re-decided.
    with open(os.path.join(GOLDEN, "config4_oracle.json")) as f:
        g = json.load(f)
    c = synth.config(4)
    assert c.digest() == g["digest"], "regenerated catalogs differ from the ones the golden file was made from"
    assert (g["nbins"], g["bin_width_deg"]) == (18000, 0.01)
    ra_d, dec_d, ra_r, dec_r = map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r))
    dd, dr, rr, om = ctx.correlate(ra_d, dec_d, ra_r, dec_r, c.bin_width_deg, c.nbins)
    torch.cuda.synchronize()
    assert ctx.info("exact_overflow") == 0
    gpu = {"DD": acf.as_uint64(dd), "DR": acf.as_uint64(dr), "RR": acf.as_uint64(rr)}
    for fam, n in (("DD", c.n_d ** 2), ("DR", c.n_d * c.n_r), ("RR", c.n_r ** 2)):
        ref = np.array(g[fam]["hist"], np.uint64)
        assert int(ref.sum()) == n
        diff = np.flatnonzero(gpu[fam] != ref)
        assert diff.size == 0, f"{fam}: {diff.size} bins differ, first {diff[:5]}"
    # omega of the oracle's counts (the file stores only the histograms at this binning)
    om = om.cpu().numpy()
    ref_om = oracle.omega(*(np.array(g[f]["hist"], np.uint64) for f in ("DD", "DR", "RR")), c.n_d, c.n_r)
    assert np.array_equal(np.isnan(om), np.isnan(ref_om))
    ok = ~np.isnan(ref_om)
    assert np.allclose(om[ok], ref_om[ok], rtol=1e-12, atol=1e-15)


def _row_sample_check(acf, ctx, c, rows, seed):
    w, nb = c.bin_width_deg, c.nbins
    fams = (("DD", c.ra_d, c.dec_d, c.ra_d, c.dec_d, seed), ("DR", c.ra_d, c.dec_d, c.ra_r, c.dec_r, seed),
            ("RR", c.ra_r, c.dec_r, c.ra_r, c.dec_r, seed + 1))
    for fam, ra1, dec1, ra2, dec2, s in fams:
        idx = synth.sample_rows(len(ra1), rows, s)
        g = acf.as_uint64(ctx.histogram(ra1[idx], dec1[idx], ra2, dec2, bin_width_deg=w, nbins=nb))
        torch.cuda.synchronize()
        o = oracle.histogram(ra1[idx], dec1[idx], ra2, dec2, w, nb, threads=0)
        rep = check.edge_flux(g, o.hist, o.near_below, o.near_above)
        assert rep.ok, f"{c.name} {fam} rows: {rep}"


def _full_totals(acf, ctx, c):
    w, nb = c.bin_width_deg, c.nbins
    ra_d, dec_d, ra_r, dec_r = map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r))
    dd = acf.as_uint64(ctx.histogram(ra_d, dec_d, bin_width_deg=w, nbins=nb))
    assert ctx.info("exact_overflow") == 0
    dr = acf.as_uint64(ctx.histogram(ra_d, dec_d, ra_r, dec_r, bin_width_deg=w, nbins=nb))
    assert ctx.info("exact_overflow") == 0
    rr = acf.as_uint64(ctx.histogram(ra_r, dec_r, bin_width_deg=w, nbins=nb))
    torch.cuda.synchronize()
    assert int(dd.sum()) == c.n_d ** 2 and int(dr.sum()) == c.n_d * c.n_r and int(rr.sum()) == c.n_r ** 2
    # split identity on the full catalog: DD(A u B) = DD(A) + DD(B) + 2 X(A, B), exactly, with the
    # full-range chord form alone (with the range forms, the bin of a pair within ~4e-7 rad of an
    # edge may depend on the form its grouping picks)
    h = c.n_d // 3
    ctx.set_option("range_forms", 0)
    try:
        full = acf.as_uint64(ctx.histogram(ra_d, dec_d, bin_width_deg=w, nbins=nb)).astype(object)
        a = acf.as_uint64(ctx.histogram(ra_d[:h], dec_d[:h], bin_width_deg=w, nbins=nb)).astype(object)
        b = acf.as_uint64(ctx.histogram(ra_d[h:], dec_d[h:], bin_width_deg=w, nbins=nb)).astype(object)
        x = acf.as_uint64(ctx.histogram(ra_d[:h], dec_d[:h], ra_d[h:], dec_d[h:], bin_width_deg=w,
                                        nbins=nb)).astype(object)
        torch.cuda.synchronize()
    finally:
        ctx.set_option("range_forms", 1)
    assert list(full) == list(a + b + 2 * x)


def test_scale_1m_rows_and_totals(acf, ctx):
    c = synth.config(3)
    _row_sample_check(acf, ctx, c, 2000, seed=4)
    _full_totals(acf, ctx, c)


def test_fine_binning_200k_rows_and_totals(acf, ctx):
    c = synth.config(4)
    _row_sample_check(acf, ctx, c, 2000, seed=5)
    _full_totals(acf, ctx, c)


def test_exact_everywhere_is_bit_identical_at_full_size(acf, ctx):
    # exact mode 2 re-decides every pair within one fine unit of an edge in fp64
    with open(os.path.join(GOLDEN, "config1_oracle.json")) as f:
        g = json.load(f)
    c = synth.config(1)
    assert c.digest() == g["digest"]
    ctx.set_option("exact", 2)
    try:
        ra_d, dec_d, ra_r, dec_r = map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r))
        for fam, args in (("DD", (ra_d, dec_d)), ("DR", (ra_d, dec_d, ra_r, dec_r)), ("RR", (ra_r, dec_r))):
            h = acf.as_uint64(ctx.histogram(*args, bin_width_deg=c.bin_width_deg, nbins=c.nbins))
            torch.cuda.synchronize()
            assert np.array_equal(h, np.array(g[fam]["hist"], np.uint64)), fam
            assert ctx.info("exact_overflow") == 0
            # the double-single pass decides all but a sliver; the rest is redone in fp64
            flagged, redone = ctx.info("exact_flagged"), ctx.info("exact_redone_fp64")
            assert flagged > 0 and redone * 1000 <= flagged, (fam, flagged, redone)
    finally:
        ctx.set_option("exact", DEFAULT_EXACT)
