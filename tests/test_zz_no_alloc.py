"""acf_histogram_noalloc: the histogram for callers that cannot allocate device memory.

Such callers (a process whose device memory all belongs to another allocator, or code that cannot
afford the device synchronisation an allocation brings) get their scratch from the library's
static 16 MiB device array. This file checks, through the C ABI, that two calls in a row give
exactly the counts of the allocating entry point (histogram counts are integers, so the tolerance
is zero), that its results obey the oracle's edge rule, and that requests larger than the static
array are refused with a clear error. When the static array's exact-mode queue overflows, the
call still succeeds, reports the shortfall and keeps the totals and the edge rule. It is named to run last so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import check

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_no_alloc_matches_allocating_entry_point_twice(acf):
    ctx = acf.Context(0)
    lib = acf.load()
    c = synth.catalogs(6000, 5000, 10, 30.0, seed=321)
    ra_d, dec_d, ra_r, dec_r = map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r))
    w, nb = 0.25, 720
    calls = [(ra_d, dec_d, c.n_d, None, None, 0),          # DD (auto-correlation)
             (ra_d, dec_d, c.n_d, ra_r, dec_r, c.n_r)]     # then DR: two calls in a row
    for ra1, dec1, n1, ra2, dec2, n2 in calls:
        ref = torch.empty(nb, dtype=torch.int64, device="cuda")
        got = torch.full((nb,), -1, dtype=torch.int64, device="cuda")
        acf.acf_histogram(ctx.handle, ra1, dec1, n1, ra2, dec2, n2, w, nb, ref)
        acf.acf_histogram_noalloc(ctx.handle, ra1, dec1, n1, ra2, dec2, n2, w, nb, got)
        torch.cuda.synchronize()
        assert torch.equal(ref, got)
        g = acf.as_uint64(got)
        o = oracle.histogram(c.ra_d, c.dec_d, None if ra2 is None else c.ra_r, None if ra2 is None else c.dec_r,
                             w, nb)
        assert check.edge_flux(g, o.hist, o.near_below, o.near_above).ok
        assert int(g.sum()) == n1 * (n2 if ra2 is not None else n1)
    # too large for the static array (20k galaxies fill the 152-block grid; 152 x 18000 bins x
    # 8 bytes of block rows = 21.9 MB): refused, and the context keeps working
    big = synth.catalogs(20000, 0, 0, 0.0, seed=5)
    ra_b, dec_b = _dev(big.ra_d), _dev(big.dec_d)
    out = torch.empty(18000, dtype=torch.int64, device="cuda")
    rc = lib.acf_histogram_noalloc(ctx.handle, ra_b.data_ptr(), dec_b.data_ptr(), big.n_d, None, None, 0, 0.01,
                                   18000, out.data_ptr())
    assert rc == acf.ACF_ERR_UNSUPPORTED
    assert "static array" in acf.acf_last_error(ctx.handle)
    ref = torch.empty(nb, dtype=torch.int64, device="cuda")
    got = torch.empty(nb, dtype=torch.int64, device="cuda")
    acf.acf_histogram(ctx.handle, ra_r, dec_r, c.n_r, None, None, 0, w, nb, ref)
    acf.acf_histogram_noalloc(ctx.handle, ra_r, dec_r, c.n_r, None, None, 0, w, nb, got)
    torch.cuda.synchronize()
    assert torch.equal(ref, got)
    ctx.close()


def test_no_alloc_queue_overflow_keeps_sums_and_edge_rule(acf):
    # Two 60k catalogs fit the static array (about 10 MB of vectors, caps and block rows), but the
    # ~6 MB left for the exact-mode queue holds far fewer pairs than their DR histogram flags near
    # bin edges. The pairs that do not fit keep their fp32 bin: the call still succeeds, reports the
    # shortfall, keeps every total exact and stays within the edge rule against the oracle.
    ctx = acf.Context(0)
    c = synth.catalogs(60000, 60000, 20, 30.0, seed=17)
    ra_d, dec_d, ra_r, dec_r = map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r))
    w, nb = 0.25, 720
    got = torch.full((nb,), -1, dtype=torch.int64, device="cuda")
    acf.acf_histogram_noalloc(ctx.handle, ra_d, dec_d, c.n_d, ra_r, dec_r, c.n_r, w, nb, got)
    torch.cuda.synchronize()
    overflow, flagged = ctx.info("exact_overflow"), ctx.info("exact_flagged")
    assert overflow > 0 and flagged > overflow, (overflow, flagged)
    g = acf.as_uint64(got)
    assert int(g.sum()) == c.n_d * c.n_r
    o = oracle.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, w, nb)
    rep = check.edge_flux(g, o.hist, o.near_below, o.near_above)
    assert rep.ok, rep
    ctx.close()


def test_no_alloc_group_records_split_launches(acf):
    # 2000 bins of 0.09 deg take the block-shared histogram, whose exact mode keeps its flags in
    # group records: a fixed slot for every lane and j-group of every unit of a launch. What the
    # static array has left after two 20k catalogs and 152 block rows holds a few thousand units,
    # so the call runs more, smaller launches than the allocating one; the histograms must still be
    # equal to it and to the oracle, bin for bin.
    ctx = acf.Context(0)
    c = synth.catalogs(20000, 20000, 20, 30.0, seed=23)
    ra_d, dec_d, ra_r, dec_r = map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r))
    w, nb = 0.09, 2000
    for ra2, dec2, n2 in ((None, None, 0), (ra_r, dec_r, c.n_r)):
        ref = torch.empty(nb, dtype=torch.int64, device="cuda")
        got = torch.full((nb,), -1, dtype=torch.int64, device="cuda")
        acf.acf_histogram(ctx.handle, ra_d, dec_d, c.n_d, ra2, dec2, n2, w, nb, ref)
        launches_alloc = ctx.info("launches")
        acf.acf_histogram_noalloc(ctx.handle, ra_d, dec_d, c.n_d, ra2, dec2, n2, w, nb, got)
        torch.cuda.synchronize()
        assert ctx.info("layout") == 2
        assert ctx.info("launches") > launches_alloc, (ctx.info("launches"), launches_alloc)
        assert ctx.info("exact_overflow") == 0
        assert torch.equal(ref, got)
        g = acf.as_uint64(got)
        o = oracle.histogram(c.ra_d, c.dec_d, None if ra2 is None else c.ra_r, None if ra2 is None else c.dec_r,
                             w, nb)
        assert np.array_equal(g, o.hist)
    ctx.close()
