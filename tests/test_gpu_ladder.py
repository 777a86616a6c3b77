"""The page's optimisation ladder (levels 0-5) rebuilt on this GPU: totals, the levels' bitwise
agreements the page reports ("the tiled output is bit-identical to the output of L2", L5's "output is
bit-identical to that of L4"), and how far their fp32 acos binning is from the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def runs(acf):
    c = synth.config(0)
    w, nb = c.bin_width_deg, c.nbins
    t = {k: torch.from_numpy(getattr(c, k)).cuda() for k in ("ra_d", "dec_d", "ra_r", "dec_r")}
    out = {}
    for level in range(6):
        h = [torch.empty(nb, dtype=torch.int64, device="cuda") for _ in range(3)]
        ms = acf.acf_ladder(level, t["ra_d"], t["dec_d"], t["ra_r"], t["dec_r"], w, nb, *h)
        assert ms > 0
        out[level] = [acf.as_uint64(x) for x in h]
    return c, out


def test_every_level_counts_every_pair(runs):
    c, out = runs
    for level, (dd, dr, rr) in out.items():
        assert int(dd.sum()) == c.n_d ** 2 and int(dr.sum()) == c.n_d * c.n_r and int(rr.sum()) == c.n_r ** 2, level


def test_levels_agree_where_the_arithmetic_is_the_same(runs):
    _, out = runs
    for a, b in ((1, 2), (2, 3), (4, 5)):
        for fam in range(3):
            assert np.array_equal(out[a][fam], out[b][fam]), (a, b, fam)
    # DR needs no symmetry, so levels 0 and 1 compute it identically
    assert np.array_equal(out[0][1], out[1][1])


def test_levels_against_the_oracle(runs):
    # fp32 arccos misbins pairs near edges (by up to ~3e-4 rad near 0 and 180 degrees, 6.7e-5 rad
    # more for the polynomial of levels 4 and 5): a small fraction of the pairs moves
    c, out = runs
    w, nb = c.bin_width_deg, c.nbins
    ref = (oracle.histogram(c.ra_d, c.dec_d, None, None, w, nb).hist,
           oracle.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, w, nb).hist,
           oracle.histogram(c.ra_r, c.dec_r, None, None, w, nb).hist)
    for level, hs in out.items():
        for g, o in zip(hs, ref):
            moved = int(np.abs(np.cumsum(g.astype(np.int64) - o.astype(np.int64))).sum())
            assert moved < 0.01 * int(o.sum()), (level, moved)
