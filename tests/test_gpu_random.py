"""Seeded random cases against the oracle: catalog sizes, clustering, bin widths (with 180/w an
integer, odd or even, or not), bin counts that stop short of 180 degrees or run past it, and the
three exact modes, with the automatic work units or chunk-pair units forced. Every case must pass the edge-flux rule and sum to n1*n2. In exact mode 2 every
case must equal the oracle bin for bin, except where a pair lies within 1e-15 relative of an edge;
none does in practice.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import check

pytestmark = pytest.mark.gpu

N_CASES = int(os.environ.get("ACF_RANDOM_CASES", "200"))  # a longer sweep on request (1000 passed)


def _case(k):
    rng = np.random.default_rng(1000 + k)
    n1 = int(rng.choice([1, 7, 31, 128, 129, 500, 1777, 3000]))
    n2 = int(rng.choice([0, 1, 33, 256, 999, 2500]))  # 0: auto-correlation
    kind = rng.integers(3)
    if kind == 0:
        p = int(rng.choice([36, 180, 361, 720, 1001, 2556, 3600]))  # 180/w an integer
        w = 180.0 / p
    elif kind == 1:
        w = float(rng.uniform(0.05, 3.0))  # 180/w not an integer: the clamp map
    else:
        w = float(rng.choice([0.25, 0.5, 1.0, 0.01]))
    full = int(np.ceil(180.0 / w))
    nb = int(max(1, min(40000, rng.choice([full, full // 2 + 1, full + 7, 1 + rng.integers(full)]))))
    clumps = int(rng.choice([0, 3, 20]))
    sigma = float(rng.choice([1.0, 30.0, 300.0]))
    exact = int(rng.choice([0, 1, 2]))
    patch = float(rng.choice([0.0, 0.0, 300.0]))
    groups = int(rng.choice([0, 4]))  # automatic units (one j-group for these sizes), or chunk pairs
    return n1, n2, w, nb, clumps, sigma, exact, patch, k, groups


@pytest.fixture(scope="module")
def ctx(acf):
    c = acf.Context(0)
    yield c
    c.close()


@pytest.mark.parametrize("k", range(N_CASES))
def test_random_case(acf, ctx, k):
    n1, n2, w, nb, clumps, sigma, exact, patch, seed, groups = _case(k)
    c = synth.catalogs(n1, max(n2, 1), clumps, sigma, seed=500 + seed, patch_arcmin=patch)
    ra1, dec1 = c.ra_d, c.dec_d
    ra2, dec2 = (c.ra_r[:n2], c.dec_r[:n2]) if n2 else (None, None)
    ctx.set_option("exact", exact)
    ctx.set_option("unit_groups", groups)
    try:
        try:
            g = acf.as_uint64(ctx.histogram(ra1, dec1, ra2, dec2, bin_width_deg=w, nbins=nb))
        except acf.AcfError as e:
            # only a histogram larger than the shared memory may be refused
            assert e.code == acf.ACF_ERR_UNSUPPORTED, str(e)
            plan_ok = True
            try:
                acf.acf_plan_info(w, nb, exact)
                plan_ok = False
            except acf.AcfError as pe:
                assert pe.code == acf.ACF_ERR_UNSUPPORTED
            assert plan_ok
            return
        torch.cuda.synchronize()
    finally:
        ctx.set_option("exact", 2)
        ctx.set_option("unit_groups", 0)
    o = oracle.histogram(ra1, dec1, ra2, dec2, w, nb)
    m = n2 if n2 else n1
    assert int(g.sum()) == n1 * m
    rep = check.edge_flux(g, o.hist, o.near_below, o.near_above)
    assert rep.ok, (n1, n2, w, nb, exact, str(rep))
    if exact == 2:
        assert np.array_equal(g, o.hist), (n1, n2, w, nb, str(rep))
