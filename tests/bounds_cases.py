"""Run a spread of histogram cases through the bounds-checked library (ACF_DEBUG_BOUNDS=1).

Every shared-memory histogram index, tile vector, i-vector and partial-row index is checked in
that build; a violation makes the call fail with the recorded values. Exits 0 only if every case
runs clean and matches the oracle under the edge rule. Used by tests/test_gpu_bounds.py.
"""
import os
import sys

os.environ["ACF_DEBUG_BOUNDS"] = "1"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import all_pairs_angular_gb300 as acf  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from oracle import check  # noqa: E402


def main() -> int:
    assert "bounds-checked" in acf.acf_version(), acf.acf_version()
    ctx = acf.Context(0)
    cases = [
        (2000, 2000, 0.25, 720, 0, 0, 0), (1, 1, 0.25, 720, 0, 0, 0), (2049, 130, 0.25, 720, 0, 0, 0),
        (3000, 2500, 0.01, 18000, 0, 0, 0), (3000, 2500, 0.35, 515, 0, 0, 0), (3000, 2500, 0.25, 100, 0, 0, 0),
        (3000, 2500, 0.25, 720, 2, 0, 0), (3000, 2500, 0.25, 720, 0, 512, 0), (3000, 2500, 0.25, 720, 0, 1024, 0), (3000, 2500, 0.25, 720, 0, 0, 1),
        (3000, 2500, 60.0, 3, 0, 0, 0),
    ]
    bad = 0
    cases += [(3000, 2500, 0.25, 720, 0, 0, 10), (3000, 2500, 0.01, 18000, 0, 0, 10), (3000, 2500, 0.35, 515, 0, 0, 10),
              (3000, 2500, 0.25, 720, 0, 0, 20)]
    # every case with the automatic unit choice (small catalogs: one j-group per unit), then the
    # chunk-pair units forced
    cases = [cs + (g,) for g in (0, 4) for cs in cases]
    for n1, n2, w, nb, layout, threads, method, groups in cases:
        # method 10 / 20: chord method with exact mode 2 / 0
        exact = {10: 2, 20: 0}.get(method, 1)
        method = 0 if method >= 10 else method
        ctx.set_option("exact", exact)
        ctx.set_option("layout", layout)
        ctx.set_option("threads", threads)
        ctx.set_option("bin_method", method)
        ctx.set_option("unit_groups", groups)
        c = synth.catalogs(n1, n2, 5 if n1 > 10 else 0, 30.0, seed=n1 * 7 + n2)
        for args in ((c.ra_d, c.dec_d, None, None), (c.ra_d, c.dec_d, c.ra_r, c.dec_r)):
            try:
                g = ctx.histogram(*args, bin_width_deg=w, nbins=nb)
                torch.cuda.synchronize()
            except acf.AcfError as e:
                print("VIOLATION", (n1, n2, w, nb, layout, threads, method, groups), e, flush=True)
                bad += 1
                continue
            gh = acf.as_uint64(g)
            o = oracle.histogram(*args, bin_width_deg=w, nbins=nb)
            rep = check.edge_flux(gh, o.hist, o.near_below, o.near_above)
            ok = rep.ok if method == 0 else int(gh.sum()) == int(o.hist.sum())
            if exact == 2:
                ok = ok and np.array_equal(gh, o.hist)
            print("case", (n1, n2, w, nb, layout, threads, method, exact, ctx.info("unit_groups")),
                  "ok" if ok else "MISMATCH " + str(rep),
                  flush=True)
            bad += 0 if ok else 1
    ctx.close()
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main())
