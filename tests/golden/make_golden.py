"""Write the oracle's histograms for the full-size workloads to tests/golden/.

Calls only the fp64 oracle (oracle/) and the seeded generator (synth/); nothing here touches the
CUDA library. Each file records the generator digest of its inputs so a test can prove that it
regenerated the same catalogs before comparing.

Usage: python tests/golden/make_golden.py [config ...]      (default: 1 2 4)

For binnings of more than 2000 bins (the 18,000 x 0.01 degree fine-binning workload) only the
histograms are stored, not the per-edge near-edge counts nor omega, to keep the fixture small: the
tests compare those histograms bin for bin and take omega from them through the oracle.
"""
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def main(configs):
    for idx in configs:
        c = synth.config(idx)
        out = {"config": idx, "name": c.name, "seed": c.seed, "n_d": c.n_d, "n_r": c.n_r,
               "bin_width_deg": c.bin_width_deg, "nbins": c.nbins, "digest": c.digest(),
               "edge_tol_rad": oracle.EDGE_TOL_RAD}
        t0 = time.time()
        for fam, args in (("DD", (c.ra_d, c.dec_d, None, None)), ("DR", (c.ra_d, c.dec_d, c.ra_r, c.dec_r)),
                          ("RR", (c.ra_r, c.dec_r, None, None))):
            h = oracle.histogram(*args, bin_width_deg=c.bin_width_deg, nbins=c.nbins, threads=0)
            out[fam] = {"hist": [int(x) for x in h.hist]}
            if c.nbins <= 2000:
                out[fam]["near_below"] = [int(x) for x in h.near_below]
                out[fam]["near_above"] = [int(x) for x in h.near_above]
            print(f"config {idx} {fam}: {time.time() - t0:.1f} s", flush=True)
        if c.nbins <= 2000:  # (fine binnings: omega follows from the stored histograms)
            om = oracle.omega(out["DD"]["hist"], out["DR"]["hist"], out["RR"]["hist"], c.n_d, c.n_r)
            out["omega"] = [None if x != x else float(x) for x in om]
        out["oracle_seconds"] = round(time.time() - t0, 1)
        out["oracle_threads"] = os.cpu_count()
        path = os.path.join(HERE, f"config{idx}_oracle.json")
        with open(path, "w") as f:
            json.dump(out, f, separators=(",", ":"))
        print("wrote", path, flush=True)


if __name__ == "__main__":
    main([int(a) for a in sys.argv[1:]] or [1, 2, 4])
