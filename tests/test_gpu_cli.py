"""acf_cli end to end: catalog files in, the result table out (the page's program shape), on the GPU.

The tiny workload is written as text, run through the command-line program, and the table is read
back: its DD, DR and RR equal the oracle's histograms bin for bin (exact mode 2, the default) and
its omega equals the oracle's to the six printed decimals.
"""
import subprocess

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


def _write_catalog(path, ra, dec):
    with open(path, "w") as f:
        f.write(f"{len(ra)}\n")
        for a, d in zip(ra, dec):
            f.write(f"{float(a):.9g} {float(d):.9g}\n")


def test_cli_writes_the_oracle_table(acf, tmp_path):
    c = synth.config(0)
    w, nb = c.bin_width_deg, c.nbins
    _write_catalog(tmp_path / "data.txt", c.ra_d, c.dec_d)
    _write_catalog(tmp_path / "random.txt", c.ra_r, c.dec_r)
    out = tmp_path / "omega.out"
    res = subprocess.run([acf.cli_path(), str(tmp_path / "data.txt"), str(tmp_path / "random.txt"), str(out),
                          str(w), str(nb)], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "histogram sums correct" in res.stdout
    rows = [line.split("\t") for line in out.read_text().splitlines()[1:]]
    dd = oracle.histogram(c.ra_d, c.dec_d, None, None, w, nb).hist
    dr = oracle.histogram(c.ra_d, c.dec_d, c.ra_r, c.dec_r, w, nb).hist
    rr = oracle.histogram(c.ra_r, c.dec_r, None, None, w, nb).hist
    om = oracle.omega(dd, dr, rr, c.n_d, c.n_r)
    want = [k for k in range(nb) if rr[k] > 0]
    assert len(rows) == len(want)
    for k, r in zip(want, rows):
        assert abs(float(r[0]) - k * w) < 1e-9
        assert (int(r[2]), int(r[3]), int(r[4])) == (int(dd[k]), int(dr[k]), int(rr[k]))
        assert float(r[1]) == float(f"{om[k]:.6f}")
