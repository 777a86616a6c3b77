"""Catalog files and the result table (host code of libacf.so; no GPU).

The formats are those of the program on "CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080": a
catalog is a count line, then "ra dec" rows in arcminutes; the result table has a header and one
tab-separated row per bin with RR > 0 (bin start in degrees, omega, DD, DR, RR).
"""
import numpy as np
import pytest

import synth


def _write_catalog(path, ra, dec, count=None, sep=" "):
    with open(path, "w") as f:
        f.write(f"{len(ra) if count is None else count}\n")
        for a, d in zip(ra, dec):
            # nine significant digits give every float32 back exactly
            f.write(f"{float(a):.9g}{sep}{float(d):.9g}\n")


def test_read_catalog_roundtrips_float32(acf, tmp_path):
    c = synth.catalogs(3000, 0, 10, 30.0, seed=41)
    p = tmp_path / "data.txt"
    _write_catalog(p, c.ra_d, c.dec_d)
    ra, dec = acf.acf_read_catalog(str(p))
    assert ra.dtype == np.float32 and dec.dtype == np.float32
    assert np.array_equal(ra.view(np.uint32), c.ra_d.view(np.uint32))
    assert np.array_equal(dec.view(np.uint32), c.dec_d.view(np.uint32))


def test_read_catalog_whitespace_and_extremes(acf, tmp_path):
    p = tmp_path / "odd.txt"
    p.write_text("  3\r\n0\t-5400\n21599.9990234375   5400\n\n1e-3 -0.0  \n")
    ra, dec = acf.acf_read_catalog(str(p))
    assert ra.tolist() == [0.0, np.float32(21599.9990234375), np.float32(1e-3)]
    assert dec.tolist() == [-5400.0, 5400.0, 0.0]
    empty = tmp_path / "empty_catalog.txt"
    empty.write_text("0\n")
    ra, dec = acf.acf_read_catalog(str(empty))
    assert len(ra) == 0 and len(dec) == 0


@pytest.mark.parametrize("content,msg", [
    ("5\n1 2\n3 4\n", "line 4"),          # fewer rows than the count
    ("x\n1 2\n", "count"),                # no count
    ("2\n1 2\n3 y\n", "line 3"),          # a bad number
])
def test_read_catalog_errors(acf, tmp_path, content, msg):
    p = tmp_path / "bad.txt"
    p.write_text(content)
    with pytest.raises(acf.AcfError) as e:
        acf.acf_read_catalog(str(p))
    assert e.value.code == acf.ACF_ERR_ARG and msg in str(e.value)
    with pytest.raises(acf.AcfError):
        acf.acf_read_catalog(str(tmp_path / "missing.txt"))


def test_write_omega_format(acf, tmp_path):
    dd = np.array([10, 0, 7, 3], np.uint64)
    dr = np.array([8, 1, 6, 0], np.uint64)
    rr = np.array([9, 0, 5, 2], np.uint64)
    om = np.array([0.25, np.nan, -0.123456789, 2.5])
    p = tmp_path / "omega.out"
    acf.acf_write_omega(str(p), dd, dr, rr, om, 0.25)
    lines = p.read_text().splitlines()
    assert lines[0] == "bin start\t\tomega\t        hist_DD\t        hist_DR\t        hist_RR"
    # bins with RR = 0 are left out, as on the page
    assert lines[1:] == [
        " 0.000\t       0.250000\t             10\t              8\t              9",
        " 0.500\t      -0.123457\t              7\t              6\t              5",
        " 0.750\t       2.500000\t              3\t              0\t              2",
    ]
