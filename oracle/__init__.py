"""ORACLE — test infrastructure, not part of the library.

A plain fp64 CPU statement of the galaxy two-point angular correlation ("CUDA Deep Dive: 10B
Galaxy Pairs on an RTX 5080", section "The problem" and the bin-index helper and omega writer of
its Appendix A). The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over rows only); this
module is the ctypes wrapper plus the build step. Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it; the CUDA library never does.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed forms, an
independent fp64 formula, invariants and uniform-sphere statistics (see the header of that file).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

EDGE_TOL_RAD = 1e-6  # pairs within this of a bin edge may move to the neighbouring bin

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` (fp64, no FMA contraction, OpenMP) into ``_build/liboracle.so``."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        lib.oracle_histogram.restype = ctypes.c_int
        lib.oracle_histogram.argtypes = [vp, vp, i64, vp, vp, i64, f64, i32, i32, vp, vp, vp]
        lib.oracle_pair_theta.restype = ctypes.c_int
        lib.oracle_pair_theta.argtypes = [vp, vp, vp, vp, i64, vp]
        lib.oracle_pair_bin.restype = ctypes.c_int
        lib.oracle_pair_bin.argtypes = [vp, vp, vp, vp, i64, f64, i32, vp]
        lib.oracle_omega.restype = ctypes.c_int
        lib.oracle_omega.argtypes = [vp, vp, vp, i32, i64, i64, vp]
        _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


class Histogram:
    """Oracle output for one histogram family: counts and the per-edge near-edge pair counts."""

    def __init__(self, hist, near_below, near_above):
        self.hist = hist              # uint64[nbins]
        self.near_below = near_below  # uint64[nbins+1]: pairs with theta in [e_K - tol, e_K)
        self.near_above = near_above  # uint64[nbins+1]: pairs with theta in [e_K, e_K + tol)


def histogram(ra1, dec1, ra2=None, dec2=None, bin_width_deg: float = 0.25, nbins: int = 720,
              threads: int = 0) -> Histogram:
    """Histogram of theta over ALL ordered pairs (i in catalog 1, j in catalog 2).

    With ``ra2 is None`` the catalog is paired with itself (all n^2 ordered pairs, self-pairs
    included): DD or RR.
    """
    ra1, dec1 = _f32(ra1), _f32(dec1)
    if ra2 is None:
        ra2, dec2 = ra1, dec1
    ra2, dec2 = _f32(ra2), _f32(dec2)
    h = np.zeros(nbins, np.uint64)
    lo = np.zeros(nbins + 1, np.uint64)
    hi = np.zeros(nbins + 1, np.uint64)
    rc = _load().oracle_histogram(ra1.ctypes.data, dec1.ctypes.data, ra1.shape[0], ra2.ctypes.data,
                                  dec2.ctypes.data, ra2.shape[0], float(bin_width_deg), int(nbins), int(threads),
                                  h.ctypes.data, lo.ctypes.data, hi.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_histogram rejected its arguments (rc=%d)" % rc)
    return Histogram(h, lo, hi)


def pair_theta(ra1, dec1, ra2, dec2) -> np.ndarray:
    """fp64 separation in radians of each pair (ra1[k], dec1[k]) - (ra2[k], dec2[k])."""
    ra1, dec1, ra2, dec2 = map(_f32, (ra1, dec1, ra2, dec2))
    out = np.empty(ra1.shape[0], np.float64)
    rc = _load().oracle_pair_theta(ra1.ctypes.data, dec1.ctypes.data, ra2.ctypes.data, dec2.ctypes.data,
                                   ra1.shape[0], out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_pair_theta failed")
    return out


def pair_bin(ra1, dec1, ra2, dec2, bin_width_deg: float, nbins: int) -> np.ndarray:
    """Bin of each pair under the oracle's rule."""
    ra1, dec1, ra2, dec2 = map(_f32, (ra1, dec1, ra2, dec2))
    out = np.empty(ra1.shape[0], np.int32)
    rc = _load().oracle_pair_bin(ra1.ctypes.data, dec1.ctypes.data, ra2.ctypes.data, dec2.ctypes.data,
                                 ra1.shape[0], float(bin_width_deg), int(nbins), out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_pair_bin failed")
    return out


def omega(dd, dr, rr, n_d: int, n_r: int) -> np.ndarray:
    """Landy-Szalay omega per bin in fp64 (NaN where RR = 0)."""
    dd, dr, rr = (np.ascontiguousarray(x, dtype=np.uint64) for x in (dd, dr, rr))
    out = np.empty(dd.shape[0], np.float64)
    rc = _load().oracle_omega(dd.ctypes.data, dr.ctypes.data, rr.ctypes.data, dd.shape[0], int(n_d), int(n_r),
                              out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_omega rejected its arguments")
    return out
