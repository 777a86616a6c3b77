"""Seeded synthetic galaxy catalogs shaped like the workloads of "CUDA Deep Dive: 10B Galaxy Pairs
on an RTX 5080" (section "The problem": two catalogs of RA/Dec in arcminutes, one clustered "real"
catalog D and one random catalog R).

This module makes inputs only; it contains none of the correlation arithmetic. Both the CUDA
library and the CPU oracle are fed from it. The generator is plain C (``synth.c``) that uses only
correctly rounded IEEE operations, so the same seed gives bit-identical catalogs on x86-64 and
aarch64 hosts.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` (no FMA contraction, no fast-math)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_catalogs.restype = ctypes.c_int
        lib.synth_catalogs.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double,
                                       ctypes.c_double, ctypes.c_uint64] + [ctypes.c_void_p] * 4
        lib.synth_sample_rows.restype = ctypes.c_int
        lib.synth_sample_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                          ctypes.c_void_p, ctypes.c_void_p]
        for name in ("synth_p_log", "synth_p_sin", "synth_p_cos", "synth_p_asin"):
            getattr(lib, name).restype = ctypes.c_double
            getattr(lib, name).argtypes = [ctypes.c_double]
        lib.synth_p_atan2.restype = ctypes.c_double
        lib.synth_p_atan2.argtypes = [ctypes.c_double, ctypes.c_double]
        _lib = lib
    return _lib


@dataclass
class Catalogs:
    """A D/R catalog pair plus the binning its workload uses."""
    name: str
    ra_d: np.ndarray   # float32 arcmin
    dec_d: np.ndarray
    ra_r: np.ndarray
    dec_r: np.ndarray
    bin_width_deg: float
    nbins: int
    seed: int

    @property
    def n_d(self) -> int:
        return int(self.ra_d.shape[0])

    @property
    def n_r(self) -> int:
        return int(self.ra_r.shape[0])

    def digest(self) -> str:
        """SHA-256 of the four float32 arrays, to prove two machines generated the same input."""
        h = hashlib.sha256()
        for a in (self.ra_d, self.dec_d, self.ra_r, self.dec_r):
            h.update(np.ascontiguousarray(a, dtype=np.float32).tobytes())
        return h.hexdigest()


def catalogs(n_d: int, n_r: int, n_clumps: int, sigma_arcmin: float, seed: int,
             patch_arcmin: float = 0.0, bin_width_deg: float = 0.25, nbins: int = 720,
             name: str = "custom") -> Catalogs:
    """D = n_d//2 uniform + the rest in ``n_clumps`` Gaussian clumps; R uniform.

    ``patch_arcmin > 0`` confines everything to RA, Dec in [0, patch) arcmin.
    """
    lib = _load()
    ra_d = np.empty(n_d, np.float32)
    dec_d = np.empty(n_d, np.float32)
    ra_r = np.empty(n_r, np.float32)
    dec_r = np.empty(n_r, np.float32)
    rc = lib.synth_catalogs(n_d, n_r, n_clumps, float(sigma_arcmin), float(patch_arcmin), seed,
                            ra_d.ctypes.data, dec_d.ctypes.data, ra_r.ctypes.data, dec_r.ctypes.data)
    if rc != 0:
        raise RuntimeError("synth_catalogs failed with code %d" % rc)
    return Catalogs(name, ra_d, dec_d, ra_r, dec_r, bin_width_deg, nbins, seed)


def uniform_sphere(n: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """n points uniform on the sphere (RA, Dec in arcmin, float32)."""
    c = catalogs(0, n, 0, 0.0, seed)
    return c.ra_r, c.dec_r


# The five workloads: tiny, the pages' shape (two 100k catalogs), a 5x5 degree field, a 1M scale
# case and a fine-binning case. Seeds 1..5.
CONFIGS = {
    0: dict(name="tiny-2k", n_d=2000, n_r=2000, n_clumps=20, sigma_arcmin=30.0, seed=1,
            patch_arcmin=0.0, bin_width_deg=0.25, nbins=720),
    1: dict(name="pages-shape-100k", n_d=100_000, n_r=100_000, n_clumps=20, sigma_arcmin=30.0, seed=2,
            patch_arcmin=0.0, bin_width_deg=0.25, nbins=720),
    2: dict(name="small-field-100k", n_d=100_000, n_r=100_000, n_clumps=200, sigma_arcmin=3.0, seed=3,
            patch_arcmin=300.0, bin_width_deg=0.25, nbins=720),
    3: dict(name="scale-1m", n_d=1_000_000, n_r=1_000_000, n_clumps=20, sigma_arcmin=30.0, seed=4,
            patch_arcmin=0.0, bin_width_deg=0.25, nbins=720),
    4: dict(name="fine-200k", n_d=200_000, n_r=200_000, n_clumps=20, sigma_arcmin=30.0, seed=5,
            patch_arcmin=0.0, bin_width_deg=0.01, nbins=18000),
}


def config(index: int) -> Catalogs:
    """Generate workload ``index`` (0..4)."""
    c = dict(CONFIGS[index])
    return catalogs(**c)


def sample_rows(n: int, k: int, seed: int) -> np.ndarray:
    """k distinct sorted row indices in [0, n) drawn from ``seed`` (for row-sampled checks)."""
    lib = _load()
    out = np.empty(k, np.int64)
    scratch = np.empty(max(n, 1), np.uint8)
    rc = lib.synth_sample_rows(n, k, seed, out.ctypes.data, scratch.ctypes.data)
    if rc != 0:
        raise RuntimeError("synth_sample_rows failed with code %d" % rc)
    return out


def elementary(name: str, *args: float) -> float:
    """Call one of the generator's portable elementary functions (log, sin, cos, asin, atan2)."""
    return float(getattr(_load(), "synth_p_" + name)(*args))
