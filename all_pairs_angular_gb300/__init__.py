"""Python binding of libacf.so, the GB300 galaxy angular-correlation library.

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
PyTorch supplies device memory and streams. The functions keep the C names of include/acf.h;
``Context`` wraps them for convenience. There is no CPU fallback: if the library cannot be
built or loaded, importing the functions raises.

Histograms are returned as torch.int64 tensors holding the uint64 counts bit for bit (counts stay
far below 2^63); ``as_uint64`` views a host copy as numpy uint64.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

ACF_OK = 0
ACF_ERR_ARG = -1
ACF_ERR_UNSUPPORTED = -2
ACF_ERR_NOMEM = -3
ACF_ERR_CUDA = -4

EXPORTED = ["acf_version", "acf_create", "acf_destroy", "acf_last_error", "acf_set_stream", "acf_histogram",
            "acf_omega", "acf_correlate", "acf_correlate_host", "acf_pair_bins", "acf_set_option", "acf_get_info",
            "acf_kernel_times", "acf_histogram_noalloc", "acf_fp32_peak", "acf_read_catalog", "acf_free_catalog",
            "acf_write_omega", "acf_ladder", "acf_plan_info"]
PLAN_INFO_FIELDS = ("bin_map", "entries", "layout", "threads", "smem_bytes", "fine_shift", "fine_shift_small",
                    "fine_shift_mid", "dot_form", "short_chord", "kmax", "exact")

_lib = None


class AcfError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"acf error {code}: {msg}")
        self.code = code


def library_path() -> str:
    return _build.DEBUG_LIB_PATH if os.environ.get("ACF_DEBUG_BOUNDS", "") == "1" else _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libacf.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    debug = os.environ.get("ACF_DEBUG_BOUNDS", "") == "1"
    if os.environ.get("ACF_LIB"):
        path = os.environ["ACF_LIB"]  # a prebuilt variant (tuning experiments)
    elif build_if_missing:
        path = _build.build(debug=debug)
    else:
        path = _build.DEBUG_LIB_PATH if debug else _build.LIB_PATH
    lib = ctypes.CDLL(path)
    vp, i64, i32, f64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_int
    sig = {
        "acf_version": (ctypes.c_char_p, []),
        "acf_create": (ci, [ctypes.POINTER(vp), ci, vp]),
        "acf_destroy": (None, [vp]),
        "acf_last_error": (ctypes.c_char_p, [vp]),
        "acf_set_stream": (ci, [vp, vp]),
        "acf_histogram": (ci, [vp, vp, vp, i64, vp, vp, i64, f64, i32, vp]),
        "acf_histogram_noalloc": (ci, [vp, vp, vp, i64, vp, vp, i64, f64, i32, vp]),
        "acf_omega": (ci, [vp, vp, vp, vp, i32, i64, i64, vp]),
        "acf_correlate": (ci, [vp, vp, vp, i64, vp, vp, i64, f64, i32, vp, vp, vp, vp]),
        "acf_correlate_host": (ci, [vp, vp, vp, i64, vp, vp, i64, f64, i32, vp, vp, vp, vp]),
        "acf_pair_bins": (ci, [vp, vp, vp, vp, vp, i64, f64, i32, vp]),
        "acf_set_option": (ci, [vp, ctypes.c_char_p, i64]),
        "acf_get_info": (ci, [vp, ctypes.c_char_p, ctypes.POINTER(i64)]),
        "acf_kernel_times": (ci, [vp, ctypes.POINTER(ctypes.c_float), i32, ctypes.POINTER(i32)]),
        "acf_fp32_peak": (ci, [vp, i64, ctypes.POINTER(f64), ctypes.POINTER(ctypes.c_float)]),
        "acf_plan_info": (ci, [f64, i32, i32, ctypes.POINTER(i64)]),
        "acf_read_catalog": (ci, [ctypes.c_char_p, ctypes.POINTER(ctypes.POINTER(ctypes.c_float)),
                                  ctypes.POINTER(ctypes.POINTER(ctypes.c_float)), ctypes.POINTER(i64),
                                  ctypes.c_char_p, i32]),
        "acf_free_catalog": (None, [vp, vp]),
        "acf_write_omega": (ci, [ctypes.c_char_p, vp, vp, vp, vp, i32, f64]),
        "acf_ladder": (ci, [ci, vp, vp, vp, vp, i64, f64, i32, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_float)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _check(ctx, rc: int):
    if rc != ACF_OK:
        msg = load().acf_last_error(ctx).decode() if ctx else ""
        raise AcfError(rc, msg)


# ------------------------------------------------------------- C names, thin wrappers

def acf_version() -> str:
    return load().acf_version().decode()


def acf_create(device: int = 0, stream=None) -> int:
    """Create a context on ``device`` using ``stream`` (a torch.cuda.Stream, a raw handle or None)."""
    h = ctypes.c_void_p()
    raw = getattr(stream, "cuda_stream", stream)
    rc = load().acf_create(ctypes.byref(h), int(device), raw)
    if rc != ACF_OK:
        raise AcfError(rc, "acf_create failed on device %d" % device)
    return h.value


def acf_destroy(ctx: int) -> None:
    load().acf_destroy(ctx)


def acf_last_error(ctx: int) -> str:
    return load().acf_last_error(ctx).decode()


def acf_set_stream(ctx: int, stream) -> None:
    _check(ctx, load().acf_set_stream(ctx, getattr(stream, "cuda_stream", stream)))


def acf_histogram(ctx: int, ra, dec, n: int, ra2, dec2, n2: int, bin_width_deg: float, nbins: int, out) -> None:
    _check(ctx, load().acf_histogram(ctx, _ptr(ra), _ptr(dec), int(n), _ptr(ra2), _ptr(dec2), int(n2),
                                     float(bin_width_deg), int(nbins), _ptr(out)))


def acf_histogram_noalloc(ctx: int, ra, dec, n: int, ra2, dec2, n2: int, bin_width_deg: float, nbins: int,
                          out) -> None:
    """acf_histogram with its scratch in the library's static 16 MiB device array (no allocation)."""
    _check(ctx, load().acf_histogram_noalloc(ctx, _ptr(ra), _ptr(dec), int(n), _ptr(ra2), _ptr(dec2), int(n2),
                                             float(bin_width_deg), int(nbins), _ptr(out)))


def acf_omega(ctx: int, dd, dr, rr, nbins: int, n_d: int, n_r: int, omega) -> None:
    _check(ctx, load().acf_omega(ctx, _ptr(dd), _ptr(dr), _ptr(rr), int(nbins), int(n_d), int(n_r), _ptr(omega)))


def acf_correlate(ctx: int, ra_d, dec_d, n_d: int, ra_r, dec_r, n_r: int, bin_width_deg: float, nbins: int,
                  dd, dr, rr, omega) -> None:
    """DD, DR, RR and omega from device catalogs into device outputs (asynchronous)."""
    _check(ctx, load().acf_correlate(ctx, _ptr(ra_d), _ptr(dec_d), int(n_d), _ptr(ra_r), _ptr(dec_r), int(n_r),
                                     float(bin_width_deg), int(nbins), _ptr(dd), _ptr(dr), _ptr(rr), _ptr(omega)))


def acf_correlate_host(ctx: int, ra_d, dec_d, n_d: int, ra_r, dec_r, n_r: int, bin_width_deg: float, nbins: int,
                       dd, dr, rr, omega) -> None:
    _check(ctx, load().acf_correlate_host(ctx, _ptr(ra_d), _ptr(dec_d), int(n_d), _ptr(ra_r), _ptr(dec_r),
                                          int(n_r), float(bin_width_deg), int(nbins), _ptr(dd), _ptr(dr),
                                          _ptr(rr), _ptr(omega)))


def acf_pair_bins(ctx: int, ra1, dec1, ra2, dec2, n: int, bin_width_deg: float, nbins: int, bins) -> None:
    _check(ctx, load().acf_pair_bins(ctx, _ptr(ra1), _ptr(dec1), _ptr(ra2), _ptr(dec2), int(n),
                                     float(bin_width_deg), int(nbins), _ptr(bins)))


def acf_set_option(ctx: int, key: str, value: int) -> None:
    _check(ctx, load().acf_set_option(ctx, key.encode(), int(value)))


def acf_get_info(ctx: int, key: str) -> int:
    v = ctypes.c_int64()
    _check(ctx, load().acf_get_info(ctx, key.encode(), ctypes.byref(v)))
    return int(v.value)


def acf_kernel_times(ctx: int, cap: int = 4096) -> list[float]:
    buf = (ctypes.c_float * cap)()
    cnt = ctypes.c_int32()
    _check(ctx, load().acf_kernel_times(ctx, buf, int(cap), ctypes.byref(cnt)))
    return [buf[k] for k in range(cnt.value)]


def acf_fp32_peak(ctx: int, iters: int = 1 << 16) -> tuple[float, float]:
    """FMA thread-instructions per second of this GPU (the FP32 issue ceiling), and thread 0's
    chain sum for a host replay."""
    rate = ctypes.c_double()
    t0 = ctypes.c_float()
    _check(ctx, load().acf_fp32_peak(ctx, int(iters), ctypes.byref(rate), ctypes.byref(t0)))
    return rate.value, t0.value


def acf_plan_info(bin_width_deg: float, nbins: int, exact: int = 2) -> dict:
    """The plan acf_histogram would make for this binning (host only, no device): a dict keyed by
    PLAN_INFO_FIELDS. Raises AcfError with the library's status for unsupported binnings."""
    info = (ctypes.c_int64 * len(PLAN_INFO_FIELDS))()
    rc = load().acf_plan_info(float(bin_width_deg), int(nbins), int(exact), info)
    if rc != ACF_OK:
        raise AcfError(rc, "acf_plan_info(%r, %r, %r)" % (bin_width_deg, nbins, exact))
    return dict(zip(PLAN_INFO_FIELDS, (int(v) for v in info)))


def acf_read_catalog(path: str) -> tuple[np.ndarray, np.ndarray]:
    """Read a catalog file (count line, then "ra dec" rows in arcminutes): float32 (ra, dec)."""
    lib = load()
    ra = ctypes.POINTER(ctypes.c_float)()
    dec = ctypes.POINTER(ctypes.c_float)()
    n = ctypes.c_int64()
    err = ctypes.create_string_buffer(512)
    rc = lib.acf_read_catalog(os.fsencode(path), ctypes.byref(ra), ctypes.byref(dec), ctypes.byref(n), err, 512)
    if rc != ACF_OK:
        raise AcfError(rc, err.value.decode())
    try:
        out = (np.ctypeslib.as_array(ra, shape=(n.value,)).copy() if n.value else np.empty(0, np.float32),
               np.ctypeslib.as_array(dec, shape=(n.value,)).copy() if n.value else np.empty(0, np.float32))
    finally:
        lib.acf_free_catalog(ctypes.cast(ra, ctypes.c_void_p), ctypes.cast(dec, ctypes.c_void_p))
    return out


def acf_write_omega(path: str, dd, dr, rr, omega, bin_width_deg: float) -> None:
    """Write the result table (one row per bin with RR > 0) from host arrays."""
    dd, dr, rr = (np.ascontiguousarray(a, dtype=np.uint64) for a in (dd, dr, rr))
    omega = np.ascontiguousarray(omega, dtype=np.float64)
    rc = load().acf_write_omega(os.fsencode(path), dd.ctypes.data, dr.ctypes.data, rr.ctypes.data, omega.ctypes.data,
                                len(dd), float(bin_width_deg))
    if rc != ACF_OK:
        raise AcfError(rc, "cannot write " + str(path))


def acf_ladder(level: int, ra_d, dec_d, ra_r, dec_r, bin_width_deg: float, nbins: int, dd, dr, rr,
               stream=None) -> float:
    """One level of the page's optimisation ladder on device catalogs; returns the kernel's ms."""
    ms = ctypes.c_float()
    rc = load().acf_ladder(int(level), _ptr(ra_d), _ptr(dec_d), _ptr(ra_r), _ptr(dec_r), ra_d.numel(),
                           float(bin_width_deg), int(nbins), _ptr(dd), _ptr(dr), _ptr(rr),
                           getattr(stream, "cuda_stream", stream), ctypes.byref(ms))
    if rc != ACF_OK:
        raise AcfError(rc, "acf_ladder level %d failed" % level)
    return ms.value


def cli_path() -> str:
    """The acf_cli program (catalog files in, omega table out), built next to the library."""
    return _build.build_cli()


# ------------------------------------------------------------- convenience layer

def as_uint64(t) -> np.ndarray:
    """Host numpy uint64 view of a histogram tensor (int64 storage)."""
    a = t.detach().cpu().numpy() if hasattr(t, "detach") else np.asarray(t)
    return a.view(np.uint64)


class Context:
    """A library context bound to one device and one torch stream."""

    def __init__(self, device: int = 0, stream=None):
        import torch
        self.torch = torch
        self.device = torch.device("cuda", device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.handle = acf_create(device, self.stream)

    def close(self):
        if getattr(self, "handle", None):
            acf_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _f32(self, a):
        t = self.torch
        if isinstance(a, np.ndarray):
            a = t.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        return a.to(device=self.device, dtype=t.float32).contiguous()

    def histogram(self, ra, dec, ra2=None, dec2=None, bin_width_deg: float = 0.25, nbins: int = 720, out=None):
        """DD/RR (``ra2 is None``) or DR histogram as an int64 device tensor holding uint64 counts."""
        ra, dec = self._f32(ra), self._f32(dec)
        n2 = 0
        if ra2 is not None:
            ra2, dec2 = self._f32(ra2), self._f32(dec2)
            n2 = ra2.numel()
            if n2 == 0:
                # an empty tensor has a NULL data pointer, which the C ABI reads as "auto-correlation";
                # hand it a one-element placeholder with n2 = 0 instead
                ra2 = dec2 = self.torch.zeros(1, dtype=self.torch.float32, device=self.device)
        if out is None:
            out = self.torch.empty(nbins, dtype=self.torch.int64, device=self.device)
        acf_histogram(self.handle, ra, dec, ra.numel(), ra2, dec2, n2, bin_width_deg, nbins, out)
        return out

    def omega(self, dd, dr, rr, n_d: int, n_r: int, out=None):
        if out is None:
            out = self.torch.empty(dd.numel(), dtype=self.torch.float64, device=self.device)
        acf_omega(self.handle, dd, dr, rr, dd.numel(), n_d, n_r, out)
        return out

    def correlate(self, ra_d, dec_d, ra_r, dec_r, bin_width_deg: float = 0.25, nbins: int = 720, out=None):
        """Whole job on the device; returns device tensors (dd, dr, rr as int64 holding uint64, omega)."""
        ra_d, dec_d, ra_r, dec_r = (self._f32(a) for a in (ra_d, dec_d, ra_r, dec_r))
        if out is None:
            t = self.torch
            out = tuple(t.empty(nbins, dtype=t.int64, device=self.device) for _ in range(3)) + (
                t.empty(nbins, dtype=t.float64, device=self.device),)
        dd, dr, rr, om = out
        acf_correlate(self.handle, ra_d, dec_d, ra_d.numel(), ra_r, dec_r, ra_r.numel(), bin_width_deg, nbins,
                      dd, dr, rr, om)
        return dd, dr, rr, om

    def correlate_host(self, ra_d, dec_d, ra_r, dec_r, bin_width_deg: float = 0.25, nbins: int = 720, out=None):
        """Whole job from host arrays; returns host (dd, dr, rr, omega)."""
        if out is None:
            out = (np.empty(nbins, np.uint64), np.empty(nbins, np.uint64), np.empty(nbins, np.uint64),
                   np.empty(nbins, np.float64))
        dd, dr, rr, om = out
        acf_correlate_host(self.handle, ra_d, dec_d, len(ra_d), ra_r, dec_r, len(ra_r), bin_width_deg, nbins,
                           dd, dr, rr, om)
        return dd, dr, rr, om

    def pair_bins(self, ra1, dec1, ra2, dec2, bin_width_deg: float, nbins: int):
        ra1, dec1, ra2, dec2 = (self._f32(a) for a in (ra1, dec1, ra2, dec2))
        bins = self.torch.empty(ra1.numel(), dtype=self.torch.int32, device=self.device)
        acf_pair_bins(self.handle, ra1, dec1, ra2, dec2, ra1.numel(), bin_width_deg, nbins, bins)
        return bins

    def set_option(self, key: str, value: int):
        acf_set_option(self.handle, key, value)

    def info(self, key: str) -> int:
        return acf_get_info(self.handle, key)

    def kernel_times(self) -> list[float]:
        return acf_kernel_times(self.handle)
