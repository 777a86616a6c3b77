"""Build libacf.so in-tree for sm_103a with nvcc (no cmake), and the acf_cli program on top of it."""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libacf.so")
DEBUG_LIB_PATH = os.path.join(BUILD_DIR, "libacf_debug.so")  # -DACF_DEBUG_BOUNDS
SOURCES = [os.path.join(HERE, "csrc", "acf.cu"), os.path.join(HERE, "csrc", "acf_io.cpp"),
           os.path.join(HERE, "csrc", "ladder.cu")]
CLI_SOURCE = os.path.join(HERE, "csrc", "acf_cli.cpp")
CLI_PATH = os.path.join(BUILD_DIR, "acf_cli")
DEPENDS = SOURCES + [os.path.join(HERE, "csrc", "acf_kernels.cuh"), os.path.join(ROOT, "include", "acf.h")]
# (acf_cli.cpp includes the header by path: build_cli passes -I include)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libacf.so")


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, debug: bool = False,
          out: str | None = None) -> str:
    """Compile (if stale) and return the path of libacf.so (libacf_debug.so with ``debug``: every
    shared-memory and global index checked, violations reported instead of accessed). ``extra``
    adds nvcc flags (e.g. -DACF_K=6) and ``out`` names another output file for such variants."""
    path = out or (DEBUG_LIB_PATH if debug else LIB_PATH)
    newest = max(os.path.getmtime(p) for p in DEPENDS)
    if not force and not extra and os.path.exists(path) and os.path.getmtime(path) >= newest:
        return path
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = path + ".tmp%d" % os.getpid()
    if debug:
        extra = list(extra or []) + ["-DACF_DEBUG_BOUNDS"]
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v" if verbose else "-O3", *(extra or []), "-o", tmp, *SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, path)
    return path


def build_cli(force: bool = False) -> str:
    """Compile acf_cli (host C++, linked against libacf.so in the same folder) and return its path."""
    lib = build()
    if not force and os.path.exists(CLI_PATH) and os.path.getmtime(CLI_PATH) >= max(
            os.path.getmtime(lib), os.path.getmtime(CLI_SOURCE)):
        return CLI_PATH
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        raise RuntimeError("no C++ compiler for acf_cli")
    tmp = CLI_PATH + ".tmp%d" % os.getpid()
    cmd = [cxx, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "include"), CLI_SOURCE, "-o", tmp, "-L", BUILD_DIR,
           "-lacf", "-Wl,-rpath,$ORIGIN"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("acf_cli failed to build:\n" + res.stdout + res.stderr)
    os.replace(tmp, CLI_PATH)
    return CLI_PATH


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
