"""The C ABI library: it builds, loads without a GPU and exports every symbol include/acf.h declares."""
import ctypes
import os
import re
import subprocess

import pytest

import all_pairs_angular_gb300 as acf
from all_pairs_angular_gb300 import build as acf_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "acf.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(acf_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("acf_create", "acf_histogram", "acf_omega", "acf_destroy", "acf_last_error"):
        assert required in names


def test_library_loads_and_exports_every_declared_symbol():
    lib = acf.load()
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in acf.EXPORTED, f"binding lacks {name}"
    out = subprocess.run(["nm", "-D", "--defined-only", acf_build.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(acf_[a-z_0-9]+)\b", out))
    assert set(_declared()) <= exported


def test_version_and_null_context_errors():
    assert "sm_103a" in acf.acf_version()
    lib = acf.load()
    assert lib.acf_histogram(None, None, None, 0, None, None, 0, 0.25, 720, None) == acf.ACF_ERR_ARG
    assert lib.acf_omega(None, None, None, None, 1, 1, 1, None) == acf.ACF_ERR_ARG
    assert lib.acf_set_option(None, b"threads", 256) == acf.ACF_ERR_ARG
    assert lib.acf_last_error(None) == b"null context"
    lib.acf_destroy(None)  # no-op
    h = ctypes.c_void_p()
    assert lib.acf_create(None, 0, None) == acf.ACF_ERR_ARG
