"""The kernel's polynomial constants are the outputs of their fit scripts, and the fits stay within
the precision budget the exact mode's windows are built on.

Each fit minimises the largest absolute theta error with R or f evaluated in 40-digit arithmetic:
- fit_arcsin2.py fits theta'^2 = q f(q) for the chord forms, degree 7 up to 90 degrees and degree
  5 up to 72.4 degrees;
- fit_asin_mid.py fits asin(d) = d R(d^2) for the dot form, degree 4, up to 54.5 degrees (the
  form is used only above 55).
The budget terms are each fit's error after its coefficients are rounded to fp32: 2.53e-8 rad
(chord), 5.5e-8 (short chord) and 1.6e-7 (dot form).
"""
import os
import re
import subprocess
import sys

import pytest

pytest.importorskip("mpmath")

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "all_pairs_angular_gb300", "csrc")


def _fit(script, *args):
    out = subprocess.run([sys.executable, os.path.join(CSRC, script), *map(str, args)], capture_output=True,
                         text=True, timeout=600, check=True).stdout
    coeffs = [float(v) for v in re.findall(r"^\s+[cr]\d+ = (\S+)$", out, re.M)]
    err32 = float(re.search(r"after fp32 rounding of the coefficients: (\S+)", out).group(1))
    return coeffs, err32


def _kernel_constants():
    with open(os.path.join(CSRC, "acf_kernels.cuh")) as f:
        src = f.read()
    kp = [float(re.search(r"\bkP%d = ([-0-9.e]+)f" % k, src).group(1)) for k in range(8)]
    ks = [float(re.search(r"\bkS%d = ([-0-9.e]+)f" % k, src).group(1)) for k in range(6)]
    body = re.search(r"constexpr double kR\[kRTerms\] = \{([^}]*)\}", src).group(1)
    kr = [float(v) for v in body.replace("\n", " ").split(",")]
    return kp, ks, kr


@pytest.mark.parametrize("form,script,args,budget", [
    ("chord", "fit_arcsin2.py", (7, 90), 2.53e-8),
    ("short", "fit_arcsin2.py", (5, 72.4), 5.5e-8),
    ("dot", "fit_asin_mid.py", (4, 54.5), 1.6e-7),
])
def test_kernel_polynomials_are_their_fits(form, script, args, budget):
    coeffs, err32 = _fit(script, *args)
    kp, ks, kr = _kernel_constants()
    kernel = {"chord": kp, "short": ks, "dot": kr}[form]
    assert len(kernel) == len(coeffs)
    for a, b in zip(kernel, coeffs):
        assert a == pytest.approx(b, rel=1e-15, abs=1e-18)
    assert err32 <= budget
