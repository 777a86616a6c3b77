"""The host-side plan (acf_plan_info: no device needed): bin map, histogram layout, shared memory,
and the exact-mode windows.

The window of a form is 2^-S bins on each side of an edge. It must cover the form's worst-case
fp32 error, and S is the largest value that still does, so that as few pairs as possible are
flagged. The worst-case errors are 1.25e-6 rad (full-range chord), 1.05e-6 (short chord, theta'
up to 72 degrees) and 6e-7 (dot form, 55 to 125 degrees). S is also capped by the room the fine
code has: (entries + 2) << S must stay below 2^23.
"""
import math

import pytest

import all_pairs_angular_gb300 as acf

BOUND = {"fine_shift": 1.25e-6, "fine_shift_small": 1.05e-6, "fine_shift_mid": 6e-7}


def test_the_two_workload_binnings():
    p = acf.acf_plan_info(0.25, 720)
    assert (p["bin_map"], p["entries"], p["layout"], p["threads"]) == (0, 722, 1, 1024)
    assert (p["fine_shift"], p["fine_shift_small"], p["fine_shift_mid"]) == (11, 12, 12)
    assert p["dot_form"] == 1 and p["short_chord"] == 1 and p["kmax"] == 719 and p["exact"] == 2
    p = acf.acf_plan_info(0.01, 18000)
    assert (p["bin_map"], p["entries"], p["layout"], p["threads"]) == (0, 18002, 2, 1024)
    assert (p["fine_shift"], p["fine_shift_small"], p["fine_shift_mid"]) == (7, 7, 8)


@pytest.mark.parametrize("p_bins", [36, 180, 360, 720, 1000, 1440, 2176, 2556, 3600, 7200, 18000, 36000])
def test_windows_cover_each_bound_and_are_the_tightest_that_do(p_bins):
    w_deg = 180.0 / p_bins
    w = math.radians(w_deg)
    p = acf.acf_plan_info(w_deg, p_bins)
    room = math.floor(math.log2(8.0e6 / (p["entries"] + 2.0)))
    for key, bound in BOUND.items():
        s = p[key]
        assert math.ldexp(w, -s) >= bound, (key, s)  # the window covers the worst case
        assert s == room or math.ldexp(w, -(s + 1)) < bound, (key, s)  # and no finer one would
        assert (p["entries"] + 2) << s < 1 << 23


def test_modes_zero_and_one():
    p0 = acf.acf_plan_info(0.25, 720, exact=0)
    assert p0["exact"] == 0 and p0["fine_shift"] == p0["fine_shift_small"] == p0["fine_shift_mid"] == 0
    # mode 1 re-decides only near 0 and 180 degrees (20 by default), where the chord's error is
    # smaller than its worst case at 90: one S for every form, at least mode 2's
    p1 = acf.acf_plan_info(0.25, 720, exact=1)
    p2 = acf.acf_plan_info(0.25, 720, exact=2)
    assert p1["fine_shift"] == p1["fine_shift_small"] == p1["fine_shift_mid"] >= p2["fine_shift_mid"]


def test_bin_maps_and_forms():
    # 180/w an integer: the direct map with two spare entries; the dot form needs it even
    assert acf.acf_plan_info(180.0 / 721, 721)["bin_map"] == 0
    assert acf.acf_plan_info(180.0 / 721, 721)["dot_form"] == 0
    assert acf.acf_plan_info(180.0 / 722, 722)["dot_form"] == 1
    # otherwise the clamp map with one entry per bin, chord forms only
    p = acf.acf_plan_info(0.35, 515)
    assert (p["bin_map"], p["entries"], p["dot_form"]) == (1, 515, 0)
    # bins beyond 180 degrees stay empty: the last bin a separation reaches
    assert acf.acf_plan_info(0.25, 1440)["kmax"] == 720


def test_shared_memory_limits():
    p = acf.acf_plan_info(180.0 / 41214, 41214)
    assert (p["entries"], p["layout"], p["threads"], p["smem_bytes"]) == (41216, 2, 512, 230400)
    # lane-private copies while they fit beside 16 warps' tiles, 1024 threads while everything fits
    assert acf.acf_plan_info(0.25, 720)["smem_bytes"] <= 230400
    for w, nb in ((180.0 / 41216, 41216), (180.0 / 41300.5, 41217)):
        with pytest.raises(acf.AcfError) as e:
            acf.acf_plan_info(w, nb)
        assert e.value.code == acf.ACF_ERR_UNSUPPORTED


@pytest.mark.parametrize("w,nb,exact", [(0.0, 720, 2), (-1.0, 720, 2), (float("nan"), 720, 2), (0.25, 0, 2),
                                        (0.25, 720, 3), (0.25, 720, -1)])
def test_bad_arguments(w, nb, exact):
    with pytest.raises(acf.AcfError) as e:
        acf.acf_plan_info(w, nb, exact)
    assert e.value.code == acf.ACF_ERR_ARG
