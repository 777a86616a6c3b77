"""The bounds-checked build (every shared and global index checked, no trap) runs clean."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounds_checked_build_runs_clean():
    env = dict(os.environ, ACF_DEBUG_BOUNDS="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_cases.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    print(r.stdout[-4000:], r.stderr[-2000:])
    assert r.returncode == 0
