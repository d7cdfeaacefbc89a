"""The bounds-checked build (-DDISCO_DEBUG_BOUNDS) on the small parity cases.

compute-sanitizer is not available on the GPUs this library is tested on, so
this build stands in for it: every kernel range-checks its gather indices
and TMA / bulk-copy coordinates against the tensors' extents, skips an
access that fails and reports it through disco_device_status.  The cases run
in a child process that loads that build (tests/_bounds_child.py); they must
match the oracle with a clean status, and psi handed over with understated
element counts must be flagged."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_build_runs_small_cases_clean():
    from sparse_spherical_convolution_gb300 import build
    build.build(debug_bounds=True)
    env = dict(os.environ, DISCO_GB300_BOUNDS_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_bounds_child.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-4000:])
    assert "bounds-checked:" in r.stdout and "cases clean" in r.stdout, r.stdout[-2000:]
