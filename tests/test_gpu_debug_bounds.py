"""The bounds-checked debug build of the library on the GPU.

The debug build (ECC_DEBUG_BOUNDS=1; loaded by the binding when ECC_DEBUG=1) checks the
data-dependent indices of every kernel -- histogram bins from keys, global rows and columns,
staged tiles, soft-list slots, locations and global indices -- before it uses them, records a bit
in the device error word and skips the access when a check fails. Small parity cases across the
hard 2-D and 3-D kernels (both 3-D kernels, u8, search-mode keys, batches), the streamed path
and the soft forward, backward and transform run under it in a process of their own, match the
oracle, and leave the error word clean."""
import os
import subprocess
import sys

import pytest

from euler_characteristic_curves_gb300 import build

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.timeout(900)
def test_small_cases_under_the_debug_build_leave_no_error_bits():
    build.build(debug=True)
    env = dict(os.environ, ECC_DEBUG="1")
    res = subprocess.run([sys.executable, "-m", "tests._debug_run"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=800)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "debug-run ok 0" in res.stdout
