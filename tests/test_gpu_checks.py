"""The bounds-checked build (the library compiled with -DBPKV_CHECKS=1): the
scan's plan builder, copies, weight formation and group loop check every
index they compute against its array and record BPKV_DEV_BOUNDS in the status
word instead of touching memory outside it.  The decode-step (caches in
device memory), basis, calibration and scan GPU tests run once more against
that library in a child process; each of them asserts a clean status word
after its steps."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_suite_under_bounds_checks():
    from bit_plane_kv_encode_gb300 import build as B
    B.build(checks=True)
    env = dict(os.environ, BPKV_CHECKS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           "tests/test_gpu_configs.py", "tests/test_gpu_steps.py", "tests/test_gpu_basis.py",
           "tests/test_gpu_calibrate.py", "tests/test_gpu_parity.py::test_scan_scores"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
