"""The scan's shared-memory stage layout, checked on the host (no GPU): the
layout helpers of scan_core.cuh compiled by nvcc as host code
(tests/native/stage_layout_check.cu) must place every staged part inside its
row and the stage, without collisions, keep each 32-byte sector in one aligned
slot in the host-cache layout, and spread block-column reads over eight bank
groups."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "bit_plane_kv_encode_gb300", "csrc")


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_stage_layout():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "stage_layout_check")
        subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC,
                        os.path.join(HERE, "native", "stage_layout_check.cu"), "-o", exe],
                       check=True, capture_output=True, text=True)
        r = subprocess.run([exe], capture_output=True, text=True)
        assert r.returncode == 0, r.stdout + r.stderr
        assert "stage layout ok" in r.stdout
