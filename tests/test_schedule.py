"""The tcgen05 GEMM's work schedules, checked on the CPU: the schedule header
is compiled into a host-only program (tests/schedule_check.cu) that
enumerates launch shapes and SM counts and checks exact coverage of every
output tile and K block, the split-K piece bookkeeping and the pair items."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "smoothquant_w8a8_int8_gb300", "csrc")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_gemm_schedules_cover_every_tile_once(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "schedule_check")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, "-o", exe,
                    os.path.join(ROOT, "tests", "schedule_check.cu")], check=True, timeout=300)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stdout[-3000:]
    assert "0 failures" in p.stdout
