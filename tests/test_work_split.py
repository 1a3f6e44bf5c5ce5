"""Host-side check of the persistent kernel's work split and W2 partial-sum
bookkeeping (tests/split_check.cu, built with nvcc as a host-only program
from the same header the kernel includes). No GPU needed."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_split_and_partial_bookkeeping_agree(tmp_path):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "split_check")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-o", exe, os.path.join(HERE, "split_check.cu")],
                   check=True, capture_output=True, cwd=str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    # 2 K-part counts x 256 active-expert counts x grids of 80..256 CTAs
    assert r.stdout.split() == ["ok", str(2 * 256 * 177)]
