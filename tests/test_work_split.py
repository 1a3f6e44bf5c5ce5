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


def test_sliced_kernel_work_split(tmp_path):
    """The sliced decode kernel's op walker, group barrier counts, two-segment
    shares and contributor rule (tests/sliced_check.cu, host-only, the same
    header as the kernel) for inter 160 / 640, grids of 80..256 CTAs and every
    active-expert count up to min(128, grid)."""
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "sliced_check")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-o", exe, os.path.join(HERE, "sliced_check.cu")],
                   check=True, capture_output=True, cwd=str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    n = 2 * sum(min(128, G) + 1 for G in range(80, 257))
    assert r.stdout.split() == ["ok", str(n)]
