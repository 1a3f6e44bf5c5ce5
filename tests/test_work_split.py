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


def test_bench_kernel_names_follow_the_auto_rules():
    """bench.py's kernel_of (which launches a layer call makes, for the
    roofline) states the same AUTO rules as the header."""
    import bench
    sms, k = 152, 10
    assert bench.kernel_of(1, k, sms) == "sliced_layer_kernel"
    assert bench.kernel_of(2, k, sms) == "sliced_layer_kernel"
    assert bench.kernel_of(1, k, sms, inter=640) == "fused_layer_kernel"
    for M in (3, 4, 8, 16):
        assert bench.kernel_of(M, k, sms) == "fused_layer_kernel"
    for M in (17, 128, 512):
        assert bench.kernel_of(M, k, sms).startswith("route_kernel + w13_swiglu_kernel + w2_tc_kernel")
    # NVFP4 banks: the fused kernel up to 16 tokens (never the sliced one), the hybrid path above
    assert bench.kernel_of(1, k, sms, nvfp4=True) == "fused_layer_kernel"
    assert bench.kernel_of(2, k, sms, nvfp4=True) == "fused_layer_kernel"
    assert bench.kernel_of(300, k, sms, nvfp4=True).startswith("route_kernel + w13_swiglu_kernel")
    # explicit paths
    assert bench.kernel_of(8, k, sms, path="prefill").startswith("route_kernel + w13_tc_kernel")
    assert bench.kernel_of(8, k, sms, path="staged") == "route_kernel + w13_swiglu_kernel + w2_reduce_kernel"
