"""The kernels' tile schedule, compiled for the host and checked exhaustively (no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_tile_schedule_is_a_heaviest_first_permutation(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc) and shutil.which("nvcc") is None:
        pytest.skip("nvcc not available")
    exe = tmp_path / "tile_order_check"
    src = os.path.join(ROOT, "tests", "native", "tile_order_check.cu")
    inc = os.path.join(ROOT, "tiled_attention_08_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-I", inc, src, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout
