"""The per-SM rates the kernels are laid out around (tcgen05 SS / TS contraction steps at
N = 64, 128, 256, the latency of one 8-step group and of an mbarrier arrive, and the
elementwise instructions' issue rates), measured by tests/native/tcgen05_rates.cu on the GPU.

Only sanity is asserted (every CTA finished, no rate above the tensor core's 8192 FLOP per
clock per SM); the numbers themselves are printed (``pytest -s``) and summarised with their
command in the profiles."""
import json
import os
import shutil
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_tcgen05_rates(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = tmp_path / "tcgen05_rates"
    src = os.path.join(ROOT, "tests", "native", "tcgen05_rates.cu")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                    src, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout)
    print(json.dumps(res, indent=1))
    assert res["ok"]
    for kind in ("ss", "ts"):
        for n in (64, 128, 256):
            assert 0 < res[f"{kind}_N{n}_flop_per_clk"] <= 8192 * 1.02, (kind, n)
    assert res["ss_N128_group8_latency_cycles"] > 8 * 64 * 0.98
    assert res["mbarrier_arrive_to_waiter_cycles"] > 0
