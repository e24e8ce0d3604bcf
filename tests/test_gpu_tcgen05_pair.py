"""The CTA-pair tensor-core mechanics (tcgen05 cta_group::2: pair allocation of tensor memory,
one M = 256 MMA over two CTAs' shared memory and tensor memory, SS and TS forms, completion
signalled to both CTAs) checked bit for bit against a CPU product by
tests/native/tcgen05_pair_check.cu on the GPU."""
import json
import os
import shutil
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cta_pair_mma(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = tmp_path / "tcgen05_pair_check"
    src = os.path.join(ROOT, "tests", "native", "tcgen05_pair_check.cu")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                    src, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    res = json.loads(r.stdout)
    print(json.dumps(res))
    assert r.returncode == 0 and res["ok"], res
