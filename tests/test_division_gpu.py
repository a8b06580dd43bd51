"""The demotion's division (common.cuh div_by_scale: reciprocal, multiply and one
Markstein correction) equals CUDA's IEEE division __fdiv_rn bit for bit over the whole
domain the kernel uses: every finite fp16 x with |x| <= a and s = fp32_rn(a / 448) for
every positive finite fp16 a. The check is compiled from the product header."""

import os
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_div_by_scale_is_ieee_division_on_the_demotion_domain():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "div_check")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I", os.path.join(HERE, "..", "include"),
                        os.path.join(HERE, "cuda", "div_check.cu"), "-o", exe], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert "mismatches 0 " in r.stdout, r.stdout + r.stderr
    assert r.returncode == 0
