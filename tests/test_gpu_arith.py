"""Device arithmetic that replaces an IEEE operation must equal it exactly.

div6_rn (the block scale's amax / 6 as a multiply and one fused correction
step) is compared with IEEE division over every non-negative finite float,
by a small CUDA program that includes the library's device header.
"""
import os
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def test_div6_rn_equals_ieee_division_for_every_nonnegative_float():
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "div6_check")
        subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I", os.path.join(ROOT, "fp4_gemm_nvfp4_gb300", "csrc"), "-I", os.path.join(ROOT, "include"),
                        os.path.join(HERE, "cuda", "div6_check.cu"), "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("mismatches 0 "), out.stdout
