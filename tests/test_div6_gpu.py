"""The kernels round amax / 6 with a reciprocal product corrected by its fma
remainder instead of a division; this checks that function against CUDA's
correctly rounded division for every non-negative float (2^31 values)."""
import os
import subprocess

import pytest

from rmsnorm_fp4_quant_gb300 import build as fbuild

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_div6_matches_correctly_rounded_division(tmp_path):
    exe = str(tmp_path / "check_div6")
    subprocess.run([fbuild.nvcc_path(), *fbuild.ARCH_FLAGS, "-O3", "-std=c++17",
                    "-I", fbuild.CSRC, "-I", fbuild.INCLUDE,
                    os.path.join(HERE, "cuda", "check_div6.cu"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "mismatches=0 " in out.stdout, out.stdout
