"""The fused RMSNorm quantizer divides x by rms with one Markstein correction of x * RN(1 / rms)
("Activation Quantization Architecture", Fusion: y = x / rms * gamma, IEEE division in the
oracle). tests/markstein_check.cu compares that quotient with CUDA's IEEE division bit for bit
over every x significand against a stride of divisor significands (2^23 x 2048 pairs here);
with Q8_MARKSTEIN_FULL=1 it runs all 2^46 significand pairs (about 80 s on one GB300)."""
import os
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_markstein_quotient_equals_ieee_division():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    assert os.path.exists(nvcc), "nvcc is needed to build the check"
    stride = "1" if os.environ.get("Q8_MARKSTEIN_FULL") == "1" else "4096"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "markstein_check")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false", "-o", exe,
                        os.path.join(HERE, "markstein_check.cu")], check=True, capture_output=True)
        r = subprocess.run([exe, stride], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert " mismatches 0" in r.stdout
