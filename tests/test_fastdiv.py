"""Host check of the GEMM's multiply-high division constants (make_fastdiv in
csrc/wgrad_params.h): a small host program built with nvcc against the real
header compares umulhi(x, mul) >> shift with x / d for divisors 1..4096, 2000
random divisors below 2^31 and numerators up to 2^31 - 1 (edges and random)."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "native", "fastdiv_check.cu")
CSRC = os.path.join(ROOT, "grouped_fp8_weight_gb300", "csrc")


def _nvcc():
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


def test_fastdiv_constants_match_exact_division():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "fastdiv_check")
        r = subprocess.run([nvcc, "-std=c++17", "-O2", "-I", CSRC, SRC, "-o", exe],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, r.stdout + r.stderr
        assert r.stdout.startswith("ok "), r.stdout
        assert int(r.stdout.split()[1]) > 1_000_000
