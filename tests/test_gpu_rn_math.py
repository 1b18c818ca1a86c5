"""The fast correctly rounded reciprocal, division by 6 and square root
(csrc/rn_math.cuh, used by the FP4Quant encode for its two scales) against
the CUDA intrinsics __frcp_rn, __fdiv_rn(x, 6) and __fsqrt_rn, on every fp32
bit pattern: the positive and the negative half, each as one launch of
tests/cuda/rn_math_check.cu, built here with nvcc for sm_103a."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_scaled_fp4_e2m1_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "cuda", "rn_math_check.cu")


def _nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else shutil.which("nvcc")


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path_factory.mktemp("rn_math") / "rn_math_check")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-fmad=false", "-I", CSRC, SRC, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


@pytest.mark.gpu
@pytest.mark.parametrize("lo,hi", [("00000000", "80000000"), ("80000000", "ffffffff")])
def test_every_bit_pattern_matches_the_intrinsics(checker, lo, hi):
    r = subprocess.run([checker, lo, hi], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split() == ["rcp", "0", "div6", "0", "sqrt", "0"], r.stdout
