"""The persistent forward decodes each work unit with fa::FastDiv, a multiply-high by a
reciprocal made on the host instead of an integer division. A wrong quotient would send a
CTA to the wrong head or Q tile, so the division is checked on the host against plain
unsigned division (tests/native/fastdiv_check.cu, compiled here with nvcc)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_fastdiv_matches_integer_division():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    out_dir = os.path.join(ROOT, "_build", "tests")  # git-ignored build folder
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "fastdiv_check")
    subprocess.run([nvcc, "-std=c++17", "-O2",
                    "-I", os.path.join(ROOT, "exact_attention_23_gb300", "csrc"),
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "native", "fastdiv_check.cu"), "-o", exe],
                   check=True, capture_output=True, timeout=300)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "mismatches 0" in out.stdout
