"""The fused SwiGLU's fast division against IEEE division on the GPU, exhaustively per exponent pair.

The SwiGLU kernel divides g by d = 1 + exp(-g) with a Newton-Raphson reciprocal and Markstein's
final correction wherever that is exact (nvq_device.cuh, div_markstein), and with IEEE division
elsewhere. This test compiles a small CUDA program against the same header and compares the two for
every pair of bf16 significands (g, both signs) and float32 significands (d) -- 2^31 pairs per
exponent pair -- at exponent pairs across the covered range and at its edge (quotients near 2^-100).
"""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
PAIRS = ["0:0", "0:1", "5:3", "127:0", "126:125", "-99:0", "-100:0", "-80:19", "-79:21", "0:99", "0:100",
         "20:119", "-120:0"]


def test_fast_division_matches_ieee(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "division_check")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-ftz=false",
                    "-prec-div=true", "-prec-sqrt=true", "-o", exe, os.path.join(HERE, "cuda", "division_check.cu")],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([exe, *PAIRS], check=True, capture_output=True, text=True, timeout=600).stdout
    rows = [list(map(int, line.split())) for line in out.strip().splitlines()]
    assert len(rows) == len(PAIRS)
    covered = 0
    for eg, ed, bad, cov, total in rows:
        assert bad == 0, f"exponents {eg}, {ed}: {bad} covered pairs differ from IEEE division"
        covered += cov
        if (eg, ed) in ((0, 0), (127, 0), (-99, 0), (0, 99)):
            assert cov == total                      # every pair of the range's interior is covered
        if (eg, ed) == (-120, 0):
            assert cov == 0                          # quotients near 2^-120 take IEEE division
    assert covered > 10 * 2 ** 31                    # 2.2e10 pairs compared
