"""The per-block division used by the quantizers (exact_div.cuh, scalar and
packed-pair forms, scaled and unscaled: a correctly rounded reciprocal plus
Markstein's correction) against the GPU's IEEE division, bit for bit.  The
full run over all 2^23 divisor significands (about 90 s) is exhaustive; here
the first and last 16,384 divisor significands (the last ones include the
all-ones significand) are checked against every dividend significand of both
signs, plus 1.6e10 random pairs over the exponent range, plus the unscaled
form at both ends of its divisor range with quotients around 2^-64."""

import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def div_check(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("divcheck") / "div_check")
    src = os.path.join(ROOT, "tests", "cuda", "div_check.cu")
    inc = os.path.join(ROOT, "block_wise_dynamic_gb300", "csrc")
    subprocess.run([nvcc, "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", inc,
                    src, "-o", out], check=True)
    return out


@pytest.mark.parametrize("first", [0, (1 << 23) - 16384])
def test_fast_division_is_ieee_division(div_check, first):
    r = subprocess.run([div_check, "16384", str(first)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "part1: divisor significands 16384, checked 274877906944, mismatches 0" in r.stdout
    lines = r.stdout.splitlines()
    assert lines[1].startswith("part2:") and lines[1].endswith("mismatches 0")
    assert lines[2].startswith("part3:") and lines[2].endswith("mismatches 0")
