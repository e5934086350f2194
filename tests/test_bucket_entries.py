"""The kernels' search-free code lookup (one table read per value, see
csrc/tables.h) checked against the oracle's thresholds for every binary32
pattern.  Host only: the library's table builder is compiled with the check
program; the lookup is restated on the host (the GPU tests compare the
kernels themselves with the oracle)."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_wise_dynamic_gb300", "csrc")


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_every_pattern_gets_the_oracle_code(tmp_path):
    exe = tmp_path / "bucket_entries"
    subprocess.run(["g++", "-O2", "-std=c++17", "-pthread", "-ffp-contract=off",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    os.path.join(ROOT, "tests", "host", "bucket_entries.cpp"),
                    os.path.join(CSRC, "codebook.cpp"), "-o", str(exe)], check=True)
    thr = tmp_path / "thresholds.bin"
    with open(thr, "wb") as f:
        f.write(oracle.thresholds(True).astype(np.float32).tobytes())
        f.write(oracle.thresholds(False).astype(np.float32).tobytes())
    r = subprocess.run([str(exe), str(thr)], capture_output=True, text=True, timeout=600)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0 out_of_bounds 0" in r.stdout
