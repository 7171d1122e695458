"""The q8_1 quantizers compute amax / 127 with Markstein's correction for a known divisor (a
product and two fused multiply-adds, all rounded to nearest even) instead of an IEEE division.
Its exactness is a property of the method that the host checks here, with the same operations
in C, for every non-negative finite binary32 value; the GPU tests then check the kernels' scales
bit for bit against the oracle's IEEE division."""
import os
import shutil
import subprocess

import pytest


def test_div127_matches_ieee_division_for_every_value(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "div127_check.c")
    exe = str(tmp_path / "div127_check")
    flags = ["-O2", "-ffp-contract=off", "-fno-fast-math"]
    r = subprocess.run([gcc, *flags, "-fopenmp", src, "-o", exe, "-lm"], capture_output=True, text=True)
    if r.returncode != 0:   # no OpenMP runtime: the same check on one thread
        subprocess.run([gcc, *flags, src, "-o", exe, "-lm"], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=600).stdout
    assert out.strip() == "mismatches 0", out
