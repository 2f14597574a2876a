"""The quantize kernels divide a block maximum by fl(6 gs) with a reciprocal
formed once per launch and Markstein's fused multiply-add correction, falling
back to the exact division outside the range where that is proven equal.  This
CPU test compiles tests/nvfp4_division_check.c, which applies the same steps in
IEEE fp32 (no contraction) to every pair of bf16 amax and bf16 block maximum and
to random divisors, and checks that no e4m3 block scale could differ from the
one the correctly rounded quotient gives."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_block_scale_division_matches_correct_rounding(tmp_path):
    exe = tmp_path / "nvfp4_division_check"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-o", str(exe),
                           os.path.join(HERE, "nvfp4_division_check.c"), "-lm"])
    out = subprocess.run([str(exe), "400"], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip().endswith(", 0 differ"), out.stdout
