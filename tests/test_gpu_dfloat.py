"""The double-float exponential and division of the accept kernels
(long_context_self_gb300/csrc/dfloat.cuh, df_exp_diff and df_div) against the
host's long-double arithmetic: tests/dfloat_check.cu is compiled for sm_103a and run; it
checks ~300 000 float pairs (differences 0-90, dense and random, ten
magnitudes of the larger operand): 1e-11 relative down to exp(-70), an
absolute 2e-38 below (the merged sums it feeds are at least 1); and 200 000
quotients of double-float pairs over magnitudes 2^-40 .. 2^40 to 1e-13."""
import os
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_df_exp_diff_accuracy():
    from long_context_self_gb300 import build
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "dfloat_check")
        cmd = [build.nvcc(), *build.ARCH, "-O3", "-std=c++17", os.path.join(HERE, "dfloat_check.cu"), "-o", exe]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-3000:]
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        print(r.stdout)
        assert r.returncode == 0, r.stdout + r.stderr
