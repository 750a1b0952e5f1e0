"""The library with programmatic dependent launch switched off
(FP8MP_PDL=0, read once per process): the bench step's parity test and the
row-major backward GEMM's parity tests, run in a fresh interpreter."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_without_programmatic_launch():
    env = dict(os.environ, FP8MP_PDL="0")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           "tests/test_gpu_bench_step.py::test_bench_step_matches_oracle",
           "tests/test_gpu_bench_step.py::test_bench_step_skips_on_a_nan_gradient",
           "tests/test_gpu_gemm.py", "-k", "bench_step or (rowmajor_copies and 1040)"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
