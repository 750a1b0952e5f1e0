"""The library with programmatic dependent launch switched off
(FP8MP_PDL=0, read once per process): the bench step's parity test, the
row-major backward GEMM's parity tests, and the two-buffer master steps and
the backward's completion signal (whose early starts then become plain
launches after the previous kernel), run in a fresh interpreter."""

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
           "tests/test_gpu_two_buffer_step.py::test_backward_signals_dw_completion",
           "tests/test_gpu_two_buffer_step.py::test_two_buffer_steps_bit_exact",
           "tests/test_gpu_gemm.py", "-k", "bench_step or (rowmajor_copies and 1040) or signals or two_buffer"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
