"""bench.py --kernels (each kernel alone at the workloads' sizes): the
selected workloads' JSON lines and the closing clocks line, in a fresh
interpreter; the scale update is the quick case, the row casts of the
transformer activation check a line with a roofline."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_table(only):
    r = subprocess.run([sys.executable, "bench.py", "--kernels", "--only", only, "--steps", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    return [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]


def test_kernel_table_scale_update_only():
    lines = run_table("4 metas")
    kernels = [d for d in lines if "kernel" in d]
    assert [d["kernel"] for d in kernels] == ["scale_update_kernel"]
    assert kernels[0]["us"] > 0 and kernels[0]["roofline"] is None
    assert "clocks" in lines[-1] and lines[-1]["reps"] == 3


def test_kernel_table_cast_lines_carry_a_roofline():
    lines = run_table("transformer x")
    kernels = [d for d in lines if "kernel" in d]
    assert len(kernels) == 3  # row cast, row + transposed cast, current scaling
    for d in kernels:
        r = d["roofline"]
        assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
        assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3 and 0.1 < r["frac"] < 1.5
        assert d["value"] == r["achieved"] and d["workload"].startswith("transformer x")
