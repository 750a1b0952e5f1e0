"""The library's first calls from several host threads at once (its
per-device caches are filled on first use): in a fresh interpreter, eight
threads, each on its own CUDA stream, run a forward GEMM, the row-major
backward launch and a master step concurrently; every result equals the
same calls run afterwards on one thread."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading, torch
sys.path.insert(0, ROOT)
import fp8_mixed_precision_reduce_gb300 as f
import workloads

M, K, N = 512, 384, 640
torch.cuda.init()

def inputs(i):
    g = workloads.gen(100 + i, "cuda")
    x8 = (torch.randn(M, K, generator=g, device="cuda") * 4).to(torch.float8_e4m3fn).view(torch.uint8)
    w8 = (torch.randn(N, K, generator=g, device="cuda") * 4).to(torch.float8_e4m3fn).view(torch.uint8)
    d8 = (torch.randn(M, N, generator=g, device="cuda") * 4).to(torch.float8_e5m2).view(torch.uint8)
    gr = (torch.randn(N * K, generator=g, device="cuda") * 1e-3).to(torch.bfloat16)
    return x8, w8, d8, gr

def run(i, stream, ins):
    x8, w8, d8, gr = ins
    with torch.cuda.stream(stream):
        one = torch.ones(1, device="cuda")
        y = torch.empty(M, N, device="cuda")
        dx = torch.empty(M, K, device="cuda")
        dw = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
        f.fp8_linear_fwd(x8, w8, one, one, y)
        f.fp8_linear_bwd_rowmajor(d8, w8, x8, one, one, one, dx, dw)
        w = torch.full((N * K,), 0.5, device="cuda"); v = torch.zeros_like(w)
        q = torch.zeros(N * K, dtype=torch.uint8, device="cuda")
        am = torch.zeros(1, device="cuda"); S = torch.tensor([2.0 ** 16], device="cuda")
        gc = torch.zeros(1, dtype=torch.int32, device="cuda"); fi = torch.zeros(1, dtype=torch.int32, device="cuda")
        f.mp_master_step(gr, w, v, q, one, am, S, gc, fi, 1e-2, 0.9)
        stream.synchronize()
        return [y, dx, dw, w, v, q, am, S, gc, fi]

ins = [inputs(i) for i in range(8)]
torch.cuda.synchronize()
streams = [torch.cuda.Stream() for _ in range(8)]
out = [None] * 8
barrier = threading.Barrier(8)

def worker(i):
    barrier.wait()
    out[i] = run(i, streams[i], ins[i])

threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert f.fp8mp_check() == 0
for i in range(8):
    ref = run(i, torch.cuda.current_stream(), ins[i])
    assert all(torch.equal(a, b) for a, b in zip(out[i], ref)), i
print("threads ok")
"""


def test_first_calls_from_eight_threads():
    code = CHILD.replace("ROOT", repr(ROOT), 1)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert "threads ok" in r.stdout
