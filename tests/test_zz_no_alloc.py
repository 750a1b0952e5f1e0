"""The allocation-free bias-gradient cast, for callers that cannot call
cudaMalloc (a framework pool owns the device, plugin code is handed only its
tensors, or a latency-critical path cannot take cudaMalloc's implicit device
synchronisation): its results must match the workspace entry point's on two
calls in a row, and shapes beyond its fixed scratch array must be refused.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process."""

import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E5M2, np_view

pytestmark = pytest.mark.gpu


def dbias_close(got, ref, ab, rows, bf16):
    # the tolerance of the fused-dbias parity tests: fp32 summation of `rows`
    # terms plus, for bf16, one rounding with unit roundoff 2^-8
    err = np.abs(got.astype(np.float64) - ref)
    bound = rows * 2.0 ** -24 * ab + (2.0 ** -8 * (np.abs(ref) + rows * 2.0 ** -24 * ab) if bf16 else 0.0) + 1e-30
    return bool((err <= bound).all())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def run_noalloc_c_abi(lib, dy, scale, out, out_t, db, am):
    """Calls the C entry point directly through ctypes (out_t and am may be
    None: no transposed copy, no amax)."""
    rc = lib.fp8_quantize_dbias_noalloc(
        _p(dy), 1 if dy.dtype == torch.bfloat16 else 0, dy.shape[0], dy.shape[1], E5M2, _p(scale), _p(out),
        _p(out_t), _p(am), _p(db), 1 if db.dtype == torch.bfloat16 else 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("rows,cols,db_dtype", [(8192, 4096, torch.float32), (1040, 784, torch.bfloat16)])
def test_noalloc_matches_workspace_entry_point_twice(cuda_lib, orc, rows, cols, db_dtype):
    lib = cuda_lib.load()
    scale = torch.tensor([2048.0], device="cuda")
    for call in range(2):
        g = workloads.gen(rows + 31 * call)
        dy = (torch.randn((rows, cols), generator=g) * 1e-3 + 1e-4 * call).to(torch.bfloat16).cuda()
        # reference: the existing entry point with a torch-allocated workspace
        out_r = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        out_tr = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
        db_r = torch.empty(cols, dtype=db_dtype, device="cuda")
        am_r = torch.zeros(1, device="cuda")
        ws = torch.zeros(cuda_lib.fp8_quantize_dbias_workspace_bytes(rows, cols) // 4, device="cuda")
        cuda_lib.fp8_quantize_dbias(dy, E5M2, scale, out_r, out_tr, db_r, ws, amax=am_r)
        # the allocation-free entry point through the C ABI
        out = torch.empty_like(out_r)
        out_t = torch.empty_like(out_tr)
        db = torch.empty_like(db_r)
        am = torch.zeros(1, device="cuda")
        assert run_noalloc_c_abi(lib, dy, scale, out, out_t, db, am) == 0, cuda_lib.last_error()
        assert cuda_lib.fp8mp_check() == 0
        assert torch.equal(out, out_r) and torch.equal(out_t, out_tr)
        assert torch.equal(am, am_r)
        # the same kernel and summation order as the workspace entry point
        assert torch.equal(db, db_r)
        ref, ab = orc.dbias(np_view(dy))
        bf16 = db_dtype == torch.bfloat16
        assert dbias_close(np_view(db.float()), ref, ab, rows, bf16), f"call {call}"
        assert dbias_close(np_view(db_r.float()), ref, ab, rows, bf16), f"call {call}"


def test_noalloc_refuses_shapes_beyond_its_scratch(cuda_lib):
    lib = cuda_lib.load()
    rows, cols = 16384, 1040448  # its column sums and counters need more than 2^20 floats
    dy = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")  # never read: refused first
    rc = lib.fp8_quantize_dbias_noalloc(ctypes.c_void_p(dy.data_ptr()), 1, rows, cols, E5M2,
                                        ctypes.c_void_p(dy.data_ptr()), ctypes.c_void_p(dy.data_ptr()),
                                        ctypes.c_void_p(dy.data_ptr()), None, ctypes.c_void_p(dy.data_ptr()), 0,
                                        None)
    assert rc == cuda_lib.ERR_INVALID
    assert "scratch" in cuda_lib.last_error()
    assert cuda_lib.fp8mp_check() == 0


def test_noalloc_warm_call_allocates_no_device_memory(cuda_lib):
    """The promise of this entry point: once warm (the first call on a device
    looks up the scratch array's address and loads the kernel), a call leaves
    the device's free memory exactly as it was."""
    lib = cuda_lib.load()
    rows, cols = 4096, 2048
    dy = (torch.randn((rows, cols), generator=workloads.gen(77)) * 1e-3).to(torch.bfloat16).cuda()
    scale = torch.tensor([4096.0], device="cuda")
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    db = torch.empty(cols, device="cuda")
    am = torch.zeros(1, device="cuda")
    assert run_noalloc_c_abi(lib, dy, scale, out, out_t, db, am) == 0, cuda_lib.last_error()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert run_noalloc_c_abi(lib, dy, scale, out, out_t, db, am) == 0, cuda_lib.last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert cuda_lib.fp8mp_check() == 0


def test_noalloc_without_transposed_copy_or_amax(cuda_lib, orc):
    """out_t = NULL and amax = NULL: the same codes and bias gradient as the
    workspace entry point given the same NULLs, on two calls in a row."""
    lib = cuda_lib.load()
    rows, cols = 2064, 1040
    scale = torch.tensor([2048.0], device="cuda")
    ws = torch.zeros(cuda_lib.fp8_quantize_dbias_workspace_bytes(rows, cols) // 4, device="cuda")
    for call in range(2):
        dy = (torch.randn((rows, cols), generator=workloads.gen(500 + call)) * 1e-3).to(torch.bfloat16).cuda()
        out_r, db_r = torch.empty((rows, cols), dtype=torch.uint8, device="cuda"), torch.empty(cols, device="cuda")
        cuda_lib.fp8_quantize_dbias(dy, E5M2, scale, out_r, None, db_r, ws)
        out, db = torch.empty_like(out_r), torch.empty_like(db_r)
        assert run_noalloc_c_abi(lib, dy, scale, out, None, db, None) == 0, cuda_lib.last_error()
        assert cuda_lib.fp8mp_check() == 0
        assert torch.equal(out, out_r) and torch.equal(db, db_r)
        dyn = np_view(dy)
        np.testing.assert_array_equal(out.cpu().numpy(), orc.cast(dyn, 2048.0, E5M2))
        ref, ab = orc.dbias(dyn)
        assert dbias_close(np_view(db), ref, ab, rows, False), f"call {call}"
