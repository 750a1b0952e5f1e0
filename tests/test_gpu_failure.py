"""Failure detection on the GPU without a fault: a kernel's bounded wait on a
barrier nothing signals (a GEMM's mbarrier, the master step's grid barrier)
runs out, the device flag it raises comes back as FP8MP_ERR_TIMEOUT from
fp8mp_check, and the context keeps working."""

import numpy as np
import pytest
import torch

from gpu_util import E4M3, dev, finite_codes, gemm_tolerance_check, np_view

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib, orc):
    assert cuda_lib.fp8mp_check() == 0
    cuda_lib.fp8mp_selftest_timeout()
    assert cuda_lib.fp8mp_check() == cuda_lib.ERR_TIMEOUT
    assert "wait expired" in cuda_lib.last_error()
    # the flag was cleared and the context still runs GEMMs correctly
    assert cuda_lib.fp8mp_check() == 0
    rng = np.random.default_rng(1)
    A = finite_codes(rng, (256, 256), E4M3)
    B = finite_codes(rng, (256, 256), E4M3)
    one = torch.ones(1, device="cuda")
    y = torch.empty((256, 256), dtype=torch.float32, device="cuda")
    cuda_lib.fp8_linear_fwd(dev(A), dev(B), one, one, y)
    assert cuda_lib.fp8mp_check() == 0
    ref, ab = orc.gemm_ref(A, E4M3, B, E4M3, 1.0, 1.0)
    gemm_tolerance_check(np_view(y).astype(np.float64), ref, ab, "after timeout")


def test_grid_barrier_timeout_reported_and_master_step_still_exact(cuda_lib, orc):
    """The master step's grid barrier: a wait that nothing completes runs out,
    comes back as FP8MP_ERR_TIMEOUT, and a following fused step is bit-exact."""
    import workloads

    assert cuda_lib.fp8mp_check() == 0
    cuda_lib.fp8mp_selftest_barrier_timeout()
    assert cuda_lib.fp8mp_check() == cuda_lib.ERR_TIMEOUT
    assert "grid barrier" in cuda_lib.last_error()
    assert cuda_lib.fp8mp_check() == 0
    n = 100_003
    w = workloads.master_weights(n)
    g = workloads.master_step(n, 0)
    wd, v, w8 = w.cuda(), torch.zeros(n, device="cuda"), torch.zeros(n, dtype=torch.uint8, device="cuda")
    sw, am = torch.ones(1, device="cuda"), torch.zeros(1, device="cuda")
    S, gr, fi = (torch.tensor([2.0 ** 16], device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"),
                 torch.zeros(1, dtype=torch.int32, device="cuda"))
    cuda_lib.mp_master_step(g.cuda(), wd, v, w8, sw, am, S, gr, fi, 1e-4, 0.9)
    assert cuda_lib.fp8mp_check() == 0
    hw, hv, h8, ham = np_view(w).copy(), np.zeros(n, np.float32), np.zeros(n, np.uint8), np.zeros(1, np.float32)
    st = orc.LossScaleState(2.0 ** 16)
    orc.master_step(np_view(g), hw, hv, h8, 1.0, ham, st, 1e-4, 0.9)
    assert np.array_equal(np_view(wd).view(np.uint32), hw.view(np.uint32))
    assert np.array_equal(w8.cpu().numpy(), h8) and fi.item() == 0 and gr.item() == 1


def test_invalid_arguments_on_a_gpu_enqueue_nothing(cuda_lib):
    x = torch.ones((24, 16), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((24, 16), dtype=torch.uint8, device="cuda")
    out_t = torch.zeros((16, 24), dtype=torch.uint8, device="cuda")
    s = torch.ones(1, device="cuda")
    with pytest.raises(cuda_lib.Fp8mpError) as e:
        cuda_lib.fp8_quantize(x, E4M3, s, out, out_t)  # 24 rows: not a multiple of 16
    assert e.value.code == cuda_lib.ERR_INVALID
    assert cuda_lib.fp8mp_check() == 0
    assert (out.cpu() == 0).all()
