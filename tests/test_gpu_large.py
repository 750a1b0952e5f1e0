"""Kernels on more than 2^31 elements, where 32-bit index arithmetic would
wrap: the transposing bf16 -> E4M3 cast (every row-major code and the amax
against the oracle, the transposed copy against a transpose of the codes)
and the master step on 2^31 + 24 parameters (the self-scanning and the
flag-reading version, bit-exact against the oracle over a clean, a skipped
and a clean step)."""

import os

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, assert_same_bits, np_view

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def host_memory_gb() -> float:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 2 ** 20
    except OSError:
        pass
    return 0.0


def test_cast_beyond_2_31_elements(cuda_lib, orc):
    rows, cols = 65552, 32768  # 2,148,007,936 elements > 2^31
    assert rows * cols > 2 ** 31
    g = workloads.gen(2 ** 31, "cuda")
    x = (torch.randn((rows, cols), generator=g, device="cuda") * 3).to(torch.bfloat16)
    scale = torch.tensor([64.0], device="cuda")
    amax = torch.zeros(1, device="cuda")
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    cuda_lib.fp8_quantize(x, E4M3, scale, out, out_t, amax)
    assert cuda_lib.fp8mp_check() == 0
    assert torch.equal(out_t, out.t().contiguous())  # the transposed copy, every element
    del out_t
    xn = np_view(x)
    del x
    assert_same_bits(np_view(amax), np.array([orc.amax(xn)], np.float32), "amax")
    q = orc.cast(xn, 64.0, E4M3)
    del xn
    assert np.array_equal(out.cpu().numpy(), q)


def test_master_step_beyond_2_31_parameters(cuda_lib, orc):
    if host_memory_gb() < 96:
        pytest.skip("needs about 40 GB of free host memory for the oracle's copy")
    n = 2 ** 31 + 24
    w = workloads.master_weights(n, seed=11, device="cuda")
    v = torch.zeros(n, dtype=torch.float32, device="cuda")
    w8 = torch.zeros(n, dtype=torch.uint8, device="cuda")
    sw, am = torch.tensor([256.0], device="cuda"), torch.zeros(1, device="cuda")
    S, growth = torch.tensor([2.0 ** 16], device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
    found, flag = torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
    hw, hv, h8, ham = np_view(w).copy(), np.zeros(n, np.float32), np.zeros(n, np.uint8), np.zeros(1, np.float32)
    st = orc.LossScaleState(2.0 ** 16)
    for step, inject in ((0, False), (1, True), (2, False)):
        g = workloads.master_step(n, step, seed=11, inject=inject, device="cuda")
        if step == 0:  # the self-scanning step
            cuda_lib.mp_master_step(g, w, v, w8, sw, am, S, growth, found, 1e-4, 0.9)
        else:  # the step on the producer's flag
            flag.fill_(int(((g.view(torch.int16) & 0x7F80) == 0x7F80).any().item()))
            cuda_lib.mp_master_step(g, w, v, w8, sw, am, S, growth, found, 1e-4, 0.9, grad_nonfinite=flag)
        assert cuda_lib.fp8mp_check() == 0
        gn = np_view(g)
        del g
        orc.master_step(gn, hw, hv, h8, 256.0, ham, st, 1e-4, 0.9)
        del gn
        assert found.item() == st.found_inf[0] == int(inject) and flag.item() == 0
        assert S.item() == st.S[0] and growth.item() == st.growth[0]
        assert_same_bits(np_view(am), ham, f"step {step} amax")
        assert np.array_equal(np_view(w).view(np.uint32), hw.view(np.uint32)), f"step {step} master"
        assert np.array_equal(np_view(v).view(np.uint32), hv.view(np.uint32)), f"step {step} momentum"
        assert np.array_equal(w8.cpu().numpy(), h8), f"step {step} w8"
