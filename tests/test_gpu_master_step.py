"""GPU parity of mp_master_step against the oracle: master weights, momentum,
E4M3 copy, weight amax, loss scale, growth counter and overflow flag, all
bit-exact, over ragged sizes, overflow skips and growth boundaries, and the
1e9-parameter workload (steps 0, 1 with 0.01 % injected Inf/NaN, 2)."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_same_bits, np_view

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["fused", "three_launches"])
def path(request, monkeypatch):
    """Runs a test on both versions of the step: one cooperative launch
    (scan, grid barrier, update, last-block bookkeeping) and three launches
    (the library reads FP8MP_FUSED_MASTER per call)."""
    monkeypatch.setenv("FP8MP_FUSED_MASTER", "1" if request.param == "fused" else "0")
    return request.param


class DevState:
    def __init__(self, w, S, growth, device="cuda"):
        n = w.numel()
        self.w = w.to(device).clone()
        self.v = torch.zeros(n, dtype=torch.float32, device=device)
        self.w8 = torch.zeros(n, dtype=torch.uint8, device=device)
        self.scale_w = torch.ones(1, dtype=torch.float32, device=device)
        self.amax_w = torch.zeros(1, dtype=torch.float32, device=device)
        self.S = torch.tensor([S], dtype=torch.float32, device=device)
        self.growth = torch.tensor([growth], dtype=torch.int32, device=device)
        self.found = torch.zeros(1, dtype=torch.int32, device=device)


def step_both(fp8mp, orc, ds, os_, g, lr, mu, scale_w, interval=2000):
    ds.scale_w.fill_(scale_w)
    fp8mp.mp_master_step(g.cuda() if not g.is_cuda else g, ds.w, ds.v, ds.w8, ds.scale_w, ds.amax_w, ds.S,
                         ds.growth, ds.found, lr, mu, 0.5, 2.0, interval)
    assert fp8mp.fp8mp_check() == 0
    gn = np_view(g)
    orc.master_step(gn, os_["w"], os_["v"], os_["w8"], scale_w, os_["am"], os_["st"], lr, mu, 0.5, 2.0, interval)


def compare(ds, os_, what):
    assert_same_bits(np_view(ds.w), os_["w"], what + " master")
    assert_same_bits(np_view(ds.v), os_["v"], what + " momentum")
    assert_same_bits(np_view(ds.w8), os_["w8"], what + " w8")
    assert_same_bits(np_view(ds.amax_w), os_["am"], what + " amax")
    assert_same_bits(np_view(ds.S), os_["st"].S, what + " S")
    assert ds.growth.item() == os_["st"].growth[0], what
    assert ds.found.item() == os_["st"].found_inf[0], what


def host_state(w, S, growth, orc):
    n = w.numel()
    return {"w": np_view(w).copy(), "v": np.zeros(n, np.float32), "w8": np.zeros(n, np.uint8),
            "am": np.zeros(1, np.float32), "st": orc.LossScaleState(S, growth)}


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 1000, 12345, (1 << 20) + 3])
def test_ragged_sizes_with_skip_and_growth(cuda_lib, orc, path, n):
    w = workloads.master_weights(n, seed=n)
    ds = DevState(w, 2.0 ** 16, 1997)
    hs = host_state(w, 2.0 ** 16, 1997, orc)
    for step in range(5):
        g = workloads.master_step(n, step, seed=n, inject=(step == 2 and n > 0), inject_frac=1e-3)
        step_both(cuda_lib, orc, ds, hs, g, 1e-4, 0.9, scale_w=float(2 ** (step + 4)))
        compare(ds, hs, f"n={n} step={step}")
    # 1997 + 2 clean steps = growth at 1999; step 2 overflowed (reset); then 2 clean
    if n > 0:
        assert hs["st"].growth[0] == 2


def test_growth_interval_doubles_S(cuda_lib, orc, path):
    n = 4096
    w = workloads.master_weights(n)
    ds = DevState(w, 8.0, 0)
    hs = host_state(w, 8.0, 0, orc)
    for step in range(7):
        g = workloads.master_step(n, step)
        ds.found.fill_(12345)  # found_inf's content on entry does not matter
        step_both(cuda_lib, orc, ds, hs, g, 1e-3, 0.5, 1.0, interval=3)
        compare(ds, hs, f"step={step}")
    assert ds.S.item() == 32.0 and ds.growth.item() == 1


@pytest.mark.slow
def test_1e9_parameters(cuda_lib, orc):
    """The 1e9-parameter flat buffer: fp32 master ~ N(0, 0.02), bf16 grads
    ~ N(0, 1e-5) * 2^16, S = 2^16, lr 1e-4, mu 0.9; step 1 carries 0.01 %
    +-Inf/NaN and must be skipped bit-exactly."""
    n = 1_000_000_000
    w = workloads.master_weights(n, device="cuda")
    ds = DevState(w, 2.0 ** 16, 0)
    hs = host_state(w, 2.0 ** 16, 0, orc)
    del w
    for step in range(3):
        g = workloads.master_step(n, step, inject=(step == 1), device="cuda")
        step_both(cuda_lib, orc, ds, hs, g, 1e-4, 0.9, scale_w=float(2 ** 9))
        del g
        compare(ds, hs, f"1e9 step={step}")
    assert hs["st"].found_inf[0] == 0 and hs["st"].S[0] == 2.0 ** 15


# ------------------------------------------------------------- Adam variant


@pytest.mark.parametrize("n", [0, 1, 9, 4096, (1 << 20) + 5])
def test_adam_steps_bit_exact(cuda_lib, orc, path, n):
    w = workloads.master_weights(n, seed=n + 1)
    ds = DevState(w, 2.0 ** 16, 0)
    m = torch.zeros(n, dtype=torch.float32, device="cuda")
    bp = torch.ones(2, dtype=torch.float32, device="cuda")
    hs = host_state(w, 2.0 ** 16, 0, orc)
    hm = np.zeros(n, np.float32)
    ad = orc.AdamState()
    for step in range(4):
        g = workloads.master_step(n, step, seed=n + 1, inject=(step == 2 and n > 0), inject_frac=1e-3)
        ds.scale_w.fill_(64.0)
        cuda_lib.mp_master_step_adam(g.cuda(), ds.w, m, ds.v, ds.w8, ds.scale_w, ds.amax_w, ds.S, ds.growth,
                                     ds.found, bp, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
        assert cuda_lib.fp8mp_check() == 0
        orc.adam_step(np_view(g), hs["w"], hm, hs["v"], hs["w8"], 64.0, hs["am"], hs["st"], ad, lr=1e-3,
                      beta1=0.9, beta2=0.999, eps=1e-8)
        compare(ds, hs, f"adam n={n} step={step}")
        assert_same_bits(np_view(m), hm, "exp_avg")
        assert_same_bits(np_view(bp), np.array([ad.b1p[0], ad.b2p[0]], np.float32), "beta powers")


# ------------------------------------------- steps on a producer's flag


@pytest.mark.parametrize("opt", ["sgd", "adam"])
@pytest.mark.parametrize("n", [1, 9, 4096, (1 << 20) + 3])
def test_prescanned_steps_bit_exact(cuda_lib, orc, opt, n):
    """mp_master_step(_adam) with grad_nonfinite: the flag set from a host
    scan of the gradients stands in for the producer's (the GEMM epilogue's
    flag has its own test); results bit-exact against the oracle, found_inf
    equal to the flag, the flag reset to 0."""
    w = workloads.master_weights(n, seed=n + 7)
    ds = DevState(w, 2.0 ** 16, 0)
    hs = host_state(w, 2.0 ** 16, 0, orc)
    m = torch.zeros(n, dtype=torch.float32, device="cuda")
    bp = torch.ones(2, dtype=torch.float32, device="cuda")
    hm = np.zeros(n, np.float32)
    ad = orc.AdamState()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(4):
        g = workloads.master_step(n, step, seed=n + 7, inject=(step == 1), inject_frac=1e-3)
        gb = np_view(g)
        flag.fill_(int(((gb & 0x7F80) == 0x7F80).any()))
        ds.found.fill_(0x5A5A)  # no memset precedes this step: found_inf is written whatever it held
        ds.scale_w.fill_(32.0)
        if opt == "sgd":
            cuda_lib.mp_master_step(g.cuda(), ds.w, ds.v, ds.w8, ds.scale_w, ds.amax_w, ds.S, ds.growth, ds.found,
                                    1e-4, 0.9, grad_nonfinite=flag)
            orc.master_step(gb, hs["w"], hs["v"], hs["w8"], 32.0, hs["am"], hs["st"], 1e-4, 0.9)
        else:
            cuda_lib.mp_master_step_adam(g.cuda(), ds.w, m, ds.v, ds.w8, ds.scale_w, ds.amax_w, ds.S, ds.growth,
                                         ds.found, bp, lr=1e-3, grad_nonfinite=flag)
            orc.adam_step(gb, hs["w"], hm, hs["v"], hs["w8"], 32.0, hs["am"], hs["st"], ad, lr=1e-3)
        assert cuda_lib.fp8mp_check() == 0
        compare(ds, hs, f"{opt} prescanned n={n} step={step}")
        assert flag.item() == 0
        if opt == "adam":
            assert_same_bits(np_view(m), hm, "exp_avg")
            assert_same_bits(np_view(bp), np.array([ad.b1p[0], ad.b2p[0]], np.float32), "beta powers")
    assert hs["st"].S[0] == 2.0 ** 15  # the injected step backed off once
