"""GPU parity of delayed_scaling_update (bit-exact histories, scales, scale_inv,
cur_amax) and of the 768 -> 768 linear workloads end to end: the one-step
forward, and the 32-step HYBRID drift run (fwd + dgrad + wgrad + update per
step) where every code, amax and scale must match the oracle bit-exactly and
every GEMM output must be within tolerance."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, E5M2, assert_same_bits, dev, gemm_tolerance_check, np_view

pytestmark = pytest.mark.gpu


def set_meta(dm, om):
    dm.amax_history.copy_(torch.from_numpy(om.hist))
    dm.scale.copy_(torch.from_numpy(om.scale))
    dm.scale_inv.copy_(torch.from_numpy(om.scale_inv))
    dm.cur_amax.copy_(torch.from_numpy(om.cur_amax))


def assert_meta_equal(dm, om, what):
    assert_same_bits(np_view(dm.amax_history), om.hist, what + " history")
    assert_same_bits(np_view(dm.scale), om.scale, what + " scale")
    assert_same_bits(np_view(dm.scale_inv), om.scale_inv, what + " scale_inv")
    assert_same_bits(np_view(dm.cur_amax), om.cur_amax, what + " cur_amax")


@pytest.mark.parametrize("L", [1, 3, 16, 1024, 8192])
@pytest.mark.parametrize("algo", [0, 1])
def test_update_sequences(cuda_lib, orc, L, algo):
    rng = np.random.default_rng(L + algo)
    fmts = [E4M3, E5M2, E4M3, E5M2, E4M3]
    dms = [cuda_lib.Meta(L, f) for f in fmts]
    oms = [orc.Meta(L) for _ in fmts]
    for step in range(40):
        margin = step % 3
        for i, (dm, om) in enumerate(zip(dms, oms)):
            a = np.float32(10.0 ** rng.uniform(-30, 30))
            if step % 11 == 5 + i:
                a = np.float32(0.0)
            if step == 17 and i == 1:
                a = np.float32(np.inf)
            if step == 23 and i == 2:
                a = np.float32(1e-39)  # fmt_max / a overflows: scale kept
            om.cur_amax[0] = a
            dm.cur_amax.fill_(float(a))
        cuda_lib.delayed_scaling_update(dms, algo, margin)
        for dm, om, f in zip(dms, oms, fmts):
            orc.scale_update(om, f, algo, margin)
        torch.cuda.synchronize()
        for i, (dm, om) in enumerate(zip(dms, oms)):
            assert_meta_equal(dm, om, f"step {step} meta {i}")


def test_more_metas_than_one_launch(cuda_lib, orc):
    n = 70  # spans three launches of the batched kernel
    dms = [cuda_lib.Meta(4, i % 2) for i in range(n)]
    oms = [orc.Meta(4) for _ in range(n)]
    for step in range(3):
        for i in range(n):
            a = np.float32(1.0 + i + 100 * step)
            oms[i].cur_amax[0] = a
            dms[i].cur_amax.fill_(float(a))
        cuda_lib.delayed_scaling_update(dms, 0, 1)
        for i in range(n):
            orc.scale_update(oms[i], i % 2, 0, 1)
    torch.cuda.synchronize()
    for i in range(n):
        assert_meta_equal(dms[i], oms[i], f"meta {i}")


def test_linear768_forward_one_step(cuda_lib, orc):
    """1024 x 768 fp32 input U[0,1), 768 x 768 weight, bias, E4M3,
    DelayedScaling(L=16, max, margin 0): one step at the initial scale 1,
    then one update; output fp32 as the input."""
    lw = workloads.linear768()
    xn, wn = np_view(lw.x), np_view(lw.w)
    mx, mw, my = (cuda_lib.Meta(16, E4M3) for _ in range(3))
    ox, ow, oy = (orc.Meta(16) for _ in range(3))
    X8 = torch.empty((1024, 768), dtype=torch.uint8, device="cuda")
    W8 = torch.empty((768, 768), dtype=torch.uint8, device="cuda")
    cuda_lib.fp8_quantize(lw.x.cuda(), E4M3, mx.scale, X8, None, mx.cur_amax)
    cuda_lib.fp8_quantize(lw.w.cuda(), E4M3, mw.scale, W8, None, mw.cur_amax)
    y = torch.empty((1024, 768), dtype=torch.float32, device="cuda")
    cuda_lib.fp8_linear_fwd(X8, W8, mx.scale_inv, mw.scale_inv, y, bias=lw.b.cuda(), y_amax=my.cur_amax)
    assert cuda_lib.fp8mp_check() == 0
    qx, qw = orc.cast(xn, 1.0, E4M3), orc.cast(wn, 1.0, E4M3)
    ox.record_amax(orc.amax(xn))
    ow.record_amax(orc.amax(wn))
    assert_same_bits(X8.cpu().numpy(), qx, "X8")
    assert_same_bits(W8.cpu().numpy(), qw, "W8")
    ref, ab = orc.gemm_ref(qx, E4M3, qw, E4M3, 1.0, 1.0, bias=lw.b.double().numpy())
    yh = np_view(y)
    gemm_tolerance_check(yh.astype(np.float64), ref, ab, "linear768 fwd")
    assert my.cur_amax.item() == np.abs(yh).max()
    cuda_lib.delayed_scaling_update([mx, mw], 0, 0)
    orc.scale_update(ox, E4M3, 0, 0)
    orc.scale_update(ow, E4M3, 0, 0)
    torch.cuda.synchronize()
    assert_meta_equal(mx, ox, "x")
    assert_meta_equal(mw, ow, "w")


def test_linear768_hybrid_drift_32_steps(cuda_lib, orc):
    """HYBRID recipe, L = 16, algo max, margin 0; x_t = x_0 * 1.1^t and
    dy_t ~ N(0, 1e-3) bf16. Each step: cast x (+T), cast w (+T), fwd (+amax),
    cast dy to E5M2 (+T), dgrad, wgrad, then one batched scale update."""
    base = workloads.linear768()
    wn = np_view(base.w)
    W = base.w.cuda()
    b = base.b.cuda()
    names = ("x", "w", "y", "dy")
    fmts = {"x": E4M3, "w": E4M3, "y": E4M3, "dy": E5M2}
    dm = {k: cuda_lib.Meta(16, fmts[k]) for k in names}
    om = {k: orc.Meta(16) for k in names}
    M = N = K = None
    for t in range(32):
        x_t, dy_t = workloads.linear768_drift_step(base, t)
        xn, dyn = np_view(x_t), np_view(dy_t)
        M, K = x_t.shape
        N = W.shape[0]
        X8 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
        X8t = torch.empty((K, M), dtype=torch.uint8, device="cuda")
        W8 = torch.empty((N, K), dtype=torch.uint8, device="cuda")
        W8t = torch.empty((K, N), dtype=torch.uint8, device="cuda")
        D8 = torch.empty((M, N), dtype=torch.uint8, device="cuda")
        D8t = torch.empty((N, M), dtype=torch.uint8, device="cuda")
        cuda_lib.fp8_quantize(x_t.cuda(), E4M3, dm["x"].scale, X8, X8t, dm["x"].cur_amax)
        cuda_lib.fp8_quantize(W, E4M3, dm["w"].scale, W8, W8t, dm["w"].cur_amax)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        cuda_lib.fp8_linear_fwd(X8, W8, dm["x"].scale_inv, dm["w"].scale_inv, y, bias=b, y_amax=dm["y"].cur_amax)
        cuda_lib.fp8_quantize(dy_t.cuda(), E5M2, dm["dy"].scale, D8, D8t, dm["dy"].cur_amax)
        dx = torch.empty((M, K), dtype=torch.float32, device="cuda")
        dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
        cuda_lib.fp8_linear_dgrad(D8, W8t, dm["dy"].scale_inv, dm["w"].scale_inv, dx)
        cuda_lib.fp8_linear_wgrad(D8t, X8t, dm["dy"].scale_inv, dm["x"].scale_inv, dw)
        assert cuda_lib.fp8mp_check() == 0

        # oracle, same step
        qx = orc.cast(xn, float(om["x"].scale[0]), E4M3)
        qw = orc.cast(wn, float(om["w"].scale[0]), E4M3)
        qd = orc.cast(dyn, float(om["dy"].scale[0]), E5M2)
        om["x"].record_amax(orc.amax(xn))
        om["w"].record_amax(orc.amax(wn))
        om["dy"].record_amax(orc.amax(dyn))
        assert_same_bits(X8.cpu().numpy(), qx, f"t={t} X8")
        assert_same_bits(X8t.cpu().numpy(), orc.transpose_u8(qx), f"t={t} X8t")
        assert_same_bits(W8.cpu().numpy(), qw, f"t={t} W8")
        assert_same_bits(W8t.cpu().numpy(), orc.transpose_u8(qw), f"t={t} W8t")
        assert_same_bits(D8.cpu().numpy(), qd, f"t={t} dY8")
        assert_same_bits(D8t.cpu().numpy(), orc.transpose_u8(qd), f"t={t} dY8t")
        sx, sw, sd = (float(om[k].scale_inv[0]) for k in ("x", "w", "dy"))
        ref, ab = orc.gemm_ref(qx, E4M3, qw, E4M3, sx, sw, bias=base.b.double().numpy())
        yh = np_view(y)
        gemm_tolerance_check(yh.astype(np.float64), ref, ab, f"t={t} fwd")
        assert dm["y"].cur_amax.item() == np.abs(yh).max()
        om["y"].record_amax(np.float32(np.abs(yh).max()))  # the output amax is defined on the stored values
        ref, ab = orc.gemm_ref(qd, E5M2, orc.transpose_u8(qw), E4M3, sd, sw)
        gemm_tolerance_check(np_view(dx).astype(np.float64), ref, ab, f"t={t} dgrad")
        ref, ab = orc.gemm_ref(orc.transpose_u8(qd), E5M2, orc.transpose_u8(qx), E4M3, sd, sx)
        gemm_tolerance_check(np_view(dw).astype(np.float64), ref, ab, f"t={t} wgrad")

        cuda_lib.delayed_scaling_update([dm[k] for k in names], 0, 0)
        for k in names:
            orc.scale_update(om[k], fmts[k], 0, 0)
        torch.cuda.synchronize()
        for k in names:
            assert_meta_equal(dm[k], om[k], f"t={t} meta {k}")
    # the drift saturates the top of x once its amax outgrows the history
    assert om["x"].scale[0] < 448.0 / 1.1 ** 20
