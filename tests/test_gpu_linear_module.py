"""FP8Linear (autograd wrapper) on the 768 -> 768 layer: forward output,
input / weight / bias gradients and the delayed-scaling state over two
steps, against the oracle's composition of the same steps."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, E5M2, assert_same_bits, gemm_tolerance_check, np_view

pytestmark = pytest.mark.gpu


def test_fp8linear_two_steps(cuda_lib, orc):
    from fp8_mixed_precision_reduce_gb300.linear import FP8Linear

    base = workloads.linear768()
    layer = FP8Linear(768, 768, bias=True, history_len=16)
    with torch.no_grad():
        layer.weight.copy_(base.w)
        layer.bias.copy_(base.b)
    om = {k: orc.Meta(16) for k in ("x", "w", "y", "dy")}
    fmts = {"x": E4M3, "w": E4M3, "y": E4M3, "dy": E5M2}
    wn = np_view(base.w)
    for t in range(2):
        x_t, dy_t = workloads.linear768_drift_step(base, t)
        dy_t = dy_t.float()  # the layer runs in fp32 like its input
        x = x_t.cuda().requires_grad_(True)
        layer.zero_grad(set_to_none=True)
        y = layer(x)
        y.backward(dy_t.cuda())
        assert cuda_lib.fp8mp_check() == 0

        xn, dyn = np_view(x_t), np_view(dy_t)
        qx = orc.cast(xn, float(om["x"].scale[0]), E4M3)
        qw = orc.cast(wn, float(om["w"].scale[0]), E4M3)
        qd = orc.cast(dyn, float(om["dy"].scale[0]), E5M2)
        sx, sw, sd = (float(om[k].scale_inv[0]) for k in ("x", "w", "dy"))
        ref, ab = orc.gemm_ref(qx, E4M3, qw, E4M3, sx, sw, bias=base.b.double().numpy())
        yh = np_view(y.detach())
        gemm_tolerance_check(yh.astype(np.float64), ref, ab, f"t={t} y")
        # the three gradients are all checked before any failure is raised:
        # which of them agree tells a wrong E5M2 copy of dY (dx, dw and the
        # codes behind them) from a wrong store of one output
        failed = []
        ref, ab = orc.gemm_ref(qd, E5M2, orc.transpose_u8(qw), E4M3, sd, sw)
        try:
            gemm_tolerance_check(np_view(x.grad).astype(np.float64), ref, ab, f"t={t} dx")
        except AssertionError as e:
            failed.append(str(e))
        ref, ab = orc.gemm_ref(orc.transpose_u8(qd), E5M2, orc.transpose_u8(qx), E4M3, sd, sx)
        try:
            gemm_tolerance_check(np_view(layer.weight.grad).astype(np.float64), ref, ab, f"t={t} dw")
        except AssertionError as e:
            failed.append(str(e))
        db_ref, db_abs = orc.dbias(dyn)
        err = np.abs(np_view(layer.bias.grad).astype(np.float64) - db_ref)
        if not (err <= 1024 * 2.0 ** -24 * db_abs + 1e-30).all():
            failed.append(f"t={t} dbias: {int((err > 1024 * 2.0 ** -24 * db_abs + 1e-30).sum())} columns out of bound")
        assert not failed, "\n".join(failed)

        om["x"].record_amax(orc.amax(xn))
        om["w"].record_amax(orc.amax(wn))
        om["dy"].record_amax(orc.amax(dyn))
        om["y"].record_amax(np.float32(np.abs(yh).max()))
        layer.update_scales()
        for k in fmts:
            orc.scale_update(om[k], fmts[k], 0, 0)
        torch.cuda.synchronize()
        for k, dm in zip(("x", "w", "y", "dy"), layer.metas()):
            assert_same_bits(np_view(dm.scale), om[k].scale, f"t={t} scale {k}")
            assert_same_bits(np_view(dm.amax_history), om[k].hist, f"t={t} history {k}")
        assert layer.dw_nonfinite.item() == 0  # finite weight gradient


def test_fp8linear_flags_a_nonfinite_weight_gradient(cuda_lib):
    """The layer's dw_nonfinite turns 1 after a backward whose weight
    gradient holds a NaN (a NaN in dY) and stays 1 over later clean ones."""
    from fp8_mixed_precision_reduce_gb300.linear import FP8Linear

    layer = FP8Linear(256, 128, bias=False)
    x = torch.randn(64, 256, device="cuda")
    dy = torch.randn(64, 128, device="cuda") * 1e-2
    layer(x).backward(dy)
    assert cuda_lib.fp8mp_check() == 0 and layer.dw_nonfinite.item() == 0
    bad = dy.clone()
    bad[3, 5] = float("nan")
    layer.zero_grad(set_to_none=True)
    layer(x).backward(bad)
    assert cuda_lib.fp8mp_check() == 0
    assert not torch.isfinite(layer.weight.grad).all() and layer.dw_nonfinite.item() == 1
    layer.zero_grad(set_to_none=True)
    layer(x).backward(dy)
    assert cuda_lib.fp8mp_check() == 0 and layer.dw_nonfinite.item() == 1


def test_fp8linear_rejects_unaligned_features(cuda_lib):
    from fp8_mixed_precision_reduce_gb300.linear import FP8Linear

    with pytest.raises(ValueError):
        FP8Linear(100, 64)
