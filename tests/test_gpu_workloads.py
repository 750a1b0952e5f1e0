"""Full-size workloads on the GPU against the oracle.

* Transformer QKV linear (4096 -> 12288 at M = 8192 tokens, bf16 activations
  with 0.1 % outliers, DelayedScaling L = 1024, most_recent): every FP8 code
  of x, W, dY (and their transposes) bit-exact; fwd, dgrad and wgrad on sampled
  rows within the GEMM tolerance; metas bit-exact after the update.
* MLP up/down (4096 -> 14336 -> 4096 at M = 16384), HYBRID, L = 16, max, 16
  steps of fwd + dgrad + wgrad + update with a new output gradient each step:
  every step's metas (history, scale, scale_inv) bit-exact; each step's output
  amax equal to the max |.| of the stored output; every step's FP8 codes (and
  transposes) bit-exact; every step 16 sampled rows of each GEMM output (8 of
  the weight gradients) within the GEMM tolerance, and on the first and last
  step 128 sampled rows plus one whole 128-row block (full 128 x 256 tiles).
"""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, E5M2, assert_same_bits, gemm_tolerance_check, np_view

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

U8 = torch.uint8


def cast_both(fp8mp, orc, x_dev, x_np, fmt, dm, om, check_codes=True):
    """Casts on the GPU (with transpose and amax) and checks against the oracle."""
    rows, cols = x_dev.shape
    q = torch.empty((rows, cols), dtype=U8, device="cuda")
    qt = torch.empty((cols, rows), dtype=U8, device="cuda")
    fp8mp.fp8_quantize(x_dev, fmt, dm.scale, q, qt, dm.cur_amax)
    codes = None
    if check_codes:
        codes = orc.cast(x_np, float(om.scale[0]), fmt)
        assert_same_bits(q.cpu().numpy(), codes, "codes")
        assert_same_bits(qt.cpu().numpy(), orc.transpose_u8(codes), "transposed codes")
    om.record_amax(orc.amax(x_np))
    return q, qt, codes


def meta_equal(dm, om, what):
    assert_same_bits(np_view(dm.amax_history), om.hist, what + " history")
    assert_same_bits(np_view(dm.scale), om.scale, what + " scale")
    assert_same_bits(np_view(dm.scale_inv), om.scale_inv, what + " scale_inv")
    assert_same_bits(np_view(dm.cur_amax), om.cur_amax, what + " cur_amax")


def sample_rows(n, rng, block=128):
    r = np.concatenate([rng.integers(0, n, 24), np.arange(block * 3, block * 4)])
    return np.unique(r).astype(np.int64)


def test_transformer_qkv_full_size(cuda_lib, orc):
    f = cuda_lib
    tb = workloads.transformer_block(device="cuda")
    x, w, dy = tb.x, tb.w_qkv, tb.dy_qkv
    M, K = x.shape
    N = w.shape[0]
    xn, wn, dyn = np_view(x), np_view(w), np_view(dy)
    names = {"x": E4M3, "w": E4M3, "y": E4M3, "dy": E5M2}
    dm = {k: f.Meta(1024, v) for k, v in names.items()}
    om = {k: orc.Meta(1024) for k in names}
    # one update from the tensors' own amaxes, so the step runs at real scales
    for k, arr in (("x", xn), ("w", wn), ("dy", dyn)):
        a = orc.amax(arr)
        om[k].record_amax(a)
        dm[k].cur_amax.fill_(float(a))
    f.delayed_scaling_update(list(dm.values()), f.AMAX_MOST_RECENT, 0)
    for k, v in names.items():
        orc.scale_update(om[k], v, orc.AMAX_MOST_RECENT, 0)

    X8, X8t, qx = cast_both(f, orc, x, xn, E4M3, dm["x"], om["x"])
    W8, W8t, qw = cast_both(f, orc, w, wn, E4M3, dm["w"], om["w"])
    D8, D8t, qd = cast_both(f, orc, dy, dyn, E5M2, dm["dy"], om["dy"])
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    f.fp8_linear_fwd(X8, W8, dm["x"].scale_inv, dm["w"].scale_inv, y, y_amax=dm["y"].cur_amax)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    f.fp8_linear_dgrad(D8, W8t, dm["dy"].scale_inv, dm["w"].scale_inv, dx)
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    f.fp8_linear_wgrad(D8t, X8t, dm["dy"].scale_inv, dm["x"].scale_inv, dw)
    assert f.fp8mp_check() == 0

    sx, sw, sd = (float(om[k].scale_inv[0]) for k in ("x", "w", "dy"))
    rng = np.random.default_rng(12288)
    rows = sample_rows(M, rng)
    yh = np_view(y.float())
    ref, ab = orc.gemm_ref(qx, E4M3, qw, E4M3, sx, sw, rows=rows)
    gemm_tolerance_check(yh[rows].astype(np.float64), ref, ab, "QKV fwd")
    assert dm["y"].cur_amax.item() == np.abs(yh).max()
    ref, ab = orc.gemm_ref(qd, E5M2, orc.transpose_u8(qw), E4M3, sd, sw, rows=rows)
    gemm_tolerance_check(np_view(dx.float())[rows].astype(np.float64), ref, ab, "QKV dgrad")
    wrows = sample_rows(N, rng)
    ref, ab = orc.gemm_ref(orc.transpose_u8(qd), E5M2, orc.transpose_u8(qx), E4M3, sd, sx, rows=wrows)
    gemm_tolerance_check(np_view(dw.float())[wrows].astype(np.float64), ref, ab, "QKV wgrad")

    om["y"].record_amax(np.float32(np.abs(yh).max()))
    f.delayed_scaling_update(list(dm.values()), f.AMAX_MOST_RECENT, 0)
    for k, v in names.items():
        orc.scale_update(om[k], v, orc.AMAX_MOST_RECENT, 0)
    torch.cuda.synchronize()
    for k in names:
        meta_equal(dm[k], om[k], k)


def test_mlp_16_steps(cuda_lib, orc):
    f = cuda_lib
    wl = workloads.mlp(device="cuda")
    M, D = wl.x_up.shape
    H = wl.w_up.shape[0]
    host = {"x_up": np_view(wl.x_up), "x_down": np_view(wl.x_down), "w_up": np_view(wl.w_up),
            "w_down": np_view(wl.w_down)}
    fmt = {"x_up": E4M3, "w_up": E4M3, "h": E4M3, "dh": E5M2,
           "x_down": E4M3, "w_down": E4M3, "y": E4M3, "dy": E5M2}
    dm = {k: f.Meta(16, v) for k, v in fmt.items()}
    om = {k: orc.Meta(16) for k in fmt}
    h = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, D), dtype=torch.bfloat16, device="cuda")
    dxu = torch.empty((M, D), dtype=torch.bfloat16, device="cuda")
    dwu = torch.empty((H, D), dtype=torch.bfloat16, device="cuda")
    dxd = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    dwd = torch.empty((D, H), dtype=torch.bfloat16, device="cuda")
    rng = np.random.default_rng(16384)
    for step in range(16):
        full = step in (0, 15)
        dy = workloads.mlp_grad(step, 1, M, D, device="cuda")     # gradient of the down output
        dh = workloads.mlp_grad(step, 0, M, H, device="cuda")     # gradient of the up output
        dyn, dhn = np_view(dy), np_view(dh)
        XU, XUt, qxu = cast_both(f, orc, wl.x_up, host["x_up"], E4M3, dm["x_up"], om["x_up"])
        WU, WUt, qwu = cast_both(f, orc, wl.w_up, host["w_up"], E4M3, dm["w_up"], om["w_up"])
        XD, XDt, qxd = cast_both(f, orc, wl.x_down, host["x_down"], E4M3, dm["x_down"], om["x_down"])
        WD, WDt, qwd = cast_both(f, orc, wl.w_down, host["w_down"], E4M3, dm["w_down"], om["w_down"])
        DY, DYt, qdy = cast_both(f, orc, dy, dyn, E5M2, dm["dy"], om["dy"])
        DH, DHt, qdh = cast_both(f, orc, dh, dhn, E5M2, dm["dh"], om["dh"])
        sinv = {k: dm[k].scale_inv for k in fmt}
        f.fp8_linear_fwd(XU, WU, sinv["x_up"], sinv["w_up"], h, y_amax=dm["h"].cur_amax)
        f.fp8_linear_fwd(XD, WD, sinv["x_down"], sinv["w_down"], y, y_amax=dm["y"].cur_amax)
        # the down projection's backward from transposed copies, the up
        # projection's from the row-major copies (both fused launches)
        f.fp8_linear_bwd(DY, DYt, WDt, XDt, sinv["dy"], sinv["w_down"], sinv["x_down"], dxd, dwd)
        f.fp8_linear_bwd_rowmajor(DH, WU, XU, sinv["dh"], sinv["w_up"], sinv["x_up"], dxu, dwu)
        assert f.fp8mp_check() == 0
        hh, yy = np_view(h.float()), np_view(y.float())
        # per-step output amax: exactly the max |.| of what was stored
        assert dm["h"].cur_amax.item() == np.abs(hh).max(), step
        assert dm["y"].cur_amax.item() == np.abs(yy).max(), step
        om["h"].record_amax(np.float32(np.abs(hh).max()))
        om["y"].record_amax(np.float32(np.abs(yy).max()))
        # every step: 16 sampled rows of every GEMM output (8 of the weight
        # gradients); steps 0 and 15: 128 sampled rows plus one whole 128-row
        # block (full 128 x 256 tiles) of each
        s = {k: float(om[k].scale_inv[0]) for k in fmt}
        nr, nw = (128, 128) if full else (16, 8)

        def rows_of(n, k):
            r = rng.integers(0, n, k)
            if full:
                blk = int(rng.integers(0, n // 128))
                r = np.concatenate([r, np.arange(128 * blk, 128 * blk + 128)])
            return np.unique(r).astype(np.int64)

        rows = rows_of(M, nr)
        ref, ab = orc.gemm_ref(qxu, E4M3, qwu, E4M3, s["x_up"], s["w_up"], rows=rows)
        gemm_tolerance_check(hh[rows].astype(np.float64), ref, ab, f"step {step} up fwd")
        ref, ab = orc.gemm_ref(qxd, E4M3, qwd, E4M3, s["x_down"], s["w_down"], rows=rows)
        gemm_tolerance_check(yy[rows].astype(np.float64), ref, ab, f"step {step} down fwd")
        ref, ab = orc.gemm_ref(qdy, E5M2, orc.transpose_u8(qwd), E4M3, s["dy"], s["w_down"], rows=rows)
        gemm_tolerance_check(np_view(dxd.float())[rows].astype(np.float64), ref, ab, f"step {step} down dgrad")
        ref, ab = orc.gemm_ref(qdh, E5M2, orc.transpose_u8(qwu), E4M3, s["dh"], s["w_up"], rows=rows)
        gemm_tolerance_check(np_view(dxu.float())[rows].astype(np.float64), ref, ab, f"step {step} up dgrad")
        wr = rows_of(D, nw)
        ref, ab = orc.gemm_ref(orc.transpose_u8(qdy), E5M2, orc.transpose_u8(qxd), E4M3, s["dy"], s["x_down"],
                               rows=wr)
        gemm_tolerance_check(np_view(dwd.float())[wr].astype(np.float64), ref, ab, f"step {step} down wgrad")
        wr = rows_of(H, nw)
        ref, ab = orc.gemm_ref(orc.transpose_u8(qdh), E5M2, orc.transpose_u8(qxu), E4M3, s["dh"], s["x_up"],
                               rows=wr)
        gemm_tolerance_check(np_view(dwu.float())[wr].astype(np.float64), ref, ab, f"step {step} up wgrad")
        f.delayed_scaling_update([dm[k] for k in fmt], f.AMAX_MAX, 0)
        for k, v in fmt.items():
            orc.scale_update(om[k], v, orc.AMAX_MAX, 0)
        torch.cuda.synchronize()
        for k in fmt:
            meta_equal(dm[k], om[k], f"step {step} {k}")
        del dy, dh, XU, XUt, WU, WUt, XD, XDt, WD, WDt, DY, DYt, DH, DHt
