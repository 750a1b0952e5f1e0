"""GPU parity of the three FP8 GEMMs (fwd, dgrad, wgrad) against the oracle's
fp64 reference, per element within |err| <= 2^-8 |ref| + 1e-5 sum|a b|, and
of the forward GEMM's output amax (bit-exact against a host reduction of the
stored output, within tolerance against the reference)."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, E5M2, dev, finite_codes, gemm_tolerance_check, np_view

pytestmark = pytest.mark.gpu

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(params=["single", "pair"])
def engine(request, monkeypatch):
    """Runs a test on both tile engines: single-SM 128x256 tiles and
    SM-pair 256x256 tiles (the library reads FP8MP_GEMM_ENGINE per call)."""
    monkeypatch.setenv("FP8MP_GEMM_ENGINE", request.param)
    return request.param


def sc(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


def fwd(fp8mp, A, B, sa, sb, bias=None, out="bf16", amax0=None):
    M, N = A.shape[0], B.shape[0]
    y = torch.empty((M, N), dtype=TORCH_DT[out], device="cuda")
    am = torch.tensor([amax0], dtype=torch.float32, device="cuda") if amax0 is not None else None
    fp8mp.fp8_linear_fwd(dev(A), dev(B), sc(sa), sc(sb), y, bias=bias, y_amax=am)
    assert fp8mp.fp8mp_check() == 0
    return y, am


# (M, N, K): single tile, several tiles, ragged in every dimension, tiny,
# the 768 layer, a long contraction
SHAPES = [(128, 256, 128), (256, 512, 256), (1040, 784, 784), (16, 16, 16), (1024, 768, 768),
          (128, 256, 16384), (384, 1280, 1152), (144, 272, 2064), (2304, 2560, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_fwd_random_codes(cuda_lib, orc, engine, M, N, K, out):
    rng = np.random.default_rng(M * 31 + N * 7 + K)
    A = finite_codes(rng, (M, K), E4M3)
    B = finite_codes(rng, (N, K), E4M3)
    sa, sb = 2.0 ** -6, 0.37
    y, _ = fwd(cuda_lib, A, B, sa, sb, out=out)
    ref, ab = orc.gemm_ref(A, E4M3, B, E4M3, float(np.float32(sa)), float(np.float32(sb)))
    gemm_tolerance_check(np_view(y.float()).astype(np.float64), ref, ab, f"fwd {M}x{N}x{K}")


@pytest.mark.parametrize("bias_dt", ["f32", "bf16"])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_fwd_bias_and_output_amax(cuda_lib, orc, engine, bias_dt, out):
    M, N, K = 1040, 784, 512
    rng = np.random.default_rng(5)
    A = finite_codes(rng, (M, K), E4M3)
    B = finite_codes(rng, (N, K), E4M3)
    bias = (torch.randn(N, generator=workloads.gen(9)) * 50).to(TORCH_DT[bias_dt])
    y, am = fwd(cuda_lib, A, B, 1e-3, 2e-3, bias=bias.cuda(), out=out, amax0=0.0)
    ref, ab = orc.gemm_ref(A, E4M3, B, E4M3, float(np.float32(1e-3)), float(np.float32(2e-3)),
                           bias=bias.double().numpy())
    yh = np_view(y.float()).astype(np.float64)
    gemm_tolerance_check(yh, ref, ab, "fwd+bias")
    # amax: exactly the max |.| of what was stored, and close to the reference's
    assert am.item() == np.abs(np_view(y.float())).max()
    assert abs(am.item() - np.abs(ref).max()) <= 2.0 ** -8 * np.abs(ref).max() + 1e-5 * ab.max()


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_fwd_output_amax_leaves_out_nan_and_keeps_inf(cuda_lib, engine, out):
    """NaN outputs (rows of x8 holding an E4M3 NaN code, and one 16-column
    group made NaN by a NaN code in w8) are left out of the output amax,
    which then equals the largest finite |y| stored; outputs that overflow
    to +-Inf (a row of +448 codes under a large scale product) make it Inf.
    Ragged tiles (1040 x 784), so masked rows and columns are in play."""
    M, N, K = 1040, 784, 512
    rng = np.random.default_rng(11)
    A = finite_codes(rng, (M, K), E4M3)
    B = finite_codes(rng, (N, K), E4M3)
    A[3, 5] = 0x7F     # row 3 of y is NaN
    A[1031, 0] = 0xFF  # a row in the last, ragged row tile
    B[40, 7] = 0x7F    # column 40 of y is NaN
    y, am = fwd(cuda_lib, A, B, 2.0 ** -6, 0.37, out=out, amax0=0.0)
    yh = np.abs(np_view(y.float()))
    assert np.isnan(yh[3]).all() and np.isnan(yh[:, 40]).all()
    assert np.isfinite(np.nanmax(yh)) and am.item() == np.nanmax(yh)
    # a row of the largest code pushes its outputs past the output type's range
    A[700, :] = 0x7E   # +448
    y, am = fwd(cuda_lib, A, B, 2.0 ** 60, 2.0 ** 60, out=out, amax0=0.0)
    yh = np.abs(np_view(y.float()))
    assert np.isinf(yh[700]).any()
    assert am.item() == np.inf and np.nanmax(yh) == np.inf


@pytest.mark.parametrize("dy_fmt", [E5M2, E4M3])
@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (1040, 784, 784), (1024, 768, 768)])
def test_dgrad_and_wgrad(cuda_lib, orc, engine, dy_fmt, M, N, K):
    rng = np.random.default_rng(M + 2 * N + 3 * K + dy_fmt)
    dy8 = finite_codes(rng, (M, N), dy_fmt)
    w8t = finite_codes(rng, (K, N), E4M3)
    x8t = finite_codes(rng, (K, M), E4M3)
    dy8t = np.ascontiguousarray(dy8.T)
    s_dy, s_w, s_x = 2.0 ** -12, 0.5, 0.125
    for out in ("bf16", "f32"):
        dx = torch.empty((M, K), dtype=TORCH_DT[out], device="cuda")
        cuda_lib.fp8_linear_dgrad(dev(dy8), dev(w8t), sc(s_dy), sc(s_w), dx, dy_fmt=dy_fmt)
        dw = torch.empty((N, K), dtype=TORCH_DT[out], device="cuda")
        cuda_lib.fp8_linear_wgrad(dev(dy8t), dev(x8t), sc(s_dy), sc(s_x), dw, dy_fmt=dy_fmt)
        assert cuda_lib.fp8mp_check() == 0
        ref, ab = orc.gemm_ref(dy8, dy_fmt, w8t, E4M3, s_dy, s_w)
        gemm_tolerance_check(np_view(dx.float()).astype(np.float64), ref, ab, "dgrad")
        ref, ab = orc.gemm_ref(dy8t, dy_fmt, x8t, E4M3, s_dy, s_x)
        gemm_tolerance_check(np_view(dw.float()).astype(np.float64), ref, ab, "wgrad")


# (M, N, K): wgrad contracts over M, dgrad over N, so these put either GEMM
# in the longer-contraction (first) slot, and include ragged tiles
BWD_SHAPES = [(256, 512, 256), (1040, 784, 784), (2048, 256, 1024), (256, 2048, 528), (16, 16, 16),
              (1024, 768, 768)]


@pytest.mark.parametrize("M,N,K", BWD_SHAPES)
@pytest.mark.parametrize("dy_fmt,dx_dt,dw_dt", [(E5M2, "bf16", "f32"), (E4M3, "f32", "bf16")])
def test_fused_backward_equals_separate_calls(cuda_lib, orc, engine, M, N, K, dy_fmt, dx_dt, dw_dt):
    """fp8_linear_bwd gives bitwise the results of fp8_linear_dgrad and
    fp8_linear_wgrad (same sums in the same order per element), and both are
    within the GEMM tolerance of the oracle."""
    rng = np.random.default_rng(3 * M + 5 * N + 7 * K + dy_fmt)
    dy8 = finite_codes(rng, (M, N), dy_fmt)
    dy8t = np.ascontiguousarray(dy8.T)
    w8t = finite_codes(rng, (K, N), E4M3)
    x8t = finite_codes(rng, (K, M), E4M3)
    s_dy, s_w, s_x = 2.0 ** -10, 0.75, 0.0625
    dx = torch.full((M, K), 5.0, dtype=TORCH_DT[dx_dt], device="cuda")
    dw = torch.full((N, K), 5.0, dtype=TORCH_DT[dw_dt], device="cuda")
    cuda_lib.fp8_linear_bwd(dev(dy8), dev(dy8t), dev(w8t), dev(x8t), sc(s_dy), sc(s_w), sc(s_x), dx, dw,
                            dy_fmt=dy_fmt)
    dx1, dw1 = torch.empty_like(dx), torch.empty_like(dw)
    cuda_lib.fp8_linear_dgrad(dev(dy8), dev(w8t), sc(s_dy), sc(s_w), dx1, dy_fmt=dy_fmt)
    cuda_lib.fp8_linear_wgrad(dev(dy8t), dev(x8t), sc(s_dy), sc(s_x), dw1, dy_fmt=dy_fmt)
    assert cuda_lib.fp8mp_check() == 0
    assert torch.equal(dx.view(torch.int16) if dx_dt == "bf16" else dx.view(torch.int32),
                       dx1.view(torch.int16) if dx_dt == "bf16" else dx1.view(torch.int32))
    assert torch.equal(dw.view(torch.int16) if dw_dt == "bf16" else dw.view(torch.int32),
                       dw1.view(torch.int16) if dw_dt == "bf16" else dw1.view(torch.int32))
    ref, ab = orc.gemm_ref(dy8, dy_fmt, w8t, E4M3, s_dy, s_w)
    gemm_tolerance_check(np_view(dx.float()).astype(np.float64), ref, ab, f"bwd dx {M}x{N}x{K}")
    ref, ab = orc.gemm_ref(dy8t, dy_fmt, x8t, E4M3, s_dy, s_x)
    gemm_tolerance_check(np_view(dw.float()).astype(np.float64), ref, ab, f"bwd dw {M}x{N}x{K}")


def test_fused_backward_empty_sides(cuda_lib, engine):
    """N == 0: dx is the empty sum (0) and dw is empty; M == 0: dw = 0."""
    one = sc(1.0)
    u8 = lambda r, c: torch.empty((r, c), dtype=torch.uint8, device="cuda")
    dx = torch.full((32, 48), 3.0, device="cuda")
    cuda_lib.fp8_linear_bwd(u8(32, 0), u8(0, 32), u8(48, 0), u8(48, 32), one, one, one, dx,
                            torch.empty((0, 48), device="cuda"))
    dw = torch.full((64, 48), 3.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.fp8_linear_bwd(u8(0, 64), u8(64, 0), u8(48, 64), u8(48, 0), one, one, one,
                            torch.empty((0, 48), device="cuda"), dw)
    assert cuda_lib.fp8mp_check() == 0
    assert (dx.cpu() == 0).all() and (dw.float().cpu() == 0).all()


@pytest.mark.parametrize("M,N,K", BWD_SHAPES + [(128, 256, 384), (4096, 1024, 2048)])
@pytest.mark.parametrize("dy_fmt,dx_dt,dw_dt", [(E5M2, "bf16", "f32"), (E4M3, "f32", "bf16")])
def test_backward_from_rowmajor_copies(cuda_lib, orc, engine, M, N, K, dy_fmt, dx_dt, dw_dt):
    """fp8_linear_bwd_rowmajor reads dY8, W8 and X8 as the forward has them
    (the tensor cores take W8, X8 and, for dW, dY8 along their rows): within
    the GEMM tolerance of the oracle, and equal to the transposed-copy path."""
    rng = np.random.default_rng(11 * M + 13 * N + 17 * K + dy_fmt)
    dy8 = finite_codes(rng, (M, N), dy_fmt)
    w8 = finite_codes(rng, (N, K), E4M3)
    x8 = finite_codes(rng, (M, K), E4M3)
    s_dy, s_w, s_x = 2.0 ** -9, 0.625, 0.125
    dx = torch.full((M, K), 5.0, dtype=TORCH_DT[dx_dt], device="cuda")
    dw = torch.full((N, K), 5.0, dtype=TORCH_DT[dw_dt], device="cuda")
    d_dy8, d_w8, d_x8 = dev(dy8), dev(w8), dev(x8)
    cuda_lib.fp8_linear_bwd_rowmajor(d_dy8, d_w8, d_x8, sc(s_dy), sc(s_w), sc(s_x), dx, dw, dy_fmt=dy_fmt)
    assert cuda_lib.fp8mp_check() == 0
    w8t, x8t, dy8t = (np.ascontiguousarray(a.T) for a in (w8, x8, dy8))
    ref, ab = orc.gemm_ref(dy8, dy_fmt, w8t, E4M3, s_dy, s_w)
    gemm_tolerance_check(np_view(dx.float()).astype(np.float64), ref, ab, f"rowmajor dx {M}x{N}x{K}")
    ref, ab = orc.gemm_ref(dy8t, dy_fmt, x8t, E4M3, s_dy, s_x)
    gemm_tolerance_check(np_view(dw.float()).astype(np.float64), ref, ab, f"rowmajor dw {M}x{N}x{K}")
    dx1, dw1 = torch.empty_like(dx), torch.empty_like(dw)
    cuda_lib.fp8_linear_bwd(d_dy8, dev(dy8t), dev(w8t), dev(x8t), sc(s_dy), sc(s_w), sc(s_x), dx1, dw1,
                            dy_fmt=dy_fmt)
    assert cuda_lib.fp8mp_check() == 0
    assert torch.equal(dx.float(), dx1.float()) and torch.equal(dw.float(), dw1.float())


@pytest.mark.parametrize("M,N,K", [(256, 2048, 528), (4096, 1024, 48), (2048, 512, 80)])
def test_ragged_edge_outputs_repeat_bitwise(cuda_lib, orc, engine, M, N, K):
    """Output widths that end inside a tile column (528 = 2 x 256 + 16, 48,
    80), so the epilogue stages and stores only some chunks of the last one:
    40 more launches of the fused backward give bitwise the first one's dX
    and dW, which is within the GEMM tolerance of the oracle. A staging box
    rewritten while its TMA store still read it would show as rows of
    another chunk's values (or zeros) in one of the repeats."""
    rng = np.random.default_rng(M + 3 * N + 5 * K)
    dy8 = finite_codes(rng, (M, N), E5M2)
    w8 = finite_codes(rng, (N, K), E4M3)
    x8 = finite_codes(rng, (M, K), E4M3)
    s_dy, s_w, s_x = 2.0 ** -9, 0.625, 0.125
    ops = (dev(dy8), dev(w8), dev(x8), sc(s_dy), sc(s_w), sc(s_x))
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    cuda_lib.fp8_linear_bwd_rowmajor(*ops, dx, dw, dy_fmt=E5M2)
    assert cuda_lib.fp8mp_check() == 0
    w8t, x8t, dy8t = (np.ascontiguousarray(a.T) for a in (w8, x8, dy8))
    ref, ab = orc.gemm_ref(dy8, E5M2, w8t, E4M3, s_dy, s_w)
    gemm_tolerance_check(np_view(dx.float()).astype(np.float64), ref, ab, f"ragged dx {M}x{N}x{K}")
    ref, ab = orc.gemm_ref(dy8t, E5M2, x8t, E4M3, s_dy, s_x)
    gemm_tolerance_check(np_view(dw).astype(np.float64), ref, ab, f"ragged dw {M}x{N}x{K}")
    dx0, dw0 = dx.clone(), dw.clone()
    for i in range(40):
        dx.fill_(7.0)
        dw.fill_(7.0)
        cuda_lib.fp8_linear_bwd_rowmajor(*ops, dx, dw, dy_fmt=E5M2)
        assert torch.equal(dx, dx0) and torch.equal(dw, dw0), f"repeat {i + 1} differs from the first launch"
    assert cuda_lib.fp8mp_check() == 0


def test_backward_from_rowmajor_copies_one_side(cuda_lib, orc, engine):
    """dx or dw None: only the other gradient is computed (and written)."""
    M, N, K = 272, 400, 528
    rng = np.random.default_rng(99)
    dy8 = finite_codes(rng, (M, N), E5M2)
    w8 = finite_codes(rng, (N, K), E4M3)
    x8 = finite_codes(rng, (M, K), E4M3)
    dx = torch.empty((M, K), dtype=torch.float32, device="cuda")
    cuda_lib.fp8_linear_bwd_rowmajor(dev(dy8), dev(w8), None, sc(1.0), sc(1.0), None, dx, None)
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    cuda_lib.fp8_linear_bwd_rowmajor(dev(dy8), None, dev(x8), sc(1.0), None, sc(1.0), None, dw)
    assert cuda_lib.fp8mp_check() == 0
    ref, ab = orc.gemm_ref(dy8, E5M2, np.ascontiguousarray(w8.T), E4M3, 1.0, 1.0)
    gemm_tolerance_check(np_view(dx).astype(np.float64), ref, ab, "rowmajor dx only")
    ref, ab = orc.gemm_ref(np.ascontiguousarray(dy8.T), E5M2, np.ascontiguousarray(x8.T), E4M3, 1.0, 1.0)
    gemm_tolerance_check(np_view(dw).astype(np.float64), ref, ab, "rowmajor dw only")


@pytest.mark.parametrize("dw_dt", ["bf16", "f32"])
def test_dw_nonfinite_flag_matches_a_scan_of_the_stored_dw(cuda_lib, orc, engine, dw_dt):
    """fp8_linear_bwd_rowmajor's dw_nonfinite is 1 exactly when a stored dW
    element is Inf or NaN: finite codes at ordinary scales; scales around the
    output type's overflow (for bf16 a finite fp32 value can round to Inf);
    and E5M2 Inf / NaN codes in dY8."""
    M, N, K = 272, 400, 528
    rng = np.random.default_rng(1234)
    dy8 = finite_codes(rng, (M, N), E5M2)
    x8 = finite_codes(rng, (M, K), E4M3)
    ref, _ = orc.gemm_ref(np.ascontiguousarray(dy8.T), E5M2, np.ascontiguousarray(x8.T), E4M3, 1.0, 1.0)
    big = float(np.abs(ref).max())
    top = float(torch.finfo(TORCH_DT[dw_dt]).max)
    dw = torch.empty((N, K), dtype=TORCH_DT[dw_dt], device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    seen = []
    for s_dy in (1.0, 0.5 * top / big, 0.999 * top / big, 1.001 * top / big, 4.0 * top / big):
        s_dy = float(np.float32(s_dy))
        if not np.isfinite(s_dy):
            continue
        flag.zero_()
        cuda_lib.fp8_linear_bwd_rowmajor(dev(dy8), None, dev(x8), sc(s_dy), None, sc(1.0), None, dw,
                                         dw_nonfinite=flag)
        assert cuda_lib.fp8mp_check() == 0
        expect = int(not torch.isfinite(dw.float()).all().item())
        assert flag.item() == expect, (s_dy, expect)
        seen.append(expect)
    assert seen[0] == 0 and seen[-1] == 1
    # Inf and NaN codes of E5M2 in the output gradient
    for code in (0x7C, 0xFC, 0x7E):
        bad = dy8.copy()
        bad[rng.integers(0, M), rng.integers(0, N)] = code
        flag.zero_()
        cuda_lib.fp8_linear_bwd_rowmajor(dev(bad), None, dev(x8), sc(1.0), None, sc(1.0), None, dw,
                                         dw_nonfinite=flag)
        assert cuda_lib.fp8mp_check() == 0
        assert not torch.isfinite(dw.float()).all().item()
        assert flag.item() == 1, hex(code)
    # the flag accumulates (OR) over calls and is left alone by clean ones
    cuda_lib.fp8_linear_bwd_rowmajor(dev(dy8), None, dev(x8), sc(1.0), None, sc(1.0), None, dw, dw_nonfinite=flag)
    assert cuda_lib.fp8mp_check() == 0 and flag.item() == 1


def test_long_contraction_e5m2_wgrad(cuda_lib, orc, engine):
    """wgrad contracts over all tokens: 16384 here (the MLP workload's M)."""
    N, K, M = 256, 384, 16384
    rng = np.random.default_rng(77)
    dy8t = finite_codes(rng, (N, M), E5M2)
    x8t = finite_codes(rng, (K, M), E4M3)
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    cuda_lib.fp8_linear_wgrad(dev(dy8t), dev(x8t), sc(1.0), sc(1.0), dw, dy_fmt=E5M2)
    assert cuda_lib.fp8mp_check() == 0
    ref, ab = orc.gemm_ref(dy8t, E5M2, x8t, E4M3, 1.0, 1.0)
    gemm_tolerance_check(np_view(dw).astype(np.float64), ref, ab, "wgrad K=16384")


def test_empty_contraction_and_empty_output(cuda_lib, engine):
    bias = torch.arange(32, dtype=torch.float32, device="cuda")
    y = torch.full((16, 32), 7.0, dtype=torch.float32, device="cuda")
    am = torch.zeros(1, device="cuda")
    e = torch.empty((16, 0), dtype=torch.uint8, device="cuda")
    w = torch.empty((32, 0), dtype=torch.uint8, device="cuda")
    cuda_lib.fp8_linear_fwd(e, w, sc(1.0), sc(1.0), y, bias=bias, y_amax=am)
    assert cuda_lib.fp8mp_check() == 0
    assert (y.cpu() == bias.cpu()[None, :]).all() and am.item() == 31.0
    dw = torch.full((32, 48), 3.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.fp8_linear_wgrad(torch.empty((32, 0), dtype=torch.uint8, device="cuda"),
                              torch.empty((48, 0), dtype=torch.uint8, device="cuda"), sc(1.0), sc(1.0), dw)
    assert cuda_lib.fp8mp_check() == 0
    assert (dw.float().cpu() == 0).all()


def test_metric_shape_full_size_sampled(cuda_lib, orc):
    """M = 8192, N = K = 4096 (the proj linear of the transformer workload),
    realistic codes cast by the oracle, every output of 40 sampled rows and of
    one whole 128 x 256 tile checked, for fwd, dgrad and wgrad."""
    tb = workloads.transformer_block(device="cuda")
    M, K, N = 8192, 4096, 4096
    xn, wn, dyn = np_view(tb.x), np_view(tb.w_proj), np_view(tb.dy_proj)
    metas = {}
    codes = {}
    for name, arr, fmt in (("x", xn, E4M3), ("w", wn, E4M3), ("dy", dyn, E5M2)):
        m = orc.Meta(1024)
        m.record_amax(orc.amax(arr))
        orc.scale_update(m, fmt, 1, 0)
        metas[name] = m
        codes[name] = orc.cast(arr, float(m.scale[0]), fmt)
    sinv = {k: float(m.scale_inv[0]) for k, m in metas.items()}
    rng = np.random.default_rng(8192)
    rows = np.unique(np.concatenate([rng.integers(0, M, 40), np.arange(128 * 37, 128 * 38)])).astype(np.int64)

    y, _ = fwd(cuda_lib, codes["x"], codes["w"], sinv["x"], sinv["w"], out="bf16")
    ref, ab = orc.gemm_ref(codes["x"], E4M3, codes["w"], E4M3, sinv["x"], sinv["w"], rows=rows)
    gemm_tolerance_check(np_view(y.float())[rows].astype(np.float64), ref, ab, "fwd 8192x4096x4096")
    del y

    w8t = orc.transpose_u8(codes["w"])
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    cuda_lib.fp8_linear_dgrad(dev(codes["dy"]), dev(w8t), sc(sinv["dy"]), sc(sinv["w"]), dx)
    assert cuda_lib.fp8mp_check() == 0
    ref, ab = orc.gemm_ref(codes["dy"], E5M2, w8t, E4M3, sinv["dy"], sinv["w"], rows=rows)
    gemm_tolerance_check(np_view(dx.float())[rows].astype(np.float64), ref, ab, "dgrad 8192x4096x4096")
    del dx

    dy8t = orc.transpose_u8(codes["dy"])
    x8t = orc.transpose_u8(codes["x"])
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    cuda_lib.fp8_linear_wgrad(dev(dy8t), dev(x8t), sc(sinv["dy"]), sc(sinv["x"]), dw)
    assert cuda_lib.fp8mp_check() == 0
    wrows = rows[rows < N]
    ref, ab = orc.gemm_ref(dy8t, E5M2, x8t, E4M3, sinv["dy"], sinv["x"], rows=wrows)
    gemm_tolerance_check(np_view(dw.float())[wrows].astype(np.float64), ref, ab, "wgrad 8192x4096x4096")

    # the fused backward launch (the bench step's) gives the same bits
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dx1 = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw1 = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    d8, d8t, w8t_d, x8t_d = dev(codes["dy"]), dev(dy8t), dev(w8t), dev(x8t)
    cuda_lib.fp8_linear_bwd(d8, d8t, w8t_d, x8t_d, sc(sinv["dy"]), sc(sinv["w"]), sc(sinv["x"]), dx1, dw1)
    cuda_lib.fp8_linear_dgrad(d8, w8t_d, sc(sinv["dy"]), sc(sinv["w"]), dx)
    assert cuda_lib.fp8mp_check() == 0
    assert torch.equal(dx1.view(torch.int16), dx.view(torch.int16))
    assert torch.equal(dw1.view(torch.int16), dw.view(torch.int16))
