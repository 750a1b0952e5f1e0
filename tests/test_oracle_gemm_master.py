"""Pins of the oracle's fp64 GEMM reference and its master step (CPU only)."""

from fractions import Fraction

import numpy as np
import pytest
import torch

E4M3, E5M2 = 0, 1
TORCH_FMT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def torch_decode(codes, fmt):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(TORCH_FMT[fmt]).to(torch.float64).numpy()


def finite_codes(rng, shape, fmt):
    """Random codes excluding NaN/Inf patterns."""
    c = rng.integers(0, 256, shape, dtype=np.uint8)
    if fmt == E4M3:
        c[(c & 0x7F) == 0x7F] = 0x3F
    else:
        c[(c & 0x7C) == 0x7C] = 0x3B
    return c


# ------------------------------------------------------------------ GEMM


@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E5M2, E4M3)])
def test_gemm_exact_rational_tiny(orc, fa, fb):
    """Exact rational sums on a 16 x 16 x 32 problem, scales and bias included."""
    rng = np.random.default_rng(2)
    A = finite_codes(rng, (16, 32), fa)
    B = finite_codes(rng, (16, 32), fb)
    sa, sb = 0.125, 3.0
    bias = rng.standard_normal(16)
    ref, ab = orc.gemm_ref(A, fa, B, fb, sa, sb, bias)
    Ad, Bd = torch_decode(A, fa), torch_decode(B, fb)
    for i in range(16):
        for j in range(16):
            s = sum(Fraction(Ad[i, k]) * Fraction(Bd[j, k]) for k in range(32))
            exp = s * Fraction(sa) * Fraction(sb) + Fraction(bias[j])
            assert Fraction(ref[i, j]) == exp or abs(float(Fraction(ref[i, j]) - exp)) <= 1e-15 * abs(float(exp))
            sabs = sum(abs(Fraction(Ad[i, k]) * Fraction(Bd[j, k])) for k in range(32))
            assert ab[i, j] == float(sabs * Fraction(sa) * Fraction(sb))


def test_gemm_e4m3_sum_is_exact_at_long_k(orc):
    """E4M3 x E4M3 products span 2^-18..2^18, so an fp64 sum over K = 4096 is exact."""
    rng = np.random.default_rng(4)
    A = finite_codes(rng, (2, 4096), E4M3)
    B = finite_codes(rng, (3, 4096), E4M3)
    ref, _ = orc.gemm_ref(A, E4M3, B, E4M3, 1.0, 1.0)
    Ad, Bd = torch_decode(A, E4M3), torch_decode(B, E4M3)
    for i in range(2):
        for j in range(3):
            exact = sum(Fraction(Ad[i, k]) * Fraction(Bd[j, k]) for k in range(4096))
            assert Fraction(ref[i, j]) == exact


@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E5M2, E4M3)])
def test_gemm_vs_library_matmul(orc, fa, fb):
    """A library matmul of the torch-decoded operands (layout A @ B^T)."""
    rng = np.random.default_rng(6)
    A = finite_codes(rng, (64, 96), fa)
    B = finite_codes(rng, (48, 96), fb)
    ref, _ = orc.gemm_ref(A, fa, B, fb, 0.5, 0.25)
    lib = (torch_decode(A, fa) @ torch_decode(B, fb).T) * 0.125
    np.testing.assert_allclose(ref, lib, rtol=1e-12, atol=1e-12)
    # a transposed operand would not match
    assert not np.allclose(ref[:48, :48], (torch_decode(A, fa)[:48] @ torch_decode(B, fb).T).T * 0.125)


def test_gemm_row_selection_and_bias(orc):
    rng = np.random.default_rng(8)
    A = finite_codes(rng, (40, 32), E4M3)
    B = finite_codes(rng, (24, 32), E4M3)
    bias = rng.standard_normal(24)
    full, _ = orc.gemm_ref(A, E4M3, B, E4M3, 1.0, 2.0, bias)
    rows = np.array([39, 0, 17], dtype=np.int64)
    part, _ = orc.gemm_ref(A, E4M3, B, E4M3, 1.0, 2.0, bias, rows=rows)
    assert (part == full[rows]).all()
    nobias, _ = orc.gemm_ref(A, E4M3, B, E4M3, 1.0, 2.0)
    np.testing.assert_allclose(full - nobias, np.broadcast_to(bias, full.shape), rtol=0,
                               atol=4e-16 * np.abs(nobias).max())


def test_gemm_empty_contraction(orc):
    A = np.zeros((4, 0), dtype=np.uint8)
    B = np.zeros((5, 0), dtype=np.uint8)
    bias = np.arange(5, dtype=np.float64)
    ref, ab = orc.gemm_ref(A, E4M3, B, E4M3, 1.0, 1.0, bias)
    assert (ref == bias).all() and (ab == 0).all()


# ----------------------------------------------------------- master step


def bf16_bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def test_master_step_hand_example(orc):
    """Two elements worked by hand. S = 2^16, lr = 2^-4, mu = 0.5:
    g = 2^15 -> u = 0.5, v = 0.5*0.25 + 0.5 = 0.625, w = 1 - 0.625/16 = 0.9609375;
    g = -2^16 -> u = -1, v = 0.5*0 - 1 = -1, w = -2 + 1/16 = -1.9375.
    w8 at scale 2: 1.921875 -> E4M3 1.875 (0x3F); -3.875 -> -4.0 (0xC8)."""
    g = bf16_bits([2.0 ** 15, -(2.0 ** 16)])
    w = np.array([1.0, -2.0], dtype=np.float32)
    v = np.array([0.25, 0.0], dtype=np.float32)
    w8 = np.zeros(2, dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    st = orc.LossScaleState(2.0 ** 16, growth=5)
    orc.master_step(g, w, v, w8, 2.0, am, st, lr=2.0 ** -4, mu=0.5)
    assert list(v) == [0.625, -1.0]
    assert list(w) == [0.9609375, -1.9375]
    assert list(w8) == [0x3F, 0xC8]
    assert am[0] == 1.9375
    assert st.found_inf[0] == 0 and st.growth[0] == 6 and st.S[0] == 2.0 ** 16


def test_master_step_overflow_skips_and_backs_off(orc):
    rng = np.random.default_rng(3)
    n = 10_000
    g = bf16_bits(rng.standard_normal(n) * 1e-5 * 2 ** 16)
    g[123] = 0x7F80  # +Inf
    g[4567] = 0xFFC1  # a NaN
    w = rng.standard_normal(n).astype(np.float32)
    v = rng.standard_normal(n).astype(np.float32)
    w8 = rng.integers(0, 256, n, dtype=np.uint8)
    w0, v0, w80 = w.copy(), v.copy(), w8.copy()
    am = np.array([0.5], dtype=np.float32)
    st = orc.LossScaleState(2.0 ** 16, growth=1999)
    orc.master_step(g, w, v, w8, 3.0, am, st, lr=1e-4, mu=0.9)
    assert st.found_inf[0] == 1 and st.S[0] == 2.0 ** 15 and st.growth[0] == 0
    assert (w.view(np.uint32) == w0.view(np.uint32)).all()
    assert (v.view(np.uint32) == v0.view(np.uint32)).all()
    assert (w8 == w80).all() and am[0] == 0.5


@pytest.mark.parametrize("bad", [0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x7F81])
def test_master_step_each_nonfinite_kind_alone_skips(orc, bad):
    """+Inf, -Inf and NaNs of either sign each trigger the skip on their own."""
    n = 256
    g = bf16_bits(np.full(n, 3.0))
    g[n // 3] = bad
    w = np.ones(n, dtype=np.float32)
    v = np.zeros(n, dtype=np.float32)
    w8 = np.zeros(n, dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    st = orc.LossScaleState(8.0, growth=3)
    orc.master_step(g, w, v, w8, 1.0, am, st, lr=0.1, mu=0.9)
    assert st.found_inf[0] == 1 and st.S[0] == 4.0 and st.growth[0] == 0
    assert (w == 1.0).all() and (v == 0.0).all() and (w8 == 0).all()


def test_master_step_growth_after_interval(orc):
    n = 64
    g = bf16_bits(np.ones(n))
    w = np.zeros(n, dtype=np.float32)
    v = np.zeros(n, dtype=np.float32)
    w8 = np.zeros(n, dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    st = orc.LossScaleState(4.0, growth=0)
    for i in range(3):
        orc.master_step(g, w, v, w8, 1.0, am, st, lr=0.0, mu=0.0, growth_interval=3)
    assert st.S[0] == 8.0 and st.growth[0] == 0


def test_master_step_vs_torch_sgd_momentum(orc):
    """torch.optim.SGD(momentum=mu) after unscaling: v = mu*v + g; w -= lr*v.
    torch rounds the multiply and the add separately, the oracle fuses them,
    so the two may differ by a rounding of each step (a few ulp)."""
    rng = np.random.default_rng(12)
    n = 50_000
    S = 2.0 ** 16
    gt = torch.from_numpy((rng.standard_normal(n) * 1e-5 * S).astype(np.float32)).to(torch.bfloat16)
    g = gt.view(torch.int16).numpy().view(np.uint16).copy()
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    v = np.zeros(n, dtype=np.float32)
    w8 = np.zeros(n, dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    st = orc.LossScaleState(S)
    p = torch.nn.Parameter(torch.from_numpy(w.copy()))
    opt = torch.optim.SGD([p], lr=1e-4, momentum=0.9)
    for _ in range(3):
        orc.master_step(g, w, v, w8, 1.0, am, st, lr=1e-4, mu=0.9)
        p.grad = gt.float() / S
        opt.step()
    np.testing.assert_allclose(w, p.detach().numpy(), rtol=0, atol=4e-9)
    buf = opt.state[p]["momentum_buffer"].numpy()
    np.testing.assert_allclose(v, buf, rtol=1e-6, atol=1e-12)


def test_master_step_unscale_exact_for_power_of_two(orc):
    """With S = 2^16 the unscale is exact: one step from v = 0 with mu = 0 and
    lr = 1 gives w = w0 - g / S exactly (the fused multiply-add rounds once)."""
    rng = np.random.default_rng(13)
    n = 4096
    gt = torch.from_numpy(rng.standard_normal(n).astype(np.float32) * 100).to(torch.bfloat16)
    g = gt.view(torch.int16).numpy().view(np.uint16).copy()
    w = np.zeros(n, dtype=np.float32)
    v = np.zeros(n, dtype=np.float32)
    w8 = np.zeros(n, dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    st = orc.LossScaleState(2.0 ** 16)
    orc.master_step(g, w, v, w8, 1.0, am, st, lr=1.0, mu=0.0)
    assert (v == gt.float().numpy() / 2 ** 16).all()
    assert (w == -v).all()
    # the FP8 copy is the E4M3 cast of the new master weights at scale_w
    assert (w8 == orc.cast(w, 1.0, E4M3)).all()


# ------------------------------------------------------------- Adam step


def test_adam_first_step_is_sign_descent(orc):
    """At t = 1 the bias corrections cancel: mh = u, vh = u^2, so with a tiny
    eps each weight moves by lr * sign(u) (worked from the update rule)."""
    g = bf16_bits([2.0 ** 16, -(2.0 ** 15), 3.0 * 2 ** 16])
    w = np.array([1.0, 1.0, -0.5], dtype=np.float32)
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    w8 = np.zeros(3, np.uint8)
    am = np.zeros(1, np.float32)
    st = orc.LossScaleState(2.0 ** 16)
    ad = orc.AdamState()
    orc.adam_step(g, w, m, v, w8, 1.0, am, st, ad, lr=2.0 ** -7, eps=1e-30)
    np.testing.assert_allclose(w, [1.0 - 2 ** -7, 1.0 + 2 ** -7, -0.5 - 2 ** -7], rtol=0, atol=2e-7)
    np.testing.assert_allclose(m, np.float32(0.1) * np.array([1.0, -0.5, 3.0], np.float32), rtol=1e-6)
    assert ad.b1p[0] == np.float32(0.9) and ad.b2p[0] == np.float32(0.999)
    assert st.growth[0] == 1


def test_adam_vs_torch_optim_adam(orc):
    """torch.optim.Adam (the optimizer the PyTorch-native FP8 page uses) on the
    unscaled gradients: same trajectory within a few fp32 roundings. beta2 =
    1 - 2^-10 is exact in fp32, so both sides use the same 1 - beta2 (with
    0.999 the fp32 complement 1 - fl32(0.999) differs from fl32(0.001) by
    1.3e-5 relative, which would show in every v)."""
    rng = np.random.default_rng(41)
    n, S = 20_000, 2.0 ** 16
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    w8 = np.zeros(n, np.uint8)
    am = np.zeros(1, np.float32)
    st = orc.LossScaleState(S)
    ad = orc.AdamState()
    p = torch.nn.Parameter(torch.from_numpy(w.copy()))
    b2 = 1.0 - 2.0 ** -10
    opt = torch.optim.Adam([p], lr=1e-3, betas=(0.9, b2), eps=1e-8)
    for step in range(4):
        gt = torch.from_numpy((rng.standard_normal(n) * 1e-4 * S).astype(np.float32)).to(torch.bfloat16)
        g = gt.view(torch.int16).numpy().view(np.uint16).copy()
        orc.adam_step(g, w, m, v, w8, 1.0, am, st, ad, lr=1e-3, beta2=b2)
        p.grad = gt.float() / S
        opt.step()
    np.testing.assert_allclose(w, p.detach().numpy(), rtol=0, atol=2e-8)
    # torch forms m with lerp (another rounding order); where 0.9 m and 0.1 u
    # nearly cancel the two differ by a few roundings of the terms, not of m
    np.testing.assert_allclose(m, opt.state[p]["exp_avg"].numpy(), rtol=2e-6, atol=1e-6 * np.abs(m).max())
    np.testing.assert_allclose(v, opt.state[p]["exp_avg_sq"].numpy(), rtol=2e-6, atol=1e-20)


def test_adam_skip_step_keeps_everything(orc):
    g = bf16_bits(np.ones(64))
    g[5] = 0xFFC0
    w = np.ones(64, np.float32)
    m = np.full(64, 0.5, np.float32)
    v = np.full(64, 0.25, np.float32)
    w8 = np.zeros(64, np.uint8)
    am = np.zeros(1, np.float32)
    st = orc.LossScaleState(8.0, growth=7)
    ad = orc.AdamState()
    ad.b1p[0], ad.b2p[0] = 0.81, 0.998
    orc.adam_step(g, w, m, v, w8, 1.0, am, st, ad, lr=0.1)
    assert st.found_inf[0] == 1 and st.S[0] == 4.0 and st.growth[0] == 0
    assert (w == 1).all() and (m == 0.5).all() and (v == 0.25).all() and (w8 == 0).all()
    assert ad.b1p[0] == np.float32(0.81) and ad.b2p[0] == np.float32(0.998)
