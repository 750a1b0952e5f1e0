"""Pins of the oracle's scaled cast, amax, transpose and delayed-scaling rule (CPU)."""

import numpy as np
import pytest
import torch

from conftest import read_golden

E4M3, E5M2 = 0, 1
TORCH_FMT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
ALGO = {"max": 0, "most_recent": 1}
FMT = {"e4m3": E4M3, "e5m2": E5M2}


# ----------------------------------------------------------------- cast / amax


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_scaled_cast_vs_torch(orc, fmt):
    """encode(fl32(x*scale)): torch's fp32 multiply then torch's float8 cast,
    on products that stay in range (torch's cast does not saturate)."""
    rng = np.random.default_rng(3 + fmt)
    x = (rng.standard_normal(100_000) * 3).astype(np.float32)
    for scale in (1.0, 0.37, 17.25, 2.0 ** -7, 448.0 / 13.7):
        s32 = np.float32(scale)
        p = torch.from_numpy(x) * torch.tensor(s32)
        keep = (p.abs() <= orc.fmt_max(fmt)).numpy()
        ref = p[torch.from_numpy(keep)].to(TORCH_FMT[fmt]).view(torch.uint8).numpy()
        got = orc.cast(x, float(s32), fmt)[keep]
        assert (got == ref).all()


def test_scaled_cast_bf16_bits(orc):
    """bf16 inputs widen exactly to fp32 before the multiply."""
    rng = np.random.default_rng(5)
    xb = torch.from_numpy(rng.standard_normal(50_000).astype(np.float32)).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    for fmt in (E4M3, E5M2):
        got = orc.cast(bits, 3.5, fmt)
        p = xb.float() * 3.5
        keep = (p.abs() <= orc.fmt_max(fmt)).numpy()
        ref = p[torch.from_numpy(keep)].to(TORCH_FMT[fmt]).view(torch.uint8).numpy()
        assert (got[keep] == ref).all()


def test_cast_saturates_under_scale(orc):
    x = np.array([1.0, -1.0, 2.0, 1e30, -np.inf, np.nan], dtype=np.float32)
    assert list(orc.cast(x, 448.0, E4M3)) == [0x7E, 0xFE, 0x7E, 0x7E, 0xFE, 0x7F]
    assert list(orc.cast(x, 57344.0, E5M2)) == [0x7B, 0xFB, 0x7B, 0x7B, 0xFB, 0x7F]


def test_amax_definition(orc):
    rng = np.random.default_rng(9)
    x = rng.standard_normal(100_001).astype(np.float32)
    x[17] = -9.5
    x[99] = np.nan
    assert orc.amax(x) == np.float32(9.5)
    assert orc.amax(np.zeros(0, dtype=np.float32)) == 0.0
    assert orc.amax(np.array([-0.0], dtype=np.float32)) == 0.0
    assert orc.amax(np.array([np.nan, np.nan], dtype=np.float32)) == 0.0
    assert orc.amax(np.array([1.0, -np.inf], dtype=np.float32)) == np.inf
    assert orc.amax(x) == np.nanmax(np.abs(x))
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    assert orc.amax(bits) == np.float32(torch.nan_to_num(xb.float().abs(), nan=0.0).max())


def test_transpose(orc):
    q = np.random.default_rng(1).integers(0, 256, (48, 80), dtype=np.uint8)
    assert (orc.transpose_u8(q) == q.T).all()


# ---------------------------------------------------------------- scale rule


def test_scale_sequences_from_hand_derivation(orc):
    cases = {}
    for row in read_golden("scale_update_hand.txt"):
        left, scale_s, hist_s = (p.strip() for p in row.split("|"))
        name, fmt, algo, L, margin, amax_in = left.split()
        cases.setdefault(name, []).append(
            (FMT[fmt], ALGO[algo], int(L), int(margin), float(amax_in),
             float.fromhex(scale_s) if scale_s.startswith("0x") else float(scale_s),
             [float(h) for h in hist_s.split()]))
    assert len(cases) == 3
    for name, steps in cases.items():
        fmt, algo, L, margin = steps[0][:4]
        m = orc.Meta(L)
        for (_, _, _, _, a_in, scale_exp, hist_exp) in steps:
            m.cur_amax[0] = a_in
            orc.scale_update(m, fmt, algo, margin)
            assert m.scale[0] == np.float32(scale_exp), (name, a_in)
            assert m.scale_inv[0] == np.float32(1.0) / np.float32(scale_exp)
            assert list(m.hist) == [np.float32(h) for h in hist_exp]
            assert m.cur_amax[0] == 0.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("algo", [0, 1])
def test_amax_element_lands_on_fmt_max(orc, fmt, algo):
    """After one update on a tensor, casting it again puts its amax element at
    exactly +-fmt_max: the scale maps the observed range onto the format's."""
    rng = np.random.default_rng(21 + fmt + 2 * algo)
    for _ in range(50):
        x = (rng.standard_normal(1000) * 10.0 ** rng.uniform(-6, 6)).astype(np.float32)
        m = orc.Meta(4)
        m.record_amax(orc.amax(x))
        orc.scale_update(m, fmt, algo, 0)
        q = orc.cast(x, float(m.scale[0]), fmt)
        i = int(np.argmax(np.abs(x)))
        assert orc.decode(fmt, q[i]) == np.sign(x[i]) * orc.fmt_max(fmt)
        # and nothing saturates past it
        assert np.abs(orc.decode(fmt, q)).max() == orc.fmt_max(fmt)


def test_margin_and_degenerate_amax(orc):
    m = orc.Meta(1)
    m.cur_amax[0] = 7.0
    orc.scale_update(m, E4M3, 0, 3)
    assert m.scale[0] == np.float32(np.float32(448.0) / np.float32(7.0)) / np.float32(8.0)
    keep = m.scale[0]
    for bad in (0.0, np.inf, np.nan):
        m.cur_amax[0] = bad
        orc.scale_update(m, E4M3, 1, 0)
        assert m.scale[0] == keep
    # an amax so small that fmt_max / amax overflows fp32 keeps the scale too
    m.cur_amax[0] = np.float32(1e-39)
    orc.scale_update(m, E4M3, 1, 0)
    assert m.scale[0] == keep
    assert m.scale_inv[0] == np.float32(1.0) / keep


def test_history_window_is_last_L(orc):
    """With algo max the scale follows the largest of the last L amaxes only."""
    L = 5
    m = orc.Meta(L)
    seq = [10.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0]
    scales = []
    for a in seq:
        m.cur_amax[0] = a
        orc.scale_update(m, E4M3, 0, 0)
        scales.append(float(m.scale[0]))
    assert scales[:L] == [44.8 if False else float(np.float32(448.0) / np.float32(10.0))] * L
    assert scales[L] == 448.0 and scales[L + 1] == 448.0


# ------------------------------------------------------ current scaling, dbias


def test_current_scaling_maps_amax_to_fmt_max(orc):
    rng = np.random.default_rng(31)
    for fmt in (E4M3, E5M2):
        x = (rng.standard_normal((64, 48)) * 7).astype(np.float32)
        q, m = orc.cast_current(x, fmt)
        i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert orc.decode(fmt, q[i]) == np.sign(x[i]) * orc.fmt_max(fmt)
        assert m.cur_amax[0] == np.abs(x).max()
        assert m.scale[0] == np.float32(orc.fmt_max(fmt)) / np.float32(np.abs(x).max())
    q, m = orc.cast_current(np.zeros((16, 16), np.float32), E4M3, scale0=3.0)
    assert m.scale[0] == 3.0 and (q == 0).all()


def test_dbias_definition(orc):
    rng = np.random.default_rng(32)
    # small integers: every summation order is exact
    dy = rng.integers(-40, 40, (300, 48)).astype(np.float32)
    s, a = orc.dbias(dy)
    assert (s == dy.astype(np.int64).sum(axis=0)).all()
    assert (a == np.abs(dy).sum(axis=0)).all()
    # bf16 bits against a library fp64 sum of the widened values
    xb = torch.from_numpy(rng.standard_normal((257, 33)).astype(np.float32)).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    s, _ = orc.dbias(bits)
    np.testing.assert_allclose(s, xb.double().sum(0).numpy(), rtol=1e-13, atol=1e-13)
    # columns, not rows
    assert not np.allclose(s[:33], xb.double().sum(1).numpy()[:33])
