"""Pins of the oracle's E4M3 / E5M2 decoder and encoder (CPU only).

The codec is checked against what the pages and the mathematics fix, never
against a retyped copy of itself:
  * the finfo table and the worked cast example the PyTorch-native-FP8 page
    prints (tests/golden);
  * torch's own float8 dtypes (the library the same page uses) for decoding
    every code and for casting in-range values;
  * brute force: the nearest representable value found by exhaustive search,
    ties to the even code;
  * exhaustive decode -> encode identity on every finite code.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden

E4M3, E5M2 = 0, 1
TORCH_FMT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
NAME = {"float8_e4m3fn": E4M3, "float8_e5m2": E5M2}


def torch_grid(fmt):
    """Value of every code according to torch's float8 dtype (a library decoder)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_FMT[fmt]).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decoder_matches_torch_dtype_on_all_codes(orc, fmt):
    ours = orc.decode(fmt, np.arange(256, dtype=np.uint8))
    ref = torch_grid(fmt)
    nan_o, nan_r = np.isnan(ours), np.isnan(ref)
    assert (nan_o == nan_r).all()
    assert (ours[~nan_o] == ref[~nan_r]).all()
    # signed zeros are distinct codes
    assert math.copysign(1.0, ours[0x00]) == 1.0 and math.copysign(1.0, ours[0x80]) == -1.0


def test_code_counts(orc):
    e4 = orc.decode(E4M3, np.arange(256, dtype=np.uint8))
    e5 = orc.decode(E5M2, np.arange(256, dtype=np.uint8))
    assert np.isfinite(e4).sum() == 254 and np.isnan(e4).sum() == 2 and np.isinf(e4).sum() == 0
    assert np.isfinite(e5).sum() == 248 and np.isnan(e5).sum() == 6 and np.isinf(e5).sum() == 2


def test_finfo_table_from_page(orc):
    rows = {r.split()[0]: r.split()[1:] for r in read_golden("finfo_pt_fp8.txt")}
    for name, fmt in NAME.items():
        bits, mx, mn, smallest_normal, eps = (float(v) for v in rows[name])
        assert bits == 8
        vals = orc.decode(fmt, np.arange(256, dtype=np.uint8))
        fin = vals[np.isfinite(vals)]
        assert fin.max() == mx and fin.min() == mn
        # smallest normal: the smallest positive value whose exponent field is non-zero
        mbits = 3 if fmt == E4M3 else 2
        normals = [orc.decode(fmt, c) for c in range(1, 128) if (c >> mbits) != 0]
        assert min(normals) == pytest.approx(smallest_normal, rel=1e-5)
        # eps: distance from 1.0 to the next larger representable value
        pos = np.sort(fin[fin > 0])
        nxt = pos[pos > 1.0][0]
        assert nxt - 1.0 == eps
        assert orc.fmt_max(fmt) == mx


def test_worked_cast_example_from_page(orc):
    rows = {r.split()[0]: [float(v) for v in r.split()[1:]] for r in read_golden("worked_cast_pt_fp8.txt")}
    x = np.array(rows["float32"], dtype=np.float32)
    for name, fmt in NAME.items():
        got = orc.decode(fmt, orc.encode(fmt, x))
        assert list(got) == rows[name], name


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_roundtrip_every_finite_code(orc, fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.decode(fmt, codes)
    fin = np.isfinite(vals)
    back = orc.encode(fmt, vals[fin].astype(np.float32))
    assert (back == codes[fin]).all()


def brute_force_encode(fmt, x, grid):
    """Nearest finite value by exhaustive search over all codes (exact rational
    distances); a tie between two values goes to the code whose mantissa LSB is
    even; |x| at or beyond the largest finite value saturates; a zero result
    keeps the sign of x; NaN -> 0x7F."""
    if math.isnan(x):
        return 0x7F
    cand = [(c, v) for c, v in enumerate(grid) if np.isfinite(v) and c != 0x80]
    vmax = max(v for _, v in cand)
    if x >= vmax:
        return [c for c, v in cand if v == vmax][0]
    if x <= -vmax:
        return [c for c, v in cand if v == -vmax][0]
    fx = Fraction(x)
    dist = [(abs(Fraction(v) - fx), c, v) for c, v in cand]
    dmin = min(d for d, _, _ in dist)
    best = [(c, v) for d, c, v in dist if d == dmin]
    if len(best) > 1:
        best = [(c, v) for c, v in best if (c & 1) == 0]
    assert len(best) == 1
    c, v = best[0]
    if v == 0.0:
        return 0x80 if math.copysign(1.0, x) < 0 else 0x00
    return c


def boundary_values(fmt):
    grid = torch_grid(fmt)
    fin = np.array(sorted(set(v for v in grid if np.isfinite(v))))
    vals = []
    # every midpoint between neighbours (exact ties), and one fp32 ulp either side
    for a, b in zip(fin[:-1], fin[1:]):
        mid = np.float32((a + b) / 2)
        vals += [mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(-np.inf))]
    vmax = fin.max()
    big = [vmax, np.nextafter(np.float32(vmax), np.float32(np.inf)), vmax * 1.03, vmax * 1.0625,
           vmax * 1.2, vmax * 2, 1e30, np.finfo(np.float32).max]
    vals += big + [-v for v in big]
    sub_min = fin[fin > 0].min()
    vals += [sub_min / 2, np.nextafter(np.float32(sub_min / 2), np.float32(1)), sub_min / 4,
             -sub_min / 2, 1e-40, -1e-40, 1e-45, 0.0, -0.0]
    return np.array(vals, dtype=np.float32)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encoder_brute_force_boundaries(orc, fmt):
    grid = torch_grid(fmt)
    x = boundary_values(fmt)
    got = orc.encode(fmt, x)
    for xi, gi in zip(x, got):
        assert gi == brute_force_encode(fmt, float(xi), grid), (fmt, float(xi), hex(gi))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encoder_brute_force_random(orc, fmt):
    grid = torch_grid(fmt)
    rng = np.random.default_rng(7 + fmt)
    x = np.concatenate([
        rng.standard_normal(300).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(200) * 10.0 ** rng.uniform(-8, 6, 200)).astype(np.float32),
    ])
    got = orc.encode(fmt, x)
    for xi, gi in zip(x, got):
        assert gi == brute_force_encode(fmt, float(xi), grid), (fmt, float(xi), hex(gi))


def test_special_values(orc):
    inf, nan = np.float32(np.inf), np.float32(np.nan)
    for fmt, maxc in ((E4M3, 0x7E), (E5M2, 0x7B)):
        got = orc.encode(fmt, np.array([inf, -inf, nan, -nan, 0.0, -0.0], dtype=np.float32))
        assert list(got) == [maxc, 0x80 | maxc, 0x7F, 0x7F, 0x00, 0x80]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encoder_matches_torch_cast_in_range(orc, fmt):
    """torch's float8 cast (no saturation) agrees for every |x| <= max."""
    rng = np.random.default_rng(11 + fmt)
    vmax = orc.fmt_max(fmt)
    x = np.concatenate([
        rng.uniform(-vmax, vmax, 200_000),
        rng.standard_normal(200_000) * 10.0 ** rng.uniform(-12, 3, 200_000),
    ]).astype(np.float32)
    x = x[np.abs(x) <= vmax]
    ours = orc.encode(fmt, x)
    ref = torch.from_numpy(x).to(TORCH_FMT[fmt]).view(torch.uint8).numpy()
    # torch keeps the sign of a zero result; both sides should give the same code
    assert (ours == ref).all(), np.flatnonzero(ours != ref)[:10]


def test_encoder_every_bf16_pattern_vs_torch(orc):
    """All 65536 bf16 values (as fp32) in range agree with torch's cast."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    for fmt in (E4M3, E5M2):
        keep = np.isfinite(x) & (np.abs(x) <= orc.fmt_max(fmt))
        ours = orc.encode(fmt, x[keep])
        ref = torch.from_numpy(x[keep].copy()).to(TORCH_FMT[fmt]).view(torch.uint8).numpy()
        assert (ours == ref).all()
        # beyond the range: saturation to the signed largest finite code
        over = np.isfinite(x) & (np.abs(x) > orc.fmt_max(fmt))
        sat = orc.encode(fmt, x[over])
        maxc = 0x7E if fmt == E4M3 else 0x7B
        exp = np.where(np.signbit(x[over]), 0x80 | maxc, maxc)
        assert (sat == exp).all()
