"""Helpers of the GPU parity tests: moving the same bits to both sides and the
GEMM tolerance. None of the method's arithmetic lives here."""

import numpy as np
import torch

E4M3, E5M2 = 0, 1


def np_view(t: torch.Tensor) -> np.ndarray:
    """Host numpy view with the oracle's conventions (bf16 -> uint16 bits)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def f32_bits(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def assert_same_bits(got, exp, what=""):
    got = np.asarray(got)
    exp = np.asarray(exp)
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    if got.dtype == np.float32:
        got, exp = got.view(np.uint32), exp.astype(np.float32).view(np.uint32)
    bad = np.flatnonzero(got.reshape(-1) != exp.reshape(-1))
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at {bad[:8]}: got {got.reshape(-1)[bad[:8]]}, " \
                          f"expected {exp.reshape(-1)[bad[:8]]}"


def gemm_tolerance_check(y: np.ndarray, ref: np.ndarray, abs_sum: np.ndarray, what=""):
    """Per element |y - ref| <= 2^-8 |ref| + 1e-5 * sum_k |a_k b_k| (scaled)."""
    y = y.astype(np.float64)
    err = np.abs(y - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * abs_sum
    bad = np.flatnonzero((err > bound).reshape(-1) | ~np.isfinite(y).reshape(-1))
    assert bad.size == 0, (f"{what}: {bad.size} elements out of tolerance; first {bad[:5]}: y={y.reshape(-1)[bad[:5]]} "
                           f"ref={ref.reshape(-1)[bad[:5]]} bound={bound.reshape(-1)[bad[:5]]}")
    return float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0


def finite_codes(rng, shape, fmt):
    """Random FP8 codes without NaN/Inf patterns (seeded, no arithmetic)."""
    c = rng.integers(0, 256, shape, dtype=np.uint8)
    if fmt == E4M3:
        c[(c & 0x7F) == 0x7F] = 0x3F
    else:
        c[(c & 0x7C) == 0x7C] = 0x3B
    return c


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()
