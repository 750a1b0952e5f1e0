"""GPU parity of fp8_quantize (cast + amax + transposed copy) against the oracle:
bit-exact codes and amax."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, E5M2, assert_same_bits, dev, np_view

pytestmark = pytest.mark.gpu


def run_quantize(fp8mp, x, fmt, scale, transpose, amax0=0.0):
    rows, cols = (x.shape if x.dim() == 2 else (1, x.numel()))
    s = torch.tensor([scale], dtype=torch.float32, device="cuda")
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda") if transpose else None
    amax = torch.tensor([amax0], dtype=torch.float32, device="cuda")
    fp8mp.fp8_quantize(x, fmt, s, out, out_t, amax)
    assert fp8mp.fp8mp_check() == 0
    return out.cpu().numpy(), (out_t.cpu().numpy() if transpose else None), amax.cpu().numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("transpose", [False, True])
def test_every_bf16_pattern(cuda_lib, orc, fmt, transpose):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    x = dev(bits.view(np.int16)).view(torch.bfloat16)
    # scale 0 turns the infinities into NaN products, which must give 0x7F
    for scale in (1.0, 2.0 ** -7, 3.0, 0.1, 1e30, 0.0, -2.0):
        got, got_t, am = run_quantize(cuda_lib, x, fmt, scale, transpose)
        exp = orc.cast(bits, scale, fmt)
        assert_same_bits(got, exp, f"codes fmt={fmt} scale={scale}")
        if transpose:
            assert_same_bits(got_t, orc.transpose_u8(exp), "transposed codes")
        assert_same_bits(am, np.array([orc.amax(bits)], dtype=np.float32), "amax")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("transpose", [False, True])
def test_fp32_special_patterns(cuda_lib, orc, fmt, transpose):
    """fp32 input: every bf16 pattern widened, plus payloads only fp32 has
    (NaNs with low mantissa bits, the smallest subnormals, values just past
    the rounding and saturation boundaries), under scales that include 0
    (Inf * 0 is a NaN product) and a negative one."""
    wide = np.arange(65536, dtype=np.uint32) << 16
    rng = np.random.default_rng(20261202)
    extra = np.array([0x7F800001, 0xFF800001, 0x7FBFFFFF, 0xFFFFFFFF, 0x7FC00001, 0x00000001, 0x80000001,
                      0x007FFFFF, 0x43E00000, 0x43E00001, 0x43DFFFFF, 0x47600000, 0x47600001, 0x475FFFFF,
                      0x3B000000, 0x3B000001, 0x3AFFFFFF, 0x37800000, 0x377FFFFF], dtype=np.uint32)
    fill = rng.integers(0, 2 ** 32, size=4096 - extra.size, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([wide, extra, fill]).reshape(256, 272)
    x = dev(bits.view(np.int32)).view(torch.float32)
    for scale in (1.0, 2.0 ** -9, 0.0, -2.0):
        got, got_t, am = run_quantize(cuda_lib, x, fmt, scale, transpose)
        exp = orc.cast(bits.view(np.float32), scale, fmt)
        assert_same_bits(got, exp, f"codes fmt={fmt} scale={scale}")
        if transpose:
            assert_same_bits(got_t, orc.transpose_u8(exp), "transposed codes")
        assert_same_bits(am, np.array([orc.amax(bits.view(np.float32))], dtype=np.float32), "amax")


@pytest.mark.slow
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_every_fp32_pattern(cuda_lib, orc, fmt):
    """All 2^32 fp32 bit patterns at scale 1, in chunks of 2^28."""
    chunk = 1 << 28
    amax_all = np.float32(0.0)
    am_dev = None
    for c in range(16):
        bits = np.arange(c * chunk, (c + 1) * chunk, dtype=np.uint32)
        x = dev(bits.view(np.int32)).view(torch.float32)
        got, _, am = run_quantize(cuda_lib, x, fmt, 1.0, False)
        exp = orc.cast(bits.view(np.float32), 1.0, fmt)
        assert_same_bits(got.reshape(-1), exp, f"chunk {c}")
        assert_same_bits(am, np.array([orc.amax(bits.view(np.float32))], dtype=np.float32), f"amax chunk {c}")
        del x


SHAPES = [(16, 16), (48, 80), (1040, 784), (1024, 768), (2048, 4096)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_shapes_transposed(cuda_lib, orc, rows, cols, dtype, fmt):
    g = workloads.gen(rows * 7 + cols)
    x = (torch.randn((rows, cols), generator=g) * 3).to(dtype)
    x.view(-1)[::97] *= 40.0  # some values beyond the range after scaling
    xn = np_view(x)
    a = orc.amax(xn)
    scale = float(np.float32(orc.fmt_max(fmt)) / np.float32(a) / np.float32(2.0))
    for transpose in (False, True):
        got, got_t, am = run_quantize(cuda_lib, x.cuda(), fmt, scale, transpose, amax0=0.25)
        exp = orc.cast(xn, scale, fmt)
        assert_same_bits(got, exp, "codes")
        if transpose:
            assert_same_bits(got_t, orc.transpose_u8(exp), "transposed")
        assert_same_bits(am, np.array([max(np.float32(0.25), a)], dtype=np.float32), "amax")


@pytest.mark.parametrize("n", [1, 5, 15, 16, 17, 1000, 4097, (1 << 20) + 3])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_flat_ragged_lengths(cuda_lib, orc, n, dtype):
    x = (torch.randn((n,), generator=workloads.gen(n)) * 100).to(dtype)
    xn = np_view(x)
    for fmt in (E4M3, E5M2):
        got, _, am = run_quantize(cuda_lib, x.cuda(), fmt, 1.5, False)
        assert_same_bits(got.reshape(-1), orc.cast(xn, 1.5, fmt), f"n={n}")
        assert_same_bits(am, np.array([orc.amax(xn)], dtype=np.float32))


def test_amax_is_atomic_max_with_existing(cuda_lib, orc):
    x = torch.full((32, 32), 2.0, dtype=torch.bfloat16)
    _, _, am = run_quantize(cuda_lib, x.cuda(), E4M3, 1.0, True, amax0=7.0)
    assert am[0] == 7.0
    _, _, am = run_quantize(cuda_lib, x.cuda(), E4M3, 1.0, True, amax0=1.0)
    assert am[0] == 2.0


def test_empty_and_no_amax(cuda_lib):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    s = torch.ones(1, device="cuda")
    out = torch.empty((0, 64), dtype=torch.uint8, device="cuda")
    cuda_lib.fp8_quantize(x, E4M3, s, out)  # no-op
    x = torch.ones((16, 32), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((16, 32), dtype=torch.uint8, device="cuda")
    cuda_lib.fp8_quantize(x, E4M3, s, out, None, None)
    assert (out.cpu() == 0x38).all()  # 1.0 in E4M3


def test_transformer_activation_full_size(cuda_lib, orc):
    """The 8192 x 4096 bf16 activation with 0.1 % outliers at 50x, E4M3,
    with its transposed copy, under the scale its own amax gives."""
    tb = workloads.transformer_block(device="cuda")
    x = tb.x
    xn = np_view(x)
    a = orc.amax(xn)
    m = orc.Meta(1024)
    m.record_amax(a)
    orc.scale_update(m, E4M3, 1, 0)
    got, got_t, am = run_quantize(cuda_lib, x, E4M3, float(m.scale[0]), True)
    exp = orc.cast(xn, float(m.scale[0]), E4M3)
    assert_same_bits(got, exp, "codes")
    assert_same_bits(got_t, orc.transpose_u8(exp), "transposed")
    assert_same_bits(am, np.array([a], dtype=np.float32), "amax")
