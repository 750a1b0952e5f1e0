"""GPU parity of the widened rows: just-in-time (current) scaling and the
bias gradient fused into the output-gradient cast."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, E5M2, assert_same_bits, np_view

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols", [(16, 16), (1040, 784), (1024, 768), (4096, 4096)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_current_scaling(cuda_lib, orc, rows, cols, dtype, fmt):
    g = workloads.gen(rows + cols + fmt)
    x = (torch.randn((rows, cols), generator=g) * 5).to(dtype)
    xn = np_view(x)
    for margin in (0, 2):
        scale = torch.tensor([0.5], device="cuda")
        sinv = torch.empty(1, device="cuda")
        am = torch.full((1,), 123.0, device="cuda")
        out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
        cuda_lib.fp8_quantize_current(x.cuda(), fmt, scale, sinv, am, out, out_t, margin=margin)
        assert cuda_lib.fp8mp_check() == 0
        q, m = orc.cast_current(xn, fmt, margin=margin, scale0=0.5)
        assert_same_bits(out.cpu().numpy(), q, "codes")
        assert_same_bits(out_t.cpu().numpy(), orc.transpose_u8(q), "transposed")
        assert_same_bits(np_view(scale), m.scale, "scale")
        assert_same_bits(np_view(sinv), m.scale_inv, "scale_inv")
        assert_same_bits(np_view(am), m.cur_amax, "amax")


@pytest.mark.parametrize("rows,cols", [(1, 7), (16, 16), (1000, 333), (4096, 4096), (8192, 4096)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_current_scaling_row_only(cuda_lib, orc, rows, cols, dtype, fmt):
    """Without a transposed copy the whole current-scaling cast is one
    cooperative launch (amax, grid barrier, scale, cast of the same share):
    codes, scale, scale_inv and amax bit-exact against the oracle, on sizes
    from a tail-only 7 elements to several grid-stride passes, twice in a row
    (the second call starts from the first call's scale)."""
    g = workloads.gen(3 * rows + cols + fmt)
    x = (torch.randn((rows, cols), generator=g) * 3).to(dtype)
    xn = np_view(x)
    xd = x.cuda()
    for margin in (0, 2):
        scale = torch.tensor([0.5], device="cuda")
        sinv = torch.full((1,), 7.0, device="cuda")
        am = torch.full((1,), 123.0, device="cuda")
        out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        scale0 = 0.5
        for call in range(2):
            cuda_lib.fp8_quantize_current(xd, fmt, scale, sinv, am, out, None, margin=margin)
            assert cuda_lib.fp8mp_check() == 0
            q, m = orc.cast_current(xn, fmt, margin=margin, scale0=scale0)
            assert_same_bits(out.cpu().numpy(), q, f"codes call {call}")
            assert_same_bits(np_view(scale), m.scale, "scale")
            assert_same_bits(np_view(sinv), m.scale_inv, "scale_inv")
            assert_same_bits(np_view(am), m.cur_amax, "amax")
            scale0 = float(m.scale[0])


def test_current_scaling_degenerate(cuda_lib, orc):
    for fill in (0.0, float("inf"), float("nan")):
        x = torch.full((32, 32), fill, dtype=torch.float32)
        scale = torch.tensor([3.0], device="cuda")
        sinv = torch.empty(1, device="cuda")
        am = torch.empty(1, device="cuda")
        out = torch.empty((32, 32), dtype=torch.uint8, device="cuda")
        cuda_lib.fp8_quantize_current(x.cuda(), E4M3, scale, sinv, am, out)
        assert cuda_lib.fp8mp_check() == 0
        q, m = orc.cast_current(np_view(x), E4M3, scale0=3.0)
        assert scale.item() == 3.0 and m.scale[0] == 3.0
        assert_same_bits(out.cpu().numpy(), q, f"codes fill={fill}")
        assert_same_bits(np_view(am), m.cur_amax, "amax")


def dbias_check(got, ref, ab, rows, bf16):
    """fp32 summation of `rows` terms in any order is off by at most
    rows * 2^-24 * sum|x|; a bf16 result adds one round-to-nearest of a value
    with an 8-bit significand: at most 2^-8 |ref| (its unit roundoff)."""
    err = np.abs(got.astype(np.float64) - ref)
    bound = rows * 2.0 ** -24 * ab + (2.0 ** -8 * (np.abs(ref) + rows * 2.0 ** -24 * ab) if bf16 else 0.0) + 1e-30
    assert (err <= bound).all(), (err / bound).max()


@pytest.mark.parametrize("rows,cols", [(16, 16), (144, 272), (1040, 784), (16, 4096), (4112, 16), (8192, 4096)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("db_dtype", [torch.float32, torch.bfloat16])
def test_dbias_fused_in_gradient_cast(cuda_lib, orc, rows, cols, dtype, db_dtype):
    g = workloads.gen(7 * rows + cols)
    dy = (torch.randn((rows, cols), generator=g) * 1e-3 + 2e-4).to(dtype)
    dyn = np_view(dy)
    scale = torch.tensor([4096.0], device="cuda")
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    am = torch.zeros(1, device="cuda")
    db = torch.empty(cols, dtype=db_dtype, device="cuda")
    ws = torch.zeros(cuda_lib.fp8_quantize_dbias_workspace_bytes(rows, cols) // 4, dtype=torch.float32,
                     device="cuda")
    cuda_lib.fp8_quantize_dbias(dy.cuda(), E5M2, scale, out, out_t, db, ws, amax=am)
    assert cuda_lib.fp8mp_check() == 0
    q = orc.cast(dyn, 4096.0, E5M2)
    assert_same_bits(out.cpu().numpy(), q, "codes")
    assert_same_bits(out_t.cpu().numpy(), orc.transpose_u8(q), "transposed")
    assert_same_bits(np_view(am), np.array([orc.amax(dyn)], np.float32), "amax")
    ref, ab = orc.dbias(dyn)
    dbias_check(np_view(db.float()), ref, ab, rows, db_dtype == torch.bfloat16)
    # deterministic: a second call gives the same bits
    db2 = torch.empty_like(db)
    cuda_lib.fp8_quantize_dbias(dy.cuda(), E5M2, scale, out, out_t, db2, ws, amax=am)
    assert cuda_lib.fp8mp_check() == 0
    assert torch.equal(db.view(torch.uint8) if db.dtype == torch.uint8 else db, db2)


@pytest.mark.parametrize("rows,cols", [(144, 272), (8192, 4096)])
def test_dbias_without_transposed_copy(cuda_lib, orc, rows, cols):
    """out_t = NULL: the same codes, amax and bias gradient, no transposed
    copy (for a backward that reads dY8 row-major)."""
    g = workloads.gen(3 * rows + cols)
    dy = (torch.randn((rows, cols), generator=g) * 1e-3).to(torch.bfloat16).cuda()
    scale = torch.tensor([8192.0], device="cuda")
    ws = torch.zeros(cuda_lib.fp8_quantize_dbias_workspace_bytes(rows, cols) // 4, dtype=torch.float32,
                     device="cuda")
    out, am, db = (torch.empty((rows, cols), dtype=torch.uint8, device="cuda"), torch.zeros(1, device="cuda"),
                   torch.empty(cols, device="cuda"))
    cuda_lib.fp8_quantize_dbias(dy, E5M2, scale, out, None, db, ws, amax=am)
    out2, am2, db2 = torch.empty_like(out), torch.zeros(1, device="cuda"), torch.empty_like(db)
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    cuda_lib.fp8_quantize_dbias(dy, E5M2, scale, out2, out_t, db2, ws, amax=am2)
    assert cuda_lib.fp8mp_check() == 0
    dyn = np_view(dy)
    assert_same_bits(out.cpu().numpy(), orc.cast(dyn, 8192.0, E5M2), "codes")
    assert torch.equal(out, out2) and torch.equal(am, am2) and torch.equal(db, db2)
    ref, ab = orc.dbias(dyn)
    dbias_check(np_view(db), ref, ab, rows, False)


def test_dbias_leaves_its_workspace_zero_across_shapes(cuda_lib, orc):
    """One zero-filled workspace serves calls of different shapes in turn:
    every call sets the tile sums and arrival counters it used back to zero
    (the last tile of each column strip does), so each call starts from a
    zero workspace and gets the oracle's codes and a bias gradient within the
    summation bound."""
    shapes = [(1040, 784), (144, 2064), (4112, 16), (2064, 1552), (1040, 784)]
    need = max(cuda_lib.fp8_quantize_dbias_workspace_bytes(r, c) for r, c in shapes)
    ws = torch.zeros(need // 4, dtype=torch.float32, device="cuda")
    scale = torch.tensor([1024.0], device="cuda")
    for i, (rows, cols) in enumerate(shapes):
        g = workloads.gen(1000 + i)
        dy = (torch.randn((rows, cols), generator=g) * 1e-3 - 3e-4 * i).to(torch.bfloat16)
        dyn = np_view(dy)
        out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda") if i % 2 == 0 else None
        db = torch.empty(cols, dtype=torch.float32, device="cuda")
        am = torch.zeros(1, device="cuda")
        cuda_lib.fp8_quantize_dbias(dy.cuda(), E5M2, scale, out, out_t, db, ws, amax=am)
        assert cuda_lib.fp8mp_check() == 0
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws)) == 0, f"call {i}: workspace not left zero"
        q = orc.cast(dyn, 1024.0, E5M2)
        assert_same_bits(out.cpu().numpy(), q, f"codes {i}")
        if out_t is not None:
            assert_same_bits(out_t.cpu().numpy(), orc.transpose_u8(q), f"transposed {i}")
        assert_same_bits(np_view(am), np.array([orc.amax(dyn)], np.float32), f"amax {i}")
        ref, ab = orc.dbias(dyn)
        dbias_check(np_view(db), ref, ab, rows, False)


def dbias_in_documented_order(x):
    """The bias gradient summed in the order the library documents for its
    fused cast, restated in numpy fp32 (each addition one IEEE round to
    nearest): k = max(1, min(tile rows, 152 // strips)) CTAs per 128-column
    strip, CTA j taking tile rows j, j + k, ...; per column, 32 running sums
    of 4-row runs (thread row ty adds rows 4ty .. 4ty + 3 of each of its
    tiles, tile after tile); the four runs of a warp combined pairwise (ty ^ 1,
    then ty ^ 2); the 8 warps in order; then the k CTA sums in order of j."""
    rows, cols = x.shape
    tr, tc = -(-rows // 128), -(-cols // 128)
    k = max(1, min(tr, 152 // tc))
    xp = np.zeros((tr * 128, tc * 128), np.float32)
    xp[:rows, :cols] = x
    ctas = []
    for j in range(k):
        s = np.zeros((32, tc * 128), np.float32)
        for t in range(j, tr, k):
            blk = xp[t * 128:(t + 1) * 128].reshape(32, 4, -1)
            for rr in range(4):
                s = s + blk[:, rr, :]
        s = s.reshape(8, 4, -1)
        w = (s[:, 0] + s[:, 1]) + (s[:, 2] + s[:, 3])
        t_sum = w[0]
        for ww in range(1, 8):
            t_sum = t_sum + w[ww]
        ctas.append(t_sum)
    tot = ctas[0]
    for j in range(1, k):
        tot = tot + ctas[j]
    return tot[:cols], k


@pytest.mark.parametrize("with_t", [False, True])
@pytest.mark.parametrize("rows,cols", [(8192, 4096), (144, 272), (1040, 784), (4112, 16), (16, 4096), (2064, 1552)])
def test_dbias_follows_its_documented_order(cuda_lib, rows, cols, with_t):
    """Bit for bit the fp32 sums of the documented order, whichever way the
    launch combined the CTAs of a strip (without a transposed copy and for
    2 <= k <= 8 a cluster reading its CTAs' sums from distributed shared
    memory, else the workspace and the strip's last arriver; nothing to
    combine at k = 1)."""
    g = workloads.gen(11 * rows + cols)
    dy = (torch.randn((rows, cols), generator=g) * 1e-2 + 1e-3).to(torch.bfloat16)
    want, k = dbias_in_documented_order(np_view(dy.float()))
    ws = torch.zeros(cuda_lib.fp8_quantize_dbias_workspace_bytes(rows, cols) // 4, dtype=torch.float32,
                     device="cuda")
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda") if with_t else None
    db = torch.empty(cols, dtype=torch.float32, device="cuda")
    cuda_lib.fp8_quantize_dbias(dy.cuda(), E5M2, torch.ones(1, device="cuda"), out, out_t, db, ws)
    assert cuda_lib.fp8mp_check() == 0
    assert int(torch.count_nonzero(ws)) == 0
    assert_same_bits(np_view(db), want, f"dbias, k={k}")


def test_dbias_rejects_small_workspace(cuda_lib):
    dy = torch.ones((256, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((256, 64), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((64, 256), dtype=torch.uint8, device="cuda")
    db = torch.empty(64, device="cuda")
    ws = torch.empty(16, device="cuda")
    with pytest.raises(cuda_lib.Fp8mpError) as e:
        cuda_lib.fp8_quantize_dbias(dy, E5M2, torch.ones(1, device="cuda"), out, out_t, db, ws)
    assert e.value.code == cuda_lib.ERR_INVALID and "workspace" in cuda_lib.last_error()


@pytest.mark.parametrize("engine", ["single", "pair"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (1040, 784, 784), (2304, 2560, 1024)])
@pytest.mark.parametrize("y_fmt", [E4M3, E5M2])
def test_fwd_with_fp8_output(cuda_lib, orc, monkeypatch, engine, M, N, K, y_fmt):
    """FP8 codes written by the GEMM epilogue: (a) the same codes a plain cast
    of the GEMM's own fp32 output gives (torch's float8 cast, a library
    routine, with saturation beyond the range); (b) every code inside the
    band of values that the GEMM tolerance around the oracle's reference
    allows; (c) the amax is the fp32 output's, close to the reference's."""
    from gpu_util import dev, finite_codes, gemm_tolerance_check

    monkeypatch.setenv("FP8MP_GEMM_ENGINE", engine)
    rng = np.random.default_rng(M + N + K + y_fmt)
    A = finite_codes(rng, (M, K), E4M3)
    B = finite_codes(rng, (N, K), E4M3)
    sa, sb = 2.0 ** -7, 0.05
    bias = (torch.randn(N, generator=workloads.gen(5)) * 10).to(torch.bfloat16)
    ref, ab = orc.gemm_ref(A, E4M3, B, E4M3, float(np.float32(sa)), float(np.float32(sb)),
                           bias=bias.double().numpy())
    ys = np.float32(orc.fmt_max(y_fmt) / (np.abs(ref).max() * 0.8))  # the top 20 % saturates
    one = lambda v: torch.tensor([v], dtype=torch.float32, device="cuda")
    y8 = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    am = torch.zeros(1, device="cuda")
    cuda_lib.fp8_linear_fwd_fp8out(dev(A), dev(B), one(sa), one(sb), one(ys), y8, y_fmt=y_fmt,
                                   bias=bias.cuda(), y_amax=am)
    y32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    cuda_lib.fp8_linear_fwd(dev(A), dev(B), one(sa), one(sb), y32, bias=bias.cuda())
    assert cuda_lib.fp8mp_check() == 0
    codes = y8.cpu().numpy()
    yh = np_view(y32)
    gemm_tolerance_check(yh.astype(np.float64), ref, ab, "fp32 output")
    # (a) the epilogue's cast of its own fp32 y
    tfmt = torch.float8_e4m3fn if y_fmt == E4M3 else torch.float8_e5m2
    prod = torch.from_numpy(yh) * torch.tensor(ys)
    vmax = orc.fmt_max(y_fmt)
    expect = prod.clamp(-vmax, vmax).to(tfmt).view(torch.uint8).numpy()
    assert (codes == expect).all()
    # (b) the band allowed by the tolerance around the fp64 reference
    tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * ab
    lo = orc.decode(y_fmt, orc.cast(((ref - tol) * ys).astype(np.float32), 1.0, y_fmt))
    hi = orc.decode(y_fmt, orc.cast(((ref + tol) * ys).astype(np.float32), 1.0, y_fmt))
    val = orc.decode(y_fmt, codes)
    assert ((val >= lo) & (val <= hi)).all()
    # (c) amax of the fp32 output
    assert am.item() == np.abs(yh).max()
