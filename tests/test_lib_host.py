"""The C-ABI library on the CPU host: it builds, loads, exports every entry
point include/fp8mp.h declares, and its argument validation (which runs before
any CUDA call) rejects bad input with FP8MP_ERR_INVALID. No compute calls."""

import ctypes
import os
import re

import pytest

import fp8_mixed_precision_reduce_gb300 as fp8mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8mp.h")


@pytest.fixture(scope="module")
def lib():
    fp8mp.build()
    return fp8mp.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fp8_quantize", "fp8_linear_fwd", "fp8_linear_dgrad", "fp8_linear_wgrad", "fp8_linear_bwd",
              "delayed_scaling_update", "mp_master_step", "fp8mp_check", "fp8mp_last_error",
              "fp8mp_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(fp8mp.EXPORTS) <= set(declared_functions())


def test_version_and_empty_error(lib):
    assert fp8mp.fp8mp_version() == 1
    assert fp8mp.last_error() == ""


def test_ctypes_meta_layout_matches_header():
    # four pointers then two int32: 40 bytes with 8-byte alignment
    assert ctypes.sizeof(fp8mp.fp8mp_meta) == 40
    assert fp8mp.fp8mp_meta.history_len.offset == 32


def test_quantize_rejects_bad_arguments(lib):
    P = 4096  # a fake, aligned address: never dereferenced, validation fails first
    assert lib.fp8_quantize(P, 7, 16, 16, 0, P, P, None, None, None) == fp8mp.ERR_INVALID
    assert "x_dtype" in fp8mp.last_error()
    assert lib.fp8_quantize(P, 1, 16, 16, 5, P, P, None, None, None) == fp8mp.ERR_INVALID
    assert lib.fp8_quantize(P, 1, -1, 16, 0, P, P, None, None, None) == fp8mp.ERR_INVALID
    # a transposed output needs both dims divisible by 16
    assert lib.fp8_quantize(P, 1, 24, 16, 0, P, P, P, None, None) == fp8mp.ERR_INVALID
    assert "multiples of 16" in fp8mp.last_error()
    # misaligned / missing pointers
    assert lib.fp8_quantize(P + 2, 1, 16, 16, 0, P, P, None, None, None) == fp8mp.ERR_INVALID
    assert "aligned" in fp8mp.last_error()
    assert lib.fp8_quantize(None, 1, 16, 16, 0, P, P, None, None, None) == fp8mp.ERR_INVALID
    assert lib.fp8_quantize(P, 1, 16, 16, 0, None, P, None, None, None) == fp8mp.ERR_INVALID
    # an empty tensor is a no-op that needs no pointer and no device
    assert lib.fp8_quantize(None, 1, 0, 16, 0, None, None, None, None, None) == fp8mp.OK


def test_gemms_reject_bad_shapes(lib):
    P = 4096
    for fn in (lambda M, N, K: lib.fp8_linear_fwd(P, P, M, N, K, P, P, None, 0, P, 1, None, None),
               lambda M, N, K: lib.fp8_linear_dgrad(P, P, M, N, K, 1, P, P, P, 1, None),
               lambda M, N, K: lib.fp8_linear_wgrad(P, P, M, N, K, 1, P, P, P, 1, None)):
        assert fn(24, 32, 32) == fp8mp.ERR_INVALID
        assert fn(32, 40, 32) == fp8mp.ERR_INVALID
        assert fn(32, 32, 8) == fp8mp.ERR_INVALID
        assert fn(-16, 32, 32) == fp8mp.ERR_INVALID
        assert fn(1 << 31, 32, 32) == fp8mp.ERR_INVALID
    # empty outputs are no-ops
    assert lib.fp8_linear_fwd(None, None, 0, 32, 32, None, None, None, 0, None, 1, None, None) == fp8mp.OK
    assert lib.fp8_linear_dgrad(None, None, 32, 32, 0, 1, None, None, None, 1, None) == fp8mp.OK
    assert lib.fp8_linear_wgrad(None, None, 32, 0, 32, 1, None, None, None, 1, None) == fp8mp.OK
    # bad enums
    assert lib.fp8_linear_fwd(P, P, 32, 32, 32, P, P, None, 0, P, 9, None, None) == fp8mp.ERR_INVALID
    assert lib.fp8_linear_dgrad(P, P, 32, 32, 32, 3, P, P, P, 1, None) == fp8mp.ERR_INVALID


def test_fused_backward_rejects_bad_arguments(lib):
    P = 1 << 20  # fake, aligned addresses: never dereferenced, validation fails first
    bwd = lambda M, N, K, dx=P, dw=2 * P, fmt=1, dxt=1, dwt=1: lib.fp8_linear_bwd(
        P, P, P, P, M, N, K, fmt, P, P, P, dx, dxt, dw, dwt, None)
    for shape in ((24, 32, 32), (32, 40, 32), (32, 32, 8), (-16, 32, 32), (1 << 31, 32, 32)):
        assert bwd(*shape) == fp8mp.ERR_INVALID
    assert bwd(32, 32, 32, fmt=2) == fp8mp.ERR_INVALID
    assert bwd(32, 32, 32, dxt=5) == fp8mp.ERR_INVALID and "dx_dtype" in fp8mp.last_error()
    assert bwd(32, 32, 32, dwt=5) == fp8mp.ERR_INVALID and "dw_dtype" in fp8mp.last_error()
    assert bwd(32, 32, 32, dw=None) == fp8mp.ERR_INVALID
    assert bwd(32, 32, 32, dx=P + 4) == fp8mp.ERR_INVALID and "aligned" in fp8mp.last_error()
    # dx (32 x 32 bf16 = 2 KiB) and dw must not overlap
    assert bwd(32, 32, 32, dx=P, dw=P + 1024) == fp8mp.ERR_INVALID and "overlap" in fp8mp.last_error()
    # empty outputs are no-ops needing no pointer and no device
    assert lib.fp8_linear_bwd(None, None, None, None, 32, 32, 0, 1, None, None, None, None, 1, None, 1,
                              None) == fp8mp.OK
    assert lib.fp8_linear_bwd(None, None, None, None, 0, 0, 32, 1, None, None, None, None, 1, None, 1,
                              None) == fp8mp.OK


def test_rowmajor_backward_rejects_bad_arguments(lib):
    P = 1 << 20
    bwd = lambda M, N, K, dx=P, dw=2 * P, fmt=1, dxt=1, dwt=1, w8=P, x8=P, nf=None: lib.fp8_linear_bwd_rowmajor(
        P, w8, x8, M, N, K, fmt, P, P, P, dx, dxt, dw, dwt, nf, None)
    for shape in ((24, 32, 32), (32, 40, 32), (32, 32, 8), (-16, 32, 32)):
        assert bwd(*shape) == fp8mp.ERR_INVALID
    assert bwd(32, 32, 32, fmt=3) == fp8mp.ERR_INVALID
    assert bwd(32, 32, 32, dwt=7) == fp8mp.ERR_INVALID and "dw_dtype" in fp8mp.last_error()
    assert bwd(32, 32, 32, w8=None) == fp8mp.ERR_INVALID and "w8" in fp8mp.last_error()
    assert bwd(32, 32, 32, x8=P + 3) == fp8mp.ERR_INVALID and "aligned" in fp8mp.last_error()
    assert bwd(32, 32, 32, dx=P, dw=P + 64) == fp8mp.ERR_INVALID and "overlap" in fp8mp.last_error()
    assert bwd(32, 32, 32, nf=P + 2) == fp8mp.ERR_INVALID and "dw_nonfinite" in fp8mp.last_error()
    # nothing requested: a no-op needing no pointer and no device
    assert lib.fp8_linear_bwd_rowmajor(None, None, None, 32, 32, 32, 1, None, None, None, None, 1, None, 1,
                                       None, None) == fp8mp.OK


def test_scale_update_rejects_bad_metas(lib):
    P = 4096
    good = fp8mp.fp8mp_meta(P, P, P, P, 16, 0)
    arr = (fp8mp.fp8mp_meta * 1)(good)
    assert lib.delayed_scaling_update(arr, 0, 0, 0, None) == fp8mp.OK
    assert lib.delayed_scaling_update(arr, 1, 2, 0, None) == fp8mp.ERR_INVALID
    assert lib.delayed_scaling_update(arr, 1, 0, -1, None) == fp8mp.ERR_INVALID
    assert lib.delayed_scaling_update(arr, 1, 0, 127, None) == fp8mp.ERR_INVALID
    for bad in (fp8mp.fp8mp_meta(P, P, P, P, 0, 0), fp8mp.fp8mp_meta(P, P, P, P, 8193, 0),
                fp8mp.fp8mp_meta(P, P, P, P, 16, 2), fp8mp.fp8mp_meta(None, P, P, P, 16, 0)):
        arr = (fp8mp.fp8mp_meta * 1)(bad)
        assert lib.delayed_scaling_update(arr, 1, 0, 0, None) == fp8mp.ERR_INVALID


def test_master_step_rejects_bad_arguments(lib):
    P = 4096
    args = [P, 1024, P, P, P, P, P, P, P, P, 1e-4, 0.9, 0.5, 2.0, 2000, None]
    bad = list(args)
    bad[14] = 0  # growth_interval
    assert lib.mp_master_step(*bad) == fp8mp.ERR_INVALID
    bad = list(args)
    bad[2] = P + 8  # master misaligned
    assert lib.mp_master_step(*bad) == fp8mp.ERR_INVALID
    bad = list(args)
    bad[7] = None  # loss_scale
    assert lib.mp_master_step(*bad) == fp8mp.ERR_INVALID
    bad = list(args)
    bad[1] = -5
    assert lib.mp_master_step(*bad) == fp8mp.ERR_INVALID


def test_prescanned_master_steps_need_their_own_flag(lib):
    P = 4096
    sgd = [P, 1024, P, P, P, P, P, P, P, P, 2 * P, 1e-4, 0.9, 0.5, 2.0, 2000, None]
    bad = list(sgd)
    bad[10] = None  # grad_nonfinite is required
    assert lib.mp_master_step_prescanned(*bad) == fp8mp.ERR_INVALID and "grad_nonfinite" in fp8mp.last_error()
    bad = list(sgd)
    bad[10] = P  # the same word as found_inf
    assert lib.mp_master_step_prescanned(*bad) == fp8mp.ERR_INVALID and "different" in fp8mp.last_error()
    bad = list(sgd)
    bad[10] = 2 * P + 1  # misaligned
    assert lib.mp_master_step_prescanned(*bad) == fp8mp.ERR_INVALID
    adam = [P, 1024, P, P, P, P, P, P, P, P, P, None, P, 1e-4, 0.9, 0.999, 1e-8, 0.5, 2.0, 2000, None]
    assert lib.mp_master_step_adam_prescanned(*adam) == fp8mp.ERR_INVALID and "grad_nonfinite" in fp8mp.last_error()
    bad = list(adam)
    bad[11] = 2 * P
    bad[14] = 1.5  # beta1 outside [0, 1)
    assert lib.mp_master_step_adam_prescanned(*bad) == fp8mp.ERR_INVALID and "betas" in fp8mp.last_error()


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(fp8mp.Fp8mpError):
        saved = fp8mp._lib
        fp8mp._lib = None
        try:
            fp8mp.load(str(tmp_path / "nope.so"))
        finally:
            fp8mp._lib = saved


def test_dbias_workspace_size_and_noalloc_limit(lib):
    """The workspace holds the column sums of each of the k CTAs of a
    128-column strip (k = min(ceil(rows / 128), max(1, 152 // strips))) plus
    one arrival counter per strip, rounded up to 16 bytes; the allocation-free
    variant refuses, before any CUDA call, shapes whose workspace exceeds its
    fixed array -- including shapes whose size product would overflow."""
    ws = fp8mp.fp8_quantize_dbias_workspace_bytes

    def closed_form(rows, cols):
        tr, tc = -(-rows // 128), -(-cols // 128)
        k = max(1, min(tr, 152 // tc if tc else 1))
        return (k * cols * 4 + tc * 4 + 15) // 16 * 16

    for rows, cols in ((8192, 4096), (16, 16), (1040, 784), (16384, 14336), (1024, 768), (128, 16), (4112, 16),
                       (0, 4096), (65536, 1 << 20)):
        assert ws(rows, cols) == closed_form(rows, cols), (rows, cols)
    assert ws(8192, 4096) == 4 * 4096 * 4 + 32 * 4  # 4 CTAs per strip
    assert ws(16, 16) == 16 * 4 + 16  # one CTA's 16 sums and one counter, padded to 16
    assert ws(-1, 16) == -1
    assert ws(1 << 40, 1 << 20) == -1  # beyond 2^40 elements: no overflowing product
    limit = 4 * fp8mp.NOALLOC_DBIAS_SCRATCH_FLOATS
    assert ws(16384, 1040432) <= limit < ws(16384, 1040448)
    assert ws(65536, 16384) <= limit
    P = 4096  # fake aligned address, never dereferenced: validation fails first
    for rows, cols in ((16384, 1040448), (1 << 40, 1 << 20), (1 << 62, 1 << 62)):
        rc = lib.fp8_quantize_dbias_noalloc(P, 1, rows, cols, 1, P, P, None, None, P, 0, None)
        assert rc == fp8mp.ERR_INVALID, (rows, cols)
        assert "scratch" in fp8mp.last_error()


def test_quantize_ex_rejects_unknown_flags(lib):
    P = 4096  # fake aligned address, never dereferenced: validation fails first
    assert lib.fp8_quantize_ex(P, 1, 16, 16, 0, P, P, None, None, 2, None) == fp8mp.ERR_INVALID
    assert "flags" in fp8mp.last_error()
    assert lib.fp8_quantize_ex(P, 1, 16, 16, 0, P, P, None, None, 1 << 31, None) == fp8mp.ERR_INVALID


def test_scale_update_ex_rejects_a_misaligned_snapshot(lib):
    P = 4096
    arr = (fp8mp.fp8mp_meta * 1)(fp8mp.fp8mp_meta(P, P, P, P, 16, 0))
    assert lib.delayed_scaling_update_ex(arr, 0, 0, 0, P + 2, None) == fp8mp.OK  # n == 0: no-op
    assert lib.delayed_scaling_update_ex(arr, 1, 0, 0, P + 2, None) == fp8mp.ERR_INVALID
    assert "prev_scale_inv" in fp8mp.last_error()
    assert lib.delayed_scaling_update_ex(arr, 1, 2, 0, None, None) == fp8mp.ERR_INVALID  # the same checks


def test_master_step_ex_rejects_bad_copies_and_flags(lib):
    """The two-buffer steps: unknown flags, a misaligned w8_in and a w8_in
    that overlaps w8_out without being it are refused before any CUDA call."""
    P, n = 1 << 20, 1024
    # grad, n, master, momentum, w8_in, w8_out, scale_w, amax_w, S, growth, found, gnf, lr, mu, bo, gf, gi, flags
    sgd = [P, n, P, P, 8 * P, 4 * P, P, P, P, P, P, 2 * P, 1e-4, 0.9, 0.5, 2.0, 2000, 0, None]
    for i, v, word in ((17, 2, "flags"), (17, 1 << 31, "flags"), (4, 8 * P + 8, "w8_in"),
                       (4, 4 * P + 512, "overlap"), (4, 4 * P - 512, "overlap"), (11, None, "grad_nonfinite")):
        bad = list(sgd)
        bad[i] = v
        assert lib.mp_master_step_prescanned_ex(*bad) == fp8mp.ERR_INVALID, (i, v)
        assert word in fp8mp.last_error(), (i, v, fp8mp.last_error())
    # adam: grad, n, master, m, v, w8_in, w8_out, scale_w, amax_w, S, growth, found, gnf, beta_pows, lr, b1, b2,
    # eps, bo, gf, gi, flags
    adam = [P, n, P, P, P, 8 * P, 4 * P, P, P, P, P, P, 2 * P, P, 1e-4, 0.9, 0.999, 1e-8, 0.5, 2.0, 2000, 8, None]
    assert lib.mp_master_step_adam_prescanned_ex(*adam) == fp8mp.ERR_INVALID and "flags" in fp8mp.last_error()
    adam[21] = fp8mp.WAIT_DW_DONE  # the wait only makes sense beside the producer
    assert lib.mp_master_step_adam_prescanned_ex(*adam) == fp8mp.ERR_INVALID
    assert "OVERLAP_PREVIOUS" in fp8mp.last_error()
    adam[21], adam[5] = 1, 4 * P + 16
    assert lib.mp_master_step_adam_prescanned_ex(*adam) == fp8mp.ERR_INVALID and "overlap" in fp8mp.last_error()


def test_binding_routes_the_two_buffer_step(monkeypatch):
    """mp_master_step(w8_in=..., flags=...) calls the _ex entry point with
    the current copy before the new one, and refuses without grad_nonfinite."""
    import torch

    calls = []

    class FakeLib:
        def __getattr__(self, name):
            def f(*a):
                calls.append((name, a))
                return 0
            return f

    monkeypatch.setattr(fp8mp, "_lib", FakeLib())
    t = {k: torch.zeros(16, dtype=torch.float32) for k in ("g", "w", "v", "s", "a", "S", "gr", "f", "nf")}
    w8, w8_in = torch.zeros(16, dtype=torch.uint8), torch.ones(16, dtype=torch.uint8)
    fp8mp.mp_master_step(t["g"], t["w"], t["v"], w8, t["s"], t["a"], t["S"], t["gr"], t["f"], 0.1, 0.9,
                         stream=0, grad_nonfinite=t["nf"], w8_in=w8_in, flags=fp8mp.OVERLAP_PREVIOUS)
    name, a = calls[-1]
    assert name == "mp_master_step_prescanned_ex"
    assert a[4] == w8_in.data_ptr() and a[5] == w8.data_ptr() and a[17] == fp8mp.OVERLAP_PREVIOUS
    with pytest.raises(fp8mp.Fp8mpError):
        fp8mp.mp_master_step(t["g"], t["w"], t["v"], w8, t["s"], t["a"], t["S"], t["gr"], t["f"], 0.1, 0.9,
                             stream=0, w8_in=w8_in)
    snap = torch.zeros(4, dtype=torch.float32)
    fp8mp.delayed_scaling_update([], fp8mp.AMAX_MAX, 0, stream=0, prev_scale_inv=snap)
    assert calls[-1][0] == "delayed_scaling_update_ex" and calls[-1][1][4] == snap.data_ptr()


def test_bwd_rowmajor_ex_rejects_bad_flags(lib):
    """Unknown flags, and the completion signal without dW or without its
    overflow word, are refused before any CUDA call."""
    P = 4096
    args = [P, P, P, 256, 256, 256, 1, P, P, P, P, 1, 2 * P, 1, 3 * P]
    assert lib.fp8_linear_bwd_rowmajor_ex(*args, 8, None) == fp8mp.ERR_INVALID and "flags" in fp8mp.last_error()
    no_word = list(args)
    no_word[14] = None
    assert lib.fp8_linear_bwd_rowmajor_ex(*no_word, fp8mp.SIGNAL_DW_DONE, None) == fp8mp.ERR_INVALID
    assert "dw_nonfinite" in fp8mp.last_error()
    no_dw = list(args)
    no_dw[12] = None
    assert lib.fp8_linear_bwd_rowmajor_ex(*no_dw, fp8mp.SIGNAL_DW_DONE, None) == fp8mp.ERR_INVALID


def test_scaling_master_step_validation(lib):
    """mp_master_step_prescanned_scaling_ex and its Adam form refuse, before
    any CUDA call: other flags than OVERLAP_PREVIOUS | WAIT_DW_DONE, more than
    8 metas, a bad meta, a weight meta (the one holding scale_w) whose
    cur_amax is not amax_w, and two metas holding scale_w."""
    P = 4096  # fake aligned addresses, never dereferenced: validation fails first
    both = fp8mp.OVERLAP_PREVIOUS | fp8mp.WAIT_DW_DONE
    scale_w, amax_w = 64 * P, 65 * P

    def metas(*specs):
        arr = (fp8mp.fp8mp_meta * max(1, len(specs)))()
        for i, (scale, amax, L) in enumerate(specs):
            arr[i] = fp8mp.fp8mp_meta(P * (100 + 8 * i), scale, P * (102 + 8 * i), amax, L, fp8mp.E4M3)
        return arr

    def sgd(arr, n_metas, flags=both, algo=fp8mp.AMAX_MOST_RECENT, margin=0):
        return lib.mp_master_step_prescanned_scaling_ex(P, 64, P, P, 8 * P, 4 * P, scale_w, amax_w, P, P, 9 * P,
                                                        10 * P, 1e-4, 0.9, 0.5, 2.0, 2000, arr, n_metas, algo,
                                                        margin, flags, None)

    ok = metas((P * 200, P * 201, 16), (scale_w, amax_w, 16))
    cases = [
        (lambda: sgd(ok, 2, flags=fp8mp.OVERLAP_PREVIOUS), "flags must be"),
        (lambda: sgd(ok, 9), "n_metas"),
        (lambda: sgd(ok, 2, algo=5), "algo"),
        (lambda: sgd(ok, 2, margin=200), "margin"),
        (lambda: sgd(metas((P * 200, P * 201, 0)), 1), "history_len"),
        (lambda: sgd(metas((scale_w, P * 201, 16)), 1), "must hold amax_w"),
        (lambda: sgd(metas((scale_w, amax_w, 16), (scale_w, amax_w, 16)), 2), "two metas"),
        (lambda: sgd(metas((P * 200, amax_w, 16)), 1), "holds amax_w but not scale_w"),
    ]
    for i, (fn, word) in enumerate(cases):
        assert fn() == fp8mp.ERR_INVALID, i
        assert word in fp8mp.last_error(), (i, fp8mp.last_error())
    adam = lib.mp_master_step_adam_prescanned_scaling_ex(P, 64, P, P, P, 8 * P, 4 * P, scale_w, amax_w, P, P, 9 * P,
                                                          10 * P, P, 1e-4, 0.9, 0.999, 1e-8, 0.5, 2.0, 2000, ok, 9,
                                                          fp8mp.AMAX_MOST_RECENT, 0, both, None)
    assert adam == fp8mp.ERR_INVALID and "n_metas" in fp8mp.last_error()


def test_binding_routes_the_scaling_step(monkeypatch):
    """mp_master_step(metas=...) calls mp_master_step_prescanned_scaling_ex
    with the metas' array, their count, the algorithm, margin and flags."""
    import torch

    calls = []

    class FakeLib:
        def __getattr__(self, name):
            def f(*a):
                calls.append((name, a))
                return 0
            return f

    monkeypatch.setattr(fp8mp, "_lib", FakeLib())
    t = {k: torch.zeros(16, dtype=torch.float32) for k in ("g", "w", "v", "s", "a", "S", "gr", "f", "nf")}
    w8, w8_in = torch.zeros(16, dtype=torch.uint8), torch.ones(16, dtype=torch.uint8)
    ms = [fp8mp.Meta(4, fp8mp.E4M3, device="cpu") for _ in range(3)]
    flags = fp8mp.OVERLAP_PREVIOUS | fp8mp.WAIT_DW_DONE
    fp8mp.mp_master_step(t["g"], t["w"], t["v"], w8, t["s"], t["a"], t["S"], t["gr"], t["f"], 0.1, 0.9,
                         stream=0, grad_nonfinite=t["nf"], w8_in=w8_in, flags=flags, metas=ms,
                         amax_algo=fp8mp.AMAX_MAX, margin=2)
    name, a = calls[-1]
    assert name == "mp_master_step_prescanned_scaling_ex"
    assert a[4] == w8_in.data_ptr() and a[5] == w8.data_ptr()
    assert a[17][1].scale == ms[1].scale.data_ptr() and a[18:22] == (3, fp8mp.AMAX_MAX, 2, flags)
    with pytest.raises(fp8mp.Fp8mpError):
        fp8mp.mp_master_step(t["g"], t["w"], t["v"], w8, t["s"], t["a"], t["S"], t["gr"], t["f"], 0.1, 0.9,
                             stream=0, metas=ms)
