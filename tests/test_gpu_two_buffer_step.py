"""The pieces of the step whose master step runs beside the dgrad GEMM:
delayed_scaling_update_ex (the update that keeps each tensor's previous
scale_inv) and the two-buffer master steps (mp_master_step_prescanned_ex and
its Adam form), in place of the serial order's update-after-backward and
in-place re-cast. Checked: the snapshot is the old scale_inv and the update
is bitwise the plain one's; the steps are bit-exact against the oracle with
the new E4M3 copy in the other buffer (a skipped step copies the current one
there) and the current copy untouched; enqueued with FP8MP_OVERLAP_PREVIOUS
behind a long GEMM, the results are the same and what follows the step sees
the GEMM's results."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, E5M2, assert_same_bits, np_view

pytestmark = pytest.mark.gpu


def test_scale_update_keeps_the_previous_scale_inv(cuda_lib):
    g = torch.Generator(device="cuda").manual_seed(5)
    fmts = (E4M3, E4M3, E4M3, E5M2)
    a = [cuda_lib.Meta(16, f) for f in fmts]
    b = [cuda_lib.Meta(16, f) for f in fmts]
    for t in range(3):  # histories, scales and scale_inv away from their initial 1.0
        for ma, mb in zip(a, b):
            v = torch.rand(1, generator=g, device="cuda") * 10 ** (t - 1)
            ma.cur_amax.copy_(v)
            mb.cur_amax.copy_(v)
        old = torch.cat([m.scale_inv for m in a]).clone()
        snap = torch.full((4,), -1.0, device="cuda")
        cuda_lib.delayed_scaling_update(a, cuda_lib.AMAX_MAX, 1, prev_scale_inv=snap)
        cuda_lib.delayed_scaling_update(b, cuda_lib.AMAX_MAX, 1)
        assert cuda_lib.fp8mp_check() == 0
        assert_same_bits(np_view(snap), np_view(old), f"snapshot {t}")
        for i, (ma, mb) in enumerate(zip(a, b)):
            for name in ("amax_history", "scale", "scale_inv", "cur_amax"):
                assert_same_bits(np_view(getattr(ma, name)), np_view(getattr(mb, name)), f"{t} meta {i} {name}")


class State:
    def __init__(self, w, opt):
        n = w.numel()
        self.w = w.cuda().clone()
        self.v = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.m = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.bp = torch.ones(2, dtype=torch.float32, device="cuda")
        # two copies with distinct junk, so a missing write or copy shows
        self.w8 = [torch.full((n,), 0x11, dtype=torch.uint8, device="cuda"),
                   torch.full((n,), 0x22, dtype=torch.uint8, device="cuda")]
        self.scale_w = torch.tensor([32.0], device="cuda")
        self.amax_w = torch.zeros(1, device="cuda")
        self.S = torch.tensor([2.0 ** 16], device="cuda")
        self.growth = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.found = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.opt = opt

    def step(self, f, g, w8_in, w8_out, flags):
        if self.opt == "sgd":
            f.mp_master_step(g, self.w, self.v, w8_out, self.scale_w, self.amax_w, self.S, self.growth, self.found,
                             1e-4, 0.9, grad_nonfinite=self.flag, w8_in=w8_in, flags=flags)
        else:
            f.mp_master_step_adam(g, self.w, self.m, self.v, w8_out, self.scale_w, self.amax_w, self.S,
                                  self.growth, self.found, self.bp, lr=1e-3, grad_nonfinite=self.flag,
                                  w8_in=w8_in, flags=flags)


def long_gemm(f):
    """A forward GEMM of about 0.3 ms on buffers the step does not touch,
    and a meta whose cur_amax is its output amax."""
    g = torch.Generator(device="cuda").manual_seed(3)
    M = K = N = 8192
    x8 = (torch.randn(M, K, generator=g, device="cuda") * 4).to(torch.float8_e4m3fn).view(torch.uint8)
    w8 = (torch.randn(N, K, generator=g, device="cuda") * 0.1).to(torch.float8_e4m3fn).view(torch.uint8)
    one = torch.ones(1, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ref = torch.zeros(1, device="cuda")
    f.fp8_linear_fwd(x8, w8, one, one, y, y_amax=ref)
    torch.cuda.synchronize()
    meta = f.Meta(4, E4M3)

    def run():
        meta.cur_amax.zero_()
        f.fp8_linear_fwd(x8, w8, one, one, y, y_amax=meta.cur_amax)

    return run, meta, ref


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("opt", ["sgd", "adam"])
@pytest.mark.parametrize("n", [1, 9, 4096, (1 << 20) + 3])
def test_two_buffer_steps_bit_exact(cuda_lib, orc, opt, n, overlap):
    f = cuda_lib
    w = workloads.master_weights(n, seed=n + 11)
    ds = State(w, opt)
    hw, hv, hm = np_view(w).copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    h8, ham = np.zeros(n, np.uint8), np.zeros(1, np.float32)
    st, ad = orc.LossScaleState(2.0 ** 16, 0), orc.AdamState()
    gemm = long_gemm(f) if overlap else None
    cur = 0
    prev8 = ds.w8[0].cpu().numpy()
    for step in range(4):
        g = workloads.master_step(n, step, seed=n + 11, inject=(step == 2), inject_frac=1e-3)
        gb = np_view(g)
        ds.flag.fill_(int(((gb & 0x7F80) == 0x7F80).any()))
        gd = g.cuda()
        torch.cuda.synchronize()
        if overlap:
            gemm[0]()
        ds.step(f, gd, ds.w8[cur], ds.w8[cur ^ 1], f.OVERLAP_PREVIOUS if overlap else 0)
        if overlap:  # enqueued after the step: must see the GEMM's output amax
            f.delayed_scaling_update([gemm[1]], f.AMAX_MOST_RECENT, 0)
        assert f.fp8mp_check() == 0
        if opt == "sgd":
            orc.master_step(gb, hw, hv, h8, 32.0, ham, st, 1e-4, 0.9)
        else:
            orc.adam_step(gb, hw, hm, hv, h8, 32.0, ham, st, ad, lr=1e-3)
        what = f"{opt} n={n} step={step} overlap={overlap}"
        assert_same_bits(np_view(ds.w), hw, what + " master")
        assert_same_bits(np_view(ds.v), hv, what + " v")
        if opt == "adam":
            assert_same_bits(np_view(ds.m), hm, what + " exp_avg")
        assert_same_bits(ds.w8[cur ^ 1].cpu().numpy(), h8, what + " next copy")
        assert_same_bits(ds.w8[cur].cpu().numpy(), prev8, what + " current copy untouched")
        assert_same_bits(np_view(ds.amax_w), ham, what + " amax")
        assert ds.S.item() == st.S[0] and ds.growth.item() == st.growth[0]
        assert ds.found.item() == st.found_inf[0] == int(step == 2) and ds.flag.item() == 0
        if overlap:
            assert_same_bits(np_view(gemm[1].amax_history[:1]), np_view(gemm[2]), what + " GEMM amax seen")
        prev8 = h8.copy()
        cur ^= 1


def test_two_buffer_step_in_place_is_the_plain_step(cuda_lib, orc):
    """w8_in == w8_out is the in-place step (and NULL w8_in with
    OVERLAP_PREVIOUS too): same bits as the oracle."""
    f = cuda_lib
    n = 40961
    w = workloads.master_weights(n, seed=2)
    ds = State(w, "sgd")
    hw, hv, h8, ham = np_view(w).copy(), np.zeros(n, np.float32), np.zeros(n, np.uint8), np.zeros(1, np.float32)
    st = orc.LossScaleState(2.0 ** 16, 0)
    for step in range(3):
        g = workloads.master_step(n, step, seed=2, inject=(step == 1), inject_frac=1e-3)
        gb = np_view(g)
        ds.flag.fill_(int(((gb & 0x7F80) == 0x7F80).any()))
        ds.step(f, g.cuda(), ds.w8[0] if step != 2 else None, ds.w8[0], f.OVERLAP_PREVIOUS if step == 2 else 0)
        assert f.fp8mp_check() == 0
        orc.master_step(gb, hw, hv, h8, 32.0, ham, st, 1e-4, 0.9)
        assert_same_bits(np_view(ds.w), hw, f"step {step} master")
        assert_same_bits(ds.w8[0].cpu().numpy(), h8, f"step {step} copy")  # a skip leaves it as it was


@pytest.mark.parametrize("shape", [(384, 256, 512), (2048, 1024, 1024), (0, 256, 512)])
def test_backward_signals_dw_completion(cuda_lib, shape):
    """fp8_linear_bwd_rowmajor_ex with FP8MP_SIGNAL_DW_DONE: the same dX and
    dW as the plain launch, bit 30 of the word set once dW is stored (at once
    for an empty contraction), bit 0 the overflow flag of the stored dW."""
    f = cuda_lib
    M, N, K = shape
    g = torch.Generator(device="cuda").manual_seed(M + N + K)
    d8 = (torch.randn(M, N, generator=g, device="cuda") * 8).to(torch.float8_e5m2).view(torch.uint8)
    w8 = torch.randn(N, K, generator=g, device="cuda").to(torch.float8_e4m3fn).view(torch.uint8)
    x8 = torch.randn(M, K, generator=g, device="cuda").to(torch.float8_e4m3fn).view(torch.uint8)
    if M > 0:
        d8[M // 2, N // 3] = 0x7F  # an E5M2 NaN code: NaN in one dW row
    one = torch.ones(1, device="cuda")
    outs = []
    for flags in (0, f.SIGNAL_DW_DONE):
        dx = torch.full((M, K), 7.0, dtype=torch.bfloat16, device="cuda")
        dw = torch.full((N, K), 7.0, dtype=torch.bfloat16, device="cuda")
        word = torch.zeros(1, dtype=torch.int32, device="cuda")
        f.fp8_linear_bwd_rowmajor(d8, w8, x8, one, one, one, dx, dw, dw_nonfinite=word, flags=flags)
        assert f.fp8mp_check() == 0
        outs.append((dx, dw, int(word.item())))
    (dx0, dw0, w0), (dx1, dw1, w1) = outs
    assert torch.equal(dx0.view(torch.int16), dx1.view(torch.int16))
    assert torch.equal(dw0.view(torch.int16), dw1.view(torch.int16))
    bad = int(not torch.isfinite(dw0.float()).all())
    assert w0 == bad
    assert w1 & (1 << 30) and (w1 & 1) == bad
    assert (w1 >> 1) & 0x7FFF == 0  # no master step counted in it


def test_waiting_master_step_times_out_without_a_signal(cuda_lib):
    """FP8MP_WAIT_DW_DONE behind a kernel that never signals: each block's
    bounded wait runs out (about 2 s), fp8mp_check reports the timeout, the
    step updates nothing and the word is left at 0."""
    f = cuda_lib
    n = 4096
    ds = State(workloads.master_weights(n, seed=9), "sgd")
    w_before = ds.w.clone()
    torch.zeros(16, device="cuda").add_(1.0)  # some earlier kernel on the stream
    ds.step(f, torch.zeros(n, dtype=torch.int16, device="cuda"), ds.w8[0], ds.w8[1],
            f.OVERLAP_PREVIOUS | f.WAIT_DW_DONE)
    assert f.fp8mp_check() == f.ERR_TIMEOUT
    assert torch.equal(ds.w.view(torch.int32), w_before.view(torch.int32))
    assert ds.flag.item() == 0
    assert f.fp8mp_check() == 0  # the flag was cleared by the first check


DONE_BIT = 1 << 30


def make_metas(f, lens, fmts, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    ms = []
    for L, fm in zip(lens, fmts):
        m = f.Meta(L, fm)
        m.amax_history.copy_(torch.rand(L, generator=g, device="cuda") * 100.0)
        m.scale.copy_(torch.rand(1, generator=g, device="cuda") * 8.0 + 0.5)
        m.scale_inv.copy_(1.0 / m.scale)
        m.cur_amax.copy_(torch.rand(1, generator=g, device="cuda") * 50.0)
        ms.append(m)
    return ms


def clone_metas(f, ms):
    out = []
    for m in ms:
        c = f.Meta(m.amax_history.numel(), m.fmt)
        for name in ("amax_history", "scale", "scale_inv", "cur_amax"):
            getattr(c, name).copy_(getattr(m, name))
        out.append(c)
    return out


@pytest.mark.parametrize("opt", ["sgd", "adam"])
@pytest.mark.parametrize("n,lens,w_at,skip", [
    (1 << 20, (1024, 1024, 1024, 1024), 1, False),   # the bench step's four metas, the weight's second
    (1 << 20, (1024, 1024, 1024, 1024), 1, True),    # a skipped step still updates the metas
    (4096, (1, 3, 8192, 513, 7, 1024, 2, 600), 5, False),  # one block runs all eight metas
    (9, (5,), -1, False),                            # no weight meta: the step casts with scale_w as it is
    ((1 << 20) + 3, (), -1, False),                  # no metas: the _ex step
])
def test_folded_update_is_the_separate_update_then_the_step(cuda_lib, opt, n, lens, w_at, skip):
    """mp_master_step_prescanned_scaling_ex (and its Adam form) against
    delayed_scaling_update_ex followed by the _ex step on copies of the same
    state, both behind a word that already holds the completion bit: every
    history, scale, scale_inv and cur_amax, the master weights and moments,
    the new E4M3 copy, the loss scale, growth counter and found_inf agree bit
    for bit, and the word is back at 0."""
    f = cuda_lib
    fmts = tuple(E5M2 if i % 4 == 3 else E4M3 for i in range(len(lens)))
    w = workloads.master_weights(n, seed=n + 5)
    g = workloads.master_step(n, 1, seed=n + 5, inject=skip, inject_frac=1e-3).cuda()
    bad = int(((np_view(g.cpu()) & 0x7F80) == 0x7F80).any())
    assert bad == int(skip)
    runs = []
    for fold in (False, True):
        ds = State(w, opt)
        metas = make_metas(f, lens, fmts, seed=17)
        if w_at >= 0:  # the weight's meta holds the step's scale_w and amax_w
            ds.scale_w = metas[w_at].scale
            ds.amax_w = metas[w_at].cur_amax
        ds.flag.fill_(DONE_BIT | bad)
        flags = f.OVERLAP_PREVIOUS | f.WAIT_DW_DONE
        if fold:
            if opt == "sgd":
                f.mp_master_step(g, ds.w, ds.v, ds.w8[1], ds.scale_w, ds.amax_w, ds.S, ds.growth, ds.found, 1e-4,
                                 0.9, grad_nonfinite=ds.flag, w8_in=ds.w8[0], flags=flags, metas=metas,
                                 amax_algo=f.AMAX_MAX, margin=1)
            else:
                f.mp_master_step_adam(g, ds.w, ds.m, ds.v, ds.w8[1], ds.scale_w, ds.amax_w, ds.S, ds.growth,
                                      ds.found, ds.bp, lr=1e-3, grad_nonfinite=ds.flag, w8_in=ds.w8[0], flags=flags,
                                      metas=metas, amax_algo=f.AMAX_MAX, margin=1)
        else:
            if metas:
                snap = torch.zeros(len(metas), device="cuda")
                f.delayed_scaling_update(metas, f.AMAX_MAX, 1, prev_scale_inv=snap)
            ds.step(f, g, ds.w8[0], ds.w8[1], flags)
        assert f.fp8mp_check() == 0, f.last_error()
        runs.append((ds, metas))
    (a, ma), (b, mb) = runs
    for name in ("w", "v", "m", "bp", "S", "growth", "found", "amax_w", "flag"):
        assert_same_bits(np_view(getattr(b, name)), np_view(getattr(a, name)), name)
    assert int(b.flag.item()) == 0 and int(b.found.item()) == int(skip)
    assert torch.equal(b.w8[1], a.w8[1]) and torch.equal(b.w8[0], a.w8[0])
    for i, (x, y) in enumerate(zip(mb, ma)):
        for name in ("amax_history", "scale", "scale_inv", "cur_amax"):
            assert_same_bits(np_view(getattr(x, name)), np_view(getattr(y, name)), f"meta {i} {name}")


def test_folded_update_validation(cuda_lib):
    f = cuda_lib
    ds = State(workloads.master_weights(64, seed=1), "sgd")
    g = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    metas = make_metas(f, (4, 4), (E4M3, E4M3), seed=3)
    both = f.OVERLAP_PREVIOUS | f.WAIT_DW_DONE

    def call(ms, flags, scale_w=None, amax_w=None):
        f.mp_master_step(g, ds.w, ds.v, ds.w8[1], ds.scale_w if scale_w is None else scale_w,
                         ds.amax_w if amax_w is None else amax_w, ds.S, ds.growth, ds.found, 1e-4, 0.9,
                         grad_nonfinite=ds.flag, w8_in=ds.w8[0], flags=flags, metas=ms)

    with pytest.raises(cuda_lib.Fp8mpError, match="flags must be"):
        call(metas, f.OVERLAP_PREVIOUS)
    with pytest.raises(cuda_lib.Fp8mpError, match="n_metas"):
        call(make_metas(f, (2,) * 9, (E4M3,) * 9, seed=4), both)
    with pytest.raises(cuda_lib.Fp8mpError, match="must hold amax_w"):
        call(metas, both, scale_w=metas[0].scale)
    twin = make_metas(f, (4,), (E4M3,), seed=5)[0]
    twin.scale = metas[0].scale
    with pytest.raises(cuda_lib.Fp8mpError, match="two metas"):
        call([metas[0], twin], both, scale_w=metas[0].scale, amax_w=metas[0].cur_amax)
