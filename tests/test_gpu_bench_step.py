"""The benchmark's training step (bench.LinearStep) against the oracle: a
small instance over three steps, and the full proj-linear workload (M = 8192,
K = N = 4096) over an eager step and steps replayed from the CUDA graphs
bench.py times.

The step casts x and dY row-major only, runs the forward GEMM on the weight's
E4M3 copy, the backward GEMMs from the row-major copies, the delayed-scaling
update and the master step, which re-casts the weight's E4M3 copy under the
just-updated weight scale for the next step. Both schedules are checked: the
serial one (one-launch backward, update, master step in place) and the
overlapped one the bench times (update first, keeping the casts' scale_inv
for the backward; the backward launch signals when dW is stored, and the
master step, started beside it, waits for that signal and writes the other
of two weight copies). Checked here: every code and every meta
bit-exact; every GEMM output within the GEMM tolerance; the master step
bit-exact on the GPU's own bf16 dW (dW is the master step's input, and its
rounding is not unique)."""

import numpy as np
import pytest
import torch

import bench
from gpu_util import E4M3, E5M2, assert_same_bits, gemm_tolerance_check, np_view

pytestmark = pytest.mark.gpu


def meta_equal(dm, om, what):
    assert_same_bits(np_view(dm.amax_history), om.hist, what + " history")
    assert_same_bits(np_view(dm.scale), om.scale, what + " scale")
    assert_same_bits(np_view(dm.scale_inv), om.scale_inv, what + " scale_inv")
    assert_same_bits(np_view(dm.cur_amax), om.cur_amax, what + " cur_amax")


class OracleRun:
    """The oracle's side of the step sequence, advanced one step at a time
    and compared with the GPU state after each step."""

    def __init__(self, orc, st):
        self.orc, self.st = orc, st
        self.xn, self.dyn = np_view(st.x), np_view(st.dy)
        self.w = np_view(st.master).copy()
        self.mom = np.zeros_like(self.w)
        self.om = [orc.Meta(bench.HIST_LEN) for _ in range(4)]
        # the weight's first copy, made when the step object was built
        self.w8 = bench.oracle_initial_weight_copy(orc, self.w, self.om)
        self.ls = orc.LossScaleState(bench.S0)
        torch.cuda.synchronize()
        assert_same_bits(st.W8.cpu().numpy().reshape(-1), self.w8, "initial W8")
        meta_equal(st.mw, self.om[1], "initial w")

    def check_step(self, label):
        orc, st = self.orc, self.st
        ox, ow, oy, od = self.om
        torch.cuda.synchronize()
        # casts (with this step's scales) and their amaxes
        X8 = orc.cast(self.xn, float(ox.scale[0]), E4M3)
        D8 = orc.cast(self.dyn, float(od.scale[0]), E5M2)
        assert_same_bits(st.X8.cpu().numpy(), X8, f"{label} X8")
        assert_same_bits(st.D8.cpu().numpy(), D8, f"{label} dY8")
        ox.record_amax(orc.amax(self.xn))
        od.record_amax(orc.amax(self.dyn))
        W8 = self.w8.reshape(st.n, st.k)
        sx, sw, sd = (float(m.scale_inv[0]) for m in (ox, ow, od))
        y = np_view(st.y.float()).astype(np.float64)
        ref, ab = orc.gemm_ref(X8, E4M3, W8, E4M3, sx, sw)
        gemm_tolerance_check(y, ref, ab, f"{label} y")
        oy.record_amax(np.float32(np.abs(y).max()))  # amax of the stored output
        del y, ref, ab
        ref, ab = orc.gemm_ref(D8, E5M2, orc.transpose_u8(W8), E4M3, sd, sw)
        gemm_tolerance_check(np_view(st.dx.float()).astype(np.float64), ref, ab, f"{label} dx")
        del ref, ab
        ref, ab = orc.gemm_ref(orc.transpose_u8(D8), E5M2, orc.transpose_u8(X8), E4M3, sd, sx)
        gemm_tolerance_check(np_view(st.dw.float()).astype(np.float64), ref, ab, f"{label} dw")
        del ref, ab
        # the update, then the master step on the GPU's dW under the new weight scale
        for m, f in zip(self.om, (E4M3, E4M3, E4M3, E5M2)):
            orc.scale_update(m, f, orc.AMAX_MOST_RECENT, 0)
        g = st.dw.reshape(-1).cpu().view(torch.int16).numpy().view(np.uint16)
        orc.master_step(g, self.w.reshape(-1), self.mom.reshape(-1), self.w8, float(ow.scale[0]), ow.cur_amax,
                        self.ls, bench.LR, bench.MU)
        assert_same_bits(np_view(st.master).reshape(-1), self.w.reshape(-1), f"{label} master")
        assert_same_bits(np_view(st.mom).reshape(-1), self.mom.reshape(-1), f"{label} momentum")
        assert_same_bits(st.W8.cpu().numpy().reshape(-1), self.w8, f"{label} next W8")
        for dm_, om_, name in zip((st.mx, st.mw, st.my, st.md), self.om, "xwyd"):
            meta_equal(dm_, om_, f"{label} meta {name}")
        assert st.S.item() == self.ls.S[0] and st.growth.item() == self.ls.growth[0]
        assert st.found.item() == self.ls.found_inf[0] == 0
        assert st.gnf.item() == 0  # dW's overflow flag, consumed and reset by the master step


@pytest.mark.parametrize("overlap", [True, False])
def test_bench_step_matches_oracle(cuda_lib, orc, overlap):
    M, K, N = 384, 512, 256  # N <= K: the step takes dY's first N columns
    st = bench.LinearStep(m=M, k=K, n=N, overlap=overlap)
    assert st.overlap_master == overlap
    run = OracleRun(orc, st)
    for step in range(3):
        st.step()
        assert cuda_lib.fp8mp_check() == 0
        run.check_step(f"step {step}")


@pytest.mark.slow
def test_bench_step_full_size_eager_then_graphs(cuda_lib, orc):
    """M = 8192, K = N = 4096, every output: one eager step, then steps
    replayed through bench.StepGraphs, the timed launches: the graph of each
    weight copy in turn (the master step beside dgrad writes the copy the
    other graph reads), then a graph with the GEMM timing events."""
    st = bench.LinearStep()
    run = OracleRun(orc, st)
    st.step()
    assert cuda_lib.fp8mp_check() == 0
    run.check_step("eager step")
    graphs = bench.StepGraphs(st, 1, upload=False)
    for label in ("graph of one copy", "graph of the other copy"):
        graphs.replay()
        assert cuda_lib.fp8mp_check() == 0
        run.check_step(label)
    graphs.replay_timed(0)
    assert cuda_lib.fp8mp_check() == 0
    run.check_step("timed graph")


def test_bench_step_skips_on_a_nan_gradient(cuda_lib):
    """A NaN in dY becomes an E5M2 NaN code, hence NaN in the stored dW; the
    wgrad epilogue flags it and the master step skips on the flag: master
    weights, momentum and W8 unchanged, S halved, growth reset, flag reset."""
    st = bench.LinearStep(m=256, k=512, n=256)
    assert st.overlap_master
    st.step()
    assert cuda_lib.fp8mp_check() == 0
    master, mom, w8 = st.master.clone(), st.mom.clone(), st.W8.clone()
    S, growth = st.S.item(), st.growth.item()
    assert growth == 1
    st.dy[17, 33] = float("nan")
    st.step()
    assert cuda_lib.fp8mp_check() == 0
    assert st.found.item() == 1 and st.gnf.item() == 0
    assert st.S.item() == S / 2 and st.growth.item() == 0
    assert torch.equal(st.master.view(torch.int32), master.view(torch.int32))
    assert torch.equal(st.mom.view(torch.int32), mom.view(torch.int32))
    assert torch.equal(st.W8, w8)
    assert not torch.isfinite(st.dw.float()).all()
