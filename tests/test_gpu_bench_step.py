"""The benchmark's training step (bench.LinearStep) against the oracle, on a
small instance of the proj-linear workload, over three steps.

The step casts x and dY row-major only, runs the forward GEMM on the weight's
E4M3 copy, both backward GEMMs from the row-major copies in one launch, the
delayed-scaling update, then the master step, which re-casts the weight's
E4M3 copy under the just-updated weight scale for the next step. Checked
here: every code and every meta bit-exact; GEMM outputs within the GEMM
tolerance; the master step bit-exact on the GPU's own bf16 dW (dW is the
master step's input, and its rounding is not unique)."""

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


def test_bench_step_matches_oracle(cuda_lib, orc):
    M, K, N = 384, 512, 256  # N <= K: the step takes dY's first N columns
    st = bench.LinearStep(m=M, k=K, n=N)
    xn, dyn = np_view(st.x), np_view(st.dy)
    w = np_view(st.master).copy()
    mom = np.zeros_like(w)
    om = [orc.Meta(bench.HIST_LEN) for _ in range(4)]
    ox, ow, oy, od = om
    # the weight's first copy, made when the step object was built
    w8 = bench.oracle_initial_weight_copy(orc, w, om)
    torch.cuda.synchronize()
    assert_same_bits(st.W8.cpu().numpy().reshape(-1), w8, "initial W8")
    meta_equal(st.mw, ow, "initial w")
    ls = orc.LossScaleState(bench.S0)
    for step in range(3):
        st.step()
        assert cuda_lib.fp8mp_check() == 0
        torch.cuda.synchronize()
        # casts (with this step's scales) and their amaxes
        X8 = orc.cast(xn, float(ox.scale[0]), E4M3)
        D8 = orc.cast(dyn, float(od.scale[0]), E5M2)
        assert_same_bits(st.X8.cpu().numpy(), X8, f"step {step} X8")
        assert_same_bits(st.D8.cpu().numpy(), D8, f"step {step} dY8")
        ox.record_amax(orc.amax(xn))
        od.record_amax(orc.amax(dyn))
        W8 = w8.reshape(N, K)
        sx, sw, sd = (float(m.scale_inv[0]) for m in (ox, ow, od))
        y = np_view(st.y.float()).astype(np.float64)
        ref, ab = orc.gemm_ref(X8, E4M3, W8, E4M3, sx, sw)
        gemm_tolerance_check(y, ref, ab, f"step {step} y")
        oy.record_amax(np.float32(np.abs(y).max()))  # amax of the stored output
        ref, ab = orc.gemm_ref(D8, E5M2, orc.transpose_u8(W8), E4M3, sd, sw)
        gemm_tolerance_check(np_view(st.dx.float()).astype(np.float64), ref, ab, f"step {step} dx")
        ref, ab = orc.gemm_ref(orc.transpose_u8(D8), E5M2, orc.transpose_u8(X8), E4M3, sd, sx)
        gemm_tolerance_check(np_view(st.dw.float()).astype(np.float64), ref, ab, f"step {step} dw")
        # the update, then the master step on the GPU's dW under the new weight scale
        for m, f in zip(om, (E4M3, E4M3, E4M3, E5M2)):
            orc.scale_update(m, f, orc.AMAX_MOST_RECENT, 0)
        g = st.dw.reshape(-1).cpu().view(torch.int16).numpy().view(np.uint16)
        orc.master_step(g, w.reshape(-1), mom.reshape(-1), w8, float(ow.scale[0]), ow.cur_amax, ls,
                        bench.LR, bench.MU)
        assert_same_bits(np_view(st.master).reshape(-1), w.reshape(-1), f"step {step} master")
        assert_same_bits(np_view(st.mom).reshape(-1), mom.reshape(-1), f"step {step} momentum")
        assert_same_bits(st.W8.cpu().numpy().reshape(-1), w8, f"step {step} next W8")
        for dm_, om_, name in zip((st.mx, st.mw, st.my, st.md), om, "xwyd"):
            meta_equal(dm_, om_, f"step {step} meta {name}")
        assert st.S.item() == ls.S[0] and st.growth.item() == ls.growth[0]
