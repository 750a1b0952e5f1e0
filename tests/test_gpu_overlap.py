"""A cast enqueued with FP8MP_OVERLAP_PREVIOUS right behind a long forward
GEMM on the same stream (the cast may run while the GEMM does): its codes
and amax are exactly the plain cast's, and what is enqueued after it sees
the GEMM's results too (the grid completes after the GEMM's)."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import E4M3, E5M2, assert_same_bits, np_view

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("transposed", [False, True])
def test_overlapped_cast_behind_a_gemm(cuda_lib, orc, transposed):
    g = torch.Generator(device="cuda").manual_seed(11)
    M = K = N = 8192  # a forward GEMM of about 0.3 ms
    x8 = (torch.randn(M, K, generator=g, device="cuda") * 4).to(torch.float8_e4m3fn).view(torch.uint8)
    w8 = (torch.randn(N, K, generator=g, device="cuda") * 0.1).to(torch.float8_e4m3fn).view(torch.uint8)
    one = torch.ones(1, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    rows, cols = 8192, 4096
    dy = (torch.randn((rows, cols), generator=workloads.gen(99)) * 1e-3).to(torch.bfloat16).cuda()
    scale = torch.tensor([8192.0], device="cuda")
    meta_y = cuda_lib.Meta(16, E4M3)
    ref_amax_y = torch.zeros(1, device="cuda")
    cuda_lib.fp8_linear_fwd(x8, w8, one, one, y, y_amax=ref_amax_y)
    torch.cuda.synchronize()
    for call in range(3):
        out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda") if transposed else None
        am = torch.zeros(1, device="cuda")
        meta_y.cur_amax.zero_()
        cuda_lib.fp8_linear_fwd(x8, w8, one, one, y, y_amax=meta_y.cur_amax)
        cuda_lib.fp8_quantize_ex(dy, E5M2, scale, out, out_t, am, flags=cuda_lib.OVERLAP_PREVIOUS)
        # enqueued after the overlapped cast: must see the GEMM's output amax
        cuda_lib.delayed_scaling_update([meta_y], cuda_lib.AMAX_MOST_RECENT, 0)
        assert cuda_lib.fp8mp_check() == 0
        q = orc.cast(np_view(dy), 8192.0, E5M2)
        assert_same_bits(out.cpu().numpy(), q, f"codes {call}")
        if transposed:
            assert_same_bits(out_t.cpu().numpy(), orc.transpose_u8(q), f"transposed {call}")
        assert_same_bits(np_view(am), np.array([orc.amax(np_view(dy))], np.float32), "amax")
        assert_same_bits(np_view(meta_y.amax_history[:1]), np_view(ref_amax_y), f"history sees the GEMM's amax {call}")
