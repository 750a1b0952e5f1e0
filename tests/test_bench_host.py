"""Host logic of bench.py on the CPU: the max-over-ranks timing reduction and
barrier on a world-size-2 gloo group, rank gating of the reference arm, the
clock-sample parsing, and the ncu-summary lookup that keys traffic to the
GEMM source it was measured on."""

import hashlib
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    v = bench.max_over_ranks(1.5 + 10 * rank, world)
    out.put((rank, v))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 11.5, 1: 11.5}


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_only_on_rank_zero():
    class A:
        cpu_tokens, steps, warmup = 16, 1, 3

    assert bench.run_reference(A(), world=2, rank=1) is None


def test_flops_per_step():
    assert bench.flops_per_step() == 3 * 2 * 8192 * 4096 * 4096


def test_clock_summary_flags_throttle():
    cs = bench.ClockSampler(0)
    cs.lines = ["1455, 2070, 900.1, Not Active, Not Active, Not Active, Active",
                "1500, 2070, 950.0, Not Active, Active, Not Active, Not Active",
                "garbage"]
    s = cs.summary()
    assert s["sm_mhz"] == pytest.approx(1477.5) and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_traffic_lookup_is_keyed_to_the_gemm_source(tmp_path, monkeypatch):
    src = tmp_path / "gemm.cu"
    src.write_text("kernel v1")
    prof = tmp_path / "prof.md"
    sha = hashlib.sha256(b"kernel v1").hexdigest()
    prof.write_text(f"- gemm_cu_sha256: `{sha}`\n- dram_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "GEMM_SRC", str(src))
    monkeypatch.setattr(bench, "PROFILE", str(prof))
    assert bench.gemm_traffic_from_profile() == 123456.0
    src.write_text("kernel v2")  # the kernel changed since the capture
    assert bench.gemm_traffic_from_profile() is None
