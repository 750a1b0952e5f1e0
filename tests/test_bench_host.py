"""Host logic of bench.py on the CPU: the max-over-ranks timing reduction and
barrier on a world-size-2 gloo group, rank gating of the reference arm, the
clock-sample parsing, the ncu CSV ingest, and the traffic lookup that keys
DRAM bytes to the GEMM source they were measured on."""

import hashlib
import json
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
    rec = tmp_path / "traffic.json"
    sha = hashlib.sha256(b"kernel v1").hexdigest()
    rec.write_text(json.dumps({"gemm_cu_sha256": sha, "dram_bytes_per_launch": {"fwd": 100.0, "bwd": 300.0}}))
    monkeypatch.setattr(bench, "GEMM_SRC", str(src))
    monkeypatch.setattr(bench, "TRAFFIC", str(rec))
    assert bench.gemm_traffic("fwd") == 100.0 and bench.gemm_traffic("bwd") == 300.0
    assert bench.gemm_traffic() == 200.0
    src.write_text("kernel v2")  # the kernel changed since the capture
    assert bench.gemm_traffic() is None and bench.gemm_traffic("fwd") is None
    rec.unlink()
    assert bench.gemm_traffic() is None


RAW_CSV = """"ID","Process ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum","gpu__time_duration.sum"
"","","","Mbyte","Kbyte","us"
"0","7","void fp8mp::gemm_fp8_kernel<1>(fp8mp::Params)","59.25","31,600.5","78.0"
"1","7","void fp8mp::cast_rows_kernel<1, 1>(const void *)","67.1","3,500.0","16.0"
"2","7","void fp8mp::gemm_fp8_kernel<1>(fp8mp::Params)","110.4","63,200","152.8"
"3","7","void fp8mp::gemm_fp8_kernel<1>(fp8mp::Params)","61.25","31,600.5","78.0"
"""

LONG_CSV = """"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Section Name","Metric Name","Metric Unit","Metric Value"
"4","7","python","box","gemm_fp8_kernel<1>","1","7","Command line profiler metrics","dram__bytes_read.sum","Gbyte","0.1104"
"4","7","python","box","gemm_fp8_kernel<1>","1","7","Command line profiler metrics","dram__bytes_write.sum","Mbyte","63.2"
"4","7","python","box","gemm_fp8_kernel<1>","1","7","Command line profiler metrics","gpu__time_duration.sum","us","152.8"
"""


def test_ncu_csv_ingest_both_exports(tmp_path, monkeypatch):
    """The GEMM launches' DRAM bytes are read from either ncu CSV export,
    units applied, other kernels skipped, launches labelled fwd / bwd in
    capture order; the record is keyed to the current gemm.cu."""
    raw = tmp_path / "raw.csv"
    raw.write_text(RAW_CSV)
    by, launches = bench.parse_ncu_dram_csv(str(raw))
    assert [e["label"] for e in launches] == ["fwd", "bwd", "fwd"]
    assert by["fwd"] == pytest.approx((59.25e6 + 31.6005e6 + 61.25e6 + 31.6005e6) / 2)
    assert by["bwd"] == pytest.approx(110.4e6 + 63.2e6)
    long = tmp_path / "long.csv"
    long.write_text(LONG_CSV)
    by2, launches2 = bench.parse_ncu_dram_csv(str(long), labels=("bwd",))
    assert by2 == {"bwd": pytest.approx(110.4e6 + 63.2e6)} and launches2[0]["id"] == 4
    out = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC", str(out))
    rec = bench.ingest_ncu(str(raw), "ncu ... python bench.py")
    assert rec["gemm_cu_sha256"] == bench.gemm_source_sha256()
    assert bench.gemm_traffic("bwd") == pytest.approx(173.6e6)
