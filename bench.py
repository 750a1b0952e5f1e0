#!/usr/bin/env python
"""Benchmark of the FP8 delayed-scaling linear layer on one GB300 per rank.

One step = one mixed-precision training step of the proj linear of the
transformer workload (M = 8192 tokens, K = N = 4096, bf16 activations with
0.1 % outliers, fp32 master weights ~ N(0, 0.02), bf16 output gradient), run
through the library's entry points on one CUDA stream:
  fp8_quantize(x -> X8, amax)                    E4M3, row-major only
  fp8_linear_fwd(X8, W8 -> Y bf16, amax_y)       W8: the weight's E4M3 copy
  fp8_quantize_ex(dY -> dY8, amax,               E5M2, row-major only; dY is an
                  FP8MP_OVERLAP_PREVIOUS)        input of the step, so its cast runs
                                                 beside the forward GEMM
  fp8_linear_bwd_rowmajor_ex(dY8, W8, X8          dgrad and wgrad GEMMs in one launch
      -> dX bf16, dW bf16; SIGNAL_DW_DONE)       from the row-major copies, wgrad
                                                 tiles first; the epilogue flags an
                                                 Inf/NaN in the stored dW and signals
                                                 when dW is complete
  mp_master_step_prescanned_scaling_ex(dW ->     SGD-momentum, loss scale 2^16,
      master, momentum, next W8; x, w, y, dy     started beside the backward launch;
      metas; OVERLAP_PREVIOUS | WAIT_DW_DONE)    its blocks first run the delayed-
                                                 scaling update of the four metas
                                                 (L = 1024, most_recent; the new
                                                 scale_inv written once the backward
                                                 launch, which reads the old ones, is
                                                 complete), then wait for that signal;
                                                 skip decided by the flag; re-casts the
                                                 weight under the updated scale into
                                                 the other of two W8 buffers while
                                                 dgrad still reads this step's
The weight's first E4M3 copy is cast once before the first step; from then
on each step's master step writes the next step's W8 (and records the amax
of the new master weights for the next scale update), so the weight is cast
once per optimizer step, inside the fused update pass. The results are
bitwise those of the serial order (the backward, then the update, then the
master step in place), which --no-overlap times.
The metric counts the FLOPs the FP8 tensor cores perform, 3 * 2 * M * N * K,
per step time. Multi-GPU runs are independent replicas (weak scaling).

The timed steps replay CUDA graphs of those library calls (captured after the
eager warm-up; one per W8 buffer, replayed in turn), as a training loop that
captures its step would; --eager
launches every call from Python instead. The step time comes from K steps
with nothing between the step's kernels; the GEMM launch durations of the
roofline come from K more steps with timing events around the GEMM launches
(an event between two kernels serialises them and costs the step ~20 us).

--impl reference times the CPU oracle on a bounded sample of the same step.
--kernels prints, instead of the step's line, one line per kernel timed alone
at the other workloads' sizes against its roofline (--only selects some).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_TOK, K_IN, N_OUT = 8192, 4096, 4096
HIST_LEN = 1024
LR, MU, S0 = 1e-4, 0.9, 2.0 ** 16
METRIC = "FP8 linear fwd+bwd TFLOP/s at M=8192,K=N=4096; % of GB300 dense FP8 peak"
WORKLOAD = "transformer proj linear 4096->4096, M=8192 tokens (seq 2048 x batch 4), bf16 in, FP8 HYBRID delayed scaling"
GEMM_SRC = os.path.join(ROOT, "fp8_mixed_precision_reduce_gb300", "csrc", "gemm.cu")
TRAFFIC = os.path.join(ROOT, "profiles", "gemm_fp8_kernel_dram_bytes.json")
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 4.5 / 2.25  # nominal dense ratio


def flops_per_step(m=M_TOK, n=N_OUT, k=K_IN) -> float:
    return 3.0 * 2.0 * m * n * k


# ------------------------------------------------------------------ peaks


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": 6800.0}, "fallback"


def gemm_source_sha256() -> str:
    with open(GEMM_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def gemm_traffic(label=None):
    """DRAM bytes (read + write) per GEMM launch from the ncu capture that
    `--ingest-ncu` recorded: the launch labelled `label` ("fwd", "bwd"), or
    the mean over both when None. None when there is no record or it was
    taken on another gemm.cu (its sha256 is stored with the numbers)."""
    try:
        with open(TRAFFIC) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("gemm_cu_sha256") != gemm_source_sha256():
        return None
    by = rec.get("dram_bytes_per_launch", {})
    try:
        if label is not None:
            return float(by[label])
        return float(statistics.mean(float(v) for v in by.values())) if by else None
    except (KeyError, TypeError, ValueError):
        return None


_BYTE_UNITS = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12,
               "kibyte": 1024.0, "mibyte": 1024.0 ** 2, "gibyte": 1024.0 ** 3}


def parse_ncu_dram_csv(path, kernel="gemm_fp8_kernel", labels=("fwd", "bwd")):
    """Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum)
    of the launches of `kernel` in an ncu CSV export -- either the raw page
    (`ncu -i REP --page raw --csv`: one row per launch, a units row after the
    header) or the metric-per-row export (`ncu --csv --metrics ...`). The
    launches are labelled in capture order, cycling through `labels` (the
    bench step alternates the forward and the fused backward launch, so a
    capture that starts at a forward launch gets them right). Returns
    {label: mean bytes per launch} and the per-launch list."""
    import csv

    with open(path, newline="") as f:
        rows = [r for r in csv.reader(f) if r and not r[0].startswith("==")]
    head = rows[0]
    col = {name: i for i, name in enumerate(head)}
    launches = {}  # id -> [kernel name, read bytes, write bytes]
    if "Metric Name" in col:  # one metric per row
        for r in rows[1:]:
            if len(r) < len(head) or kernel not in r[col["Kernel Name"]]:
                continue
            name = r[col["Metric Name"]]
            if name not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                continue
            unit = _BYTE_UNITS[r[col["Metric Unit"]].strip().lower()]
            v = float(r[col["Metric Value"]].replace(",", "")) * unit
            e = launches.setdefault(int(r[col["ID"]]), [r[col["Kernel Name"]], 0.0, 0.0])
            e[1 if name.endswith("read.sum") else 2] += v
    else:  # the raw page: header, units, one row per launch
        units = rows[1]
        rd, wr = col["dram__bytes_read.sum"], col["dram__bytes_write.sum"]
        for r in rows[2:]:
            if len(r) < len(head) or kernel not in r[col["Kernel Name"]]:
                continue
            v_r = float(r[rd].replace(",", "")) * _BYTE_UNITS[units[rd].strip().lower()]
            v_w = float(r[wr].replace(",", "")) * _BYTE_UNITS[units[wr].strip().lower()]
            launches[int(r[col["ID"]])] = [r[col["Kernel Name"]], v_r, v_w]
    per_launch = []
    for i, lid in enumerate(sorted(launches)):
        name, v_r, v_w = launches[lid]
        per_launch.append({"id": lid, "label": labels[i % len(labels)], "read": v_r, "write": v_w,
                           "bytes": v_r + v_w})
    by = {}
    for lab in labels:
        vals = [e["bytes"] for e in per_launch if e["label"] == lab]
        if vals:
            by[lab] = statistics.mean(vals)
    return by, per_launch


def ingest_ncu(csv_path, command, out_path=None):
    """Writes the GEMM launches' DRAM bytes from an ncu CSV export, keyed by
    the sha256 of the gemm.cu they were captured on, for the bench line's
    roofline.traffic."""
    by, per_launch = parse_ncu_dram_csv(csv_path)
    if not by:
        raise SystemExit(f"no gemm_fp8_kernel launch with DRAM byte counters in {csv_path}")
    rec = {"kernel": "gemm_fp8_kernel", "gemm_cu_sha256": gemm_source_sha256(),
           "dram_bytes_per_launch": by, "launches": per_launch, "command": command,
           "counters": "dram__bytes_read.sum + dram__bytes_write.sum, caches flushed by ncu before each launch"}
    with open(out_path or TRAFFIC, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ distributed


def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Max of a host float over all ranks (plain float when world == 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ our step


class LinearStep:
    """Device state and the step of the proj linear, through the library.

    With `overlap` (the default) two kernels run beside a GEMM instead of
    after it: the dY cast beside the forward GEMM (dY is an input of the
    step, not that GEMM's result), and the master step beside the dgrad
    tiles of the one-launch backward. For the latter the backward launch runs
    its wgrad tiles first and signals in dW's overflow word when dW is
    stored; the master step, started beside it, waits for that signal. The
    master step also runs the delayed-scaling update of the four metas while
    it waits (writing the new scale_inv factors only once the backward
    launch, which reads the old ones, has completed), and the weight's E4M3
    copy is double buffered: dgrad reads the current copy while the master
    step writes the next one. Every result is bitwise that of the serial
    order. Without it: the backward, the update, the master step in place."""

    def __init__(self, m=M_TOK, k=K_IN, n=N_OUT, seed=3, prescanned=True, overlap=True):
        import torch

        import fp8_mixed_precision_reduce_gb300 as fp8mp
        import workloads

        self.fp8mp = fp8mp
        self.overlap = overlap
        # the master step beside the backward needs the epilogue's overflow word
        self.overlap_master = overlap and prescanned
        self.m, self.k, self.n = m, k, n
        dev = "cuda"
        tb = workloads.transformer_block(seed=seed, m=m, d=k, device=dev)
        self.x = tb.x                                                     # (M, K) bf16
        self.dy = tb.dy_proj[:, :n].contiguous() if n != k else tb.dy_proj  # (M, N) bf16
        self.master = workloads.master_weights(n * k, seed=seed, device=dev).view(n, k)
        del tb
        u8 = torch.uint8
        self.X8 = torch.empty((m, k), dtype=u8, device=dev)
        self.W8s = [torch.empty((n, k), dtype=u8, device=dev) for _ in range(2 if self.overlap_master else 1)]
        self.cur = 0  # index of the copy the next step reads
        self.D8 = torch.empty((m, n), dtype=u8, device=dev)
        self.y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
        self.mom = torch.zeros((n, k), dtype=torch.float32, device=dev)
        self.S = torch.tensor([S0], dtype=torch.float32, device=dev)
        self.growth = torch.zeros(1, dtype=torch.int32, device=dev)
        self.found = torch.zeros(1, dtype=torch.int32, device=dev)
        # dW's overflow flag: set by the wgrad epilogue, read and reset by the
        # master step (with prescanned=False the master step scans dW itself)
        self.prescanned = prescanned
        self.gnf = torch.zeros(1, dtype=torch.int32, device=dev)
        E4, E5 = fp8mp.E4M3, fp8mp.E5M2
        self.mx, self.mw, self.my = (fp8mp.Meta(HIST_LEN, E4) for _ in range(3))
        self.md = fp8mp.Meta(HIST_LEN, E5)
        # the weight's first E4M3 copy (and its amax for the first update)
        fp8mp.fp8_quantize(self.master, E4, self.mw.scale, self.W8, None, self.mw.cur_amax)
        # 2 casts, the fwd GEMM, the fused dgrad + wgrad GEMM, the update, and the master step: one kernel
        # on the epilogue's flag (scanning dW itself: a 4-byte memset and one kernel, or three kernels with
        # FP8MP_FUSED_MASTER=0); overlapped, the update runs inside the master step
        self.launches_per_step = 6 if prescanned or os.environ.get("FP8MP_FUSED_MASTER", "1") != "0" else 8
        if self.overlap_master:
            self.launches_per_step = 5

    @property
    def W8(self):
        """The weight's E4M3 copy the next step reads."""
        return self.W8s[self.cur]

    def step(self, gemm_events=None, io=None):
        """One training step. `io` = (x, dy, y, dx) device buffers to use
        instead of the step's own (the end-to-end leg double-buffers them).
        `gemm_events`: four events recorded before and after the forward
        GEMM and before and after the backward GEMM launches."""
        f = self.fp8mp
        x, dy, y, dx = io if io is not None else (self.x, self.dy, self.y, self.dx)
        metas = [self.mx, self.mw, self.my, self.md]
        W8 = self.W8
        f.fp8_quantize(x, f.E4M3, self.mx.scale, self.X8, None, self.mx.cur_amax)
        ev = gemm_events
        if ev is not None:
            ev[0].record()
        f.fp8_linear_fwd(self.X8, W8, self.mx.scale_inv, self.mw.scale_inv, y, y_amax=self.my.cur_amax)
        if ev is not None:
            ev[1].record()
        if self.overlap:
            # dY is an input of the step, not the forward GEMM's result: its
            # cast may run beside the GEMM (it still completes after it)
            f.fp8_quantize_ex(dy, f.E5M2, self.md.scale, self.D8, None, self.md.cur_amax, flags=f.OVERLAP_PREVIOUS)
        else:
            f.fp8_quantize(dy, f.E5M2, self.md.scale, self.D8, None, self.md.cur_amax)
        if not self.overlap_master:
            if ev is not None:
                ev[2].record()
            f.fp8_linear_bwd_rowmajor(self.D8, W8, self.X8, self.md.scale_inv, self.mw.scale_inv,
                                      self.mx.scale_inv, dx, self.dw,
                                      dw_nonfinite=self.gnf if self.prescanned else None)
            if ev is not None:
                ev[3].record()
            f.delayed_scaling_update(metas, f.AMAX_MOST_RECENT, 0)
            f.mp_master_step(self.dw, self.master, self.mom, W8, self.mw.scale, self.mw.cur_amax, self.S,
                             self.growth, self.found, LR, MU, grad_nonfinite=self.gnf if self.prescanned else None)
            return
        if ev is not None:
            ev[2].record()
        # wgrad tiles first; dW's word gets its completion bit while dgrad runs
        f.fp8_linear_bwd_rowmajor(self.D8, W8, self.X8, self.md.scale_inv, self.mw.scale_inv, self.mx.scale_inv,
                                  dx, self.dw, dw_nonfinite=self.gnf, flags=f.SIGNAL_DW_DONE)
        if ev is not None:
            ev[3].record()
        nxt = self.cur ^ 1
        # the next copy, written beside the backward launch (which still reads
        # this one), and the metas' update, whose new scale_inv factors are
        # written once that launch has completed
        f.mp_master_step(self.dw, self.master, self.mom, self.W8s[nxt], self.mw.scale, self.mw.cur_amax, self.S,
                         self.growth, self.found, LR, MU, grad_nonfinite=self.gnf, w8_in=W8,
                         flags=f.OVERLAP_PREVIOUS | f.WAIT_DW_DONE, metas=metas, amax_algo=f.AMAX_MOST_RECENT,
                         margin=0)
        self.cur = nxt


class StepGraphs:
    """The step as CUDA graphs: one per copy of the weight the step reads
    (the step alternates between them), replayed in turn by `replay()`, and
    `count` graphs of one step each with four event-record nodes around the
    GEMM launches (an event node records into the same event at every
    replay, so the timed pass needs one graph per step), replayed in order
    by `replay_timed(i)`. Capture runs on a side stream after the eager
    warm-up (which made the library's one-time attribute and occupancy
    queries); every graph is replayed once here, untimed (its upload),
    unless `upload` is False."""

    def __init__(self, st, count, upload=True):
        import torch

        self.st = st
        c = st.cur
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        self.by_copy = {}
        for p in range(len(st.W8s)):
            st.cur = (c + p) % len(st.W8s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                st.step()
            self.by_copy[(c + p) % len(st.W8s)] = g
        self.timed, self.events, self.timed_copy = [], [], []
        for i in range(count):
            st.cur = (c + i) % len(st.W8s)
            self.timed_copy.append(st.cur)
            ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                st.step(ev)
            self.timed.append(g)
            self.events.append(ev)
        st.cur = c  # capture ran nothing
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        if upload:
            for _ in self.by_copy:
                self.replay()
            for i in range(count):
                self.replay_timed(i)
            torch.cuda.synchronize()

    def replay(self):
        st = self.st
        g = self.by_copy[st.cur]
        st.cur = (st.cur + 1) % len(st.W8s)
        g.replay()

    def replay_timed(self, i):
        st = self.st
        while st.cur != self.timed_copy[i]:  # untimed: bring the weight copy in line
            self.replay()
        st.cur = (st.cur + 1) % len(st.W8s)
        self.timed[i].replay()


def run_e2e(st, steps, world, with_outputs=False):
    """The step end to end through the Python API: each step's inputs x and
    dY are copied in from pinned host memory, and the step's result comes
    back to pinned host memory: the loss scaler's overflow flag and loss
    scale (8 bytes), and with `with_outputs` also Y and dX (128 MiB).
    Copies run on their own streams against two sets of device buffers, so
    step i+1's upload and step i-1's download overlap step i's kernels."""
    import torch

    E = torch.cuda.Event
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    x_h = st.x.cpu().pin_memory()
    dy_h = st.dy.cpu().pin_memory()
    res_h = [torch.empty(2, dtype=torch.int32).pin_memory() for _ in range(2)]
    res_d = [torch.empty(2, dtype=torch.int32, device="cuda") for _ in range(2)]
    y_h = [torch.empty(st.y.shape, dtype=st.y.dtype).pin_memory() for _ in range(2)] if with_outputs else None
    dx_h = [torch.empty(st.dx.shape, dtype=st.dx.dtype).pin_memory() for _ in range(2)] if with_outputs else None
    bufs = [(st.x, st.dy, st.y, st.dx),
            (torch.empty_like(st.x), torch.empty_like(st.dy), torch.empty_like(st.y), torch.empty_like(st.dx))]
    uploaded = [E() for _ in range(2)]    # inputs of buffer set b are on the device
    computed = [E() for _ in range(2)]    # the step using buffer set b has finished
    downloaded = [E() for _ in range(2)]  # results of buffer set b are on the host
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = E(enable_timing=True), E(enable_timing=True)
    t0.record(up)
    for i in range(steps):
        b = i & 1
        x, dy, y, dx = bufs[b]
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(computed[b])    # step i-2 no longer reads these inputs
            x.copy_(x_h, non_blocking=True)
            dy.copy_(dy_h, non_blocking=True)
            uploaded[b].record(up)
        comp.wait_event(uploaded[b])
        if i >= 2:
            comp.wait_event(downloaded[b])    # step i-2's results have left these buffers
        st.step(io=bufs[b])
        # this step's loss-scaler state, before the next step changes it
        res_d[b][0:1].copy_(st.found, non_blocking=True)
        res_d[b][1:2].copy_(st.S.view(torch.int32), non_blocking=True)
        computed[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            res_h[b].copy_(res_d[b], non_blocking=True)
            if with_outputs:
                y_h[b].copy_(y, non_blocking=True)
                dx_h[b].copy_(dx, non_blocking=True)
            downloaded[b].record(down)
    comp.wait_stream(down)
    t1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(t0.elapsed_time(t1) / steps, world)
    h2d = x_h.numel() * x_h.element_size() + dy_h.numel() * dy_h.element_size()
    d2h = res_h[0].numel() * res_h[0].element_size()
    if with_outputs:
        d2h += y_h[0].numel() * y_h[0].element_size() + dx_h[0].numel() * dx_h[0].element_size()
    return ms, h2d, d2h


def library_fp8_gemm_tflops(n=8192):
    """Context for the roofline: cuBLASLt's FP8 GEMM (torch._scaled_mm, E4M3 x
    E4M3 -> bf16, n^3) back to back, measured before the timed steps. None
    when this torch cannot run it."""
    import torch

    try:
        a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
        one = torch.ones((), device="cuda")
        fn = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        best = 0.0
        for _ in range(3):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            for _ in range(10):
                fn()
            t1.record()
            torch.cuda.synchronize()
            best = max(best, 2.0 * n ** 3 / (t0.elapsed_time(t1) / 10 * 1e-3) / 1e12)
        del a, b
        torch.cuda.empty_cache()
        return round(best, 1)
    except (RuntimeError, TypeError, AttributeError):
        return None


def run_ours(args, world, rank, local):
    import torch

    peaks, peak_kind = load_peaks()
    lib_fp8 = library_fp8_gemm_tflops()
    st = LinearStep(prescanned=not args.master_scans_dw, overlap=not args.no_overlap)
    torch.cuda.synchronize()
    flush = torch.empty(int(2 * 129e6 // 4) + 1, dtype=torch.float32, device="cuda")  # > 2x L2

    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    rc = st.fp8mp.fp8mp_check()
    if rc != 0:
        raise RuntimeError(f"warm-up failed: {st.fp8mp.last_error()}")

    E = torch.cuda.Event
    # Pass 1 (the step time): K steps, nothing between the step's kernels,
    # so each may start while the previous one drains (graph edges /
    # programmatic launch). Pass 2 (the roofline): K more steps with timing
    # events around the two GEMM launches; an event between two kernels
    # serialises them, which costs a step about 20 us, so those steps give
    # the GEMM launch durations only.
    if args.eager:
        plain, timed = st.step, None
        launch = "eager (one host launch per library call, programmatic dependent launch)"
    else:
        graphs = StepGraphs(st, args.steps)
        plain, timed = graphs.replay, graphs
        launch = "CUDA graph of the step's library calls, captured once and replayed"
    starts = [E(enable_timing=True) for _ in range(args.steps)]
    ends = [E(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.fill_(float(i))  # L2 flush between timed steps (outside the step events)
            starts[i].record()
            plain()
            ends[i].record()
        torch.cuda.synchronize()
        # pass 2
        gev = [[E(enable_timing=True) for _ in range(4)] for _ in range(args.steps)] if timed is None else timed.events
        starts2 = [E(enable_timing=True) for _ in range(args.steps)]
        ends2 = [E(enable_timing=True) for _ in range(args.steps)]
        if timed is not None:
            while st.cur != timed.timed_copy[0]:  # the copy the first timed graph reads (untimed step)
                plain()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts2[i].record()
            if timed is None:
                st.step(gev[i])
            else:
                timed.replay_timed(i)
            ends2[i].record()
        torch.cuda.synchronize()
        # more witnesses of the step time, after pass 2 (whose GEMM timings
        # are thus taken at the clocks of pass 1, before a second of load can
        # bring the power cap in): further passes of K steps each, the same
        # way, for about a second (the clock sampler sees it too); `value`
        # stays the first pass's
        repeat_means = [statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))]
        t_rep = time.perf_counter()
        while len(repeat_means) < 1 + args.max_repeats and time.perf_counter() - t_rep < args.repeat_seconds:
            rs = [E(enable_timing=True) for _ in range(args.steps)]
            re_ = [E(enable_timing=True) for _ in range(args.steps)]
            for i in range(args.steps):
                flush.fill_(float(i))
                rs[i].record()
                plain()
                re_[i].record()
            torch.cuda.synchronize()
            repeat_means.append(statistics.mean(s.elapsed_time(e) for s, e in zip(rs, re_)))
        torch.cuda.synchronize()
    barrier(world)
    rc = st.fp8mp.fp8mp_check()
    if rc != 0:
        raise RuntimeError(f"timed steps failed: {st.fp8mp.last_error()}")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    step2_ms = [s.elapsed_time(e) for s, e in zip(starts2, ends2)]
    gemm_ms = [[g[0].elapsed_time(g[1]), g[2].elapsed_time(g[3])] for g in gev]  # fwd, bwd (wgrad + dgrad)
    ms_per_step = max_over_ranks(statistics.mean(step_ms), world)
    ms_instrumented = max_over_ranks(statistics.mean(step2_ms), world)
    gemm_step_ms = max_over_ranks(statistics.mean(sum(g) for g in gemm_ms), world)
    fwd_ms = statistics.mean(g[0] for g in gemm_ms)
    bwd_ms = statistics.mean(g[1] for g in gemm_ms)

    # end to end through the public API: every step copies its x and dY in
    # from pinned host memory and reads its result (the loss scaler's state)
    # back; the second run also reads back the outputs Y and dX.
    e2e_ms, h2d, d2h = run_e2e(st, max(10, args.steps), world)
    e2e_out_ms, h2d_out, d2h_out = run_e2e(st, max(10, args.steps), world, with_outputs=True)
    fl = flops_per_step()
    value = world * fl / (ms_per_step * 1e-3) / 1e12
    fp8_nominal = float(peaks["bf16_tflops"]) * FP8_OVER_BF16
    # the GEMM kernel's launches per step do 2MNK (fwd) and 4MNK (dgrad +
    # wgrad: one launch, or two back to back) FLOPs: achieved = their FLOPs /
    # their summed device time
    achieved = fl / ((fwd_ms + bwd_ms) * 1e-3) / 1e12
    # the FP8 peak actually reached on this GPU in this run: the best of
    # cuBLASLt's FP8 GEMM at 8192^3 and this library's fastest GEMM launch;
    # the roofline divides by the larger of it and the nominal bf16 x 2
    own_best = max(max(fl / 3.0 / (g[0] * 1e-3), 2.0 * fl / 3.0 / (g[1] * 1e-3)) for g in gemm_ms) / 1e12
    peak_measured = max(own_best, lib_fp8 or 0.0)
    fp8_peak = max(fp8_nominal, peak_measured)
    rep_sorted = sorted(repeat_means)
    traffic = gemm_traffic()
    clk = clocks.summary()
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8 (e4m3/e5m2) x fp8 -> fp32 accumulate; bf16/fp32 tensors",
        "data": "synthetic (seeded; shapes and distributions of the transformer proj workload)",
        "config": {"workload": WORKLOAD, "M": M_TOK, "K": K_IN, "N": N_OUT, "history_len": HIST_LEN,
                   "amax_compute_algo": "most_recent", "recipe": "HYBRID", "parallelism": f"replicas x{world}",
                   "l2": "flushed (2x L2 write) between timed steps", "launch": launch,
                   "overflow_check": "master step scans dW" if args.master_scans_dw
                   else "wgrad epilogue flags Inf/NaN in the stored dW; the master step reads the flag",
                   "dy_cast": "plain, after the forward GEMM" if args.no_overlap
                   else "enqueued after the forward GEMM with FP8MP_OVERLAP_PREVIOUS: runs beside it",
                   "backward": ("dgrad + wgrad in one launch (wgrad tiles first, FP8MP_SIGNAL_DW_DONE), the master "
                                "step beside it (FP8MP_OVERLAP_PREVIOUS | FP8MP_WAIT_DW_DONE) running the scale update "
                                "of the four metas too, weight copy double-buffered")
                   if st.overlap_master else "dgrad + wgrad in one launch, the scale update, the master step"},
        "gemm_only": {"tflops": round(world * fl / (gemm_step_ms * 1e-3) / 1e12, 2), "ms_per_step": round(gemm_step_ms, 5),
                      "fwd_ms": round(fwd_ms, 5), "bwd_ms": round(bwd_ms, 5),
                      "from": "a second pass of K steps with timing events around the GEMM launches",
                      "ms_per_step_of_that_pass": round(ms_instrumented, 5)},
        "spread": {"passes": len(repeat_means), "steps_per_pass": args.steps,
                   "ms_per_step_median": round(statistics.median(repeat_means), 5),
                   "ms_per_step_min": round(rep_sorted[0], 5), "ms_per_step_max": round(rep_sorted[-1], 5),
                   "of": "per-pass mean step times, the first pass being the one `value` reports"},
        "roofline": {"kernel": "gemm_fp8_kernel", "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                     "peak_nominal": round(fp8_nominal, 1), "frac_of_nominal": round(achieved / fp8_nominal, 4),
                     "peak_measured": round(peak_measured, 1), "own_best_launch_tflops": round(own_best, 1),
                     "traffic": traffic,
                     "traffic_by_launch": {"fwd": gemm_traffic("fwd"), "bwd": gemm_traffic("bwd")},
                     "peak_source": (f"max of {peak_kind} bf16 burst x {FP8_OVER_BF16:g} (nominal fp8/bf16 dense "
                                     "ratio) and the best FP8 GEMM rate measured in this run (cuBLASLt 8192^3, "
                                     "this library's fastest launch)"),
                     "library_fp8_gemm_8192cubed": lib_fp8,
                     "frac_of_library_fp8": round(achieved / lib_fp8, 4) if lib_fp8 else None},
        "e2e": {"value": round(world * fl / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                "result_read_back": "overflow flag and loss scale (the loss scaler's state)",
                "copies": "pinned host, own H2D/D2H streams, double-buffered device tensors"},
        "e2e_with_outputs": {"value": round(world * fl / (e2e_out_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                             "h2d_bytes_per_step": h2d_out, "d2h_bytes_per_step": d2h_out,
                             "ms_per_step": round(e2e_out_ms, 5),
                             "result_read_back": "the above plus the outputs Y and dX (bf16)"},
        "gpu_launches": st.launches_per_step * args.steps,  # the step-time pass; the GEMM-timing pass repeats it
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    del flush
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.baseline_tokens)
    return out


# --------------------------------------------------- the oracle (CPU) arm


def oracle_step_sample(tokens: int, seed=3):
    """Inputs of a `tokens`-row sample of the step, prepared outside timing."""
    import numpy as np

    import workloads

    tb = workloads.transformer_block(seed=seed, m=tokens, d=K_IN)
    x = tb.x.view(__import__("torch").int16).numpy().view(np.uint16)
    dy = tb.dy_proj.view(__import__("torch").int16).numpy().view(np.uint16)
    w = workloads.master_weights(N_OUT * K_IN, seed=seed).numpy().reshape(N_OUT, K_IN)
    return x, dy, w


def oracle_step(orc, x, dy, w, mom, w8, metas):
    """The same step on the CPU oracle: codes, GEMMs in fp64 over decoded
    codes (the oracle takes both operands contiguous along the contraction,
    so it forms the transposes itself), the scale update, then the master
    step re-casting `w8` under the updated weight scale."""
    import numpy as np
    import torch

    E4, E5 = orc.E4M3, orc.E5M2
    mx, mw, my, md = metas
    X8 = orc.cast(x, float(mx.scale[0]), E4)
    mx.record_amax(orc.amax(x))
    W8 = w8.reshape(w.shape)
    y, _ = orc.gemm_ref(X8, E4, W8, E4, float(mx.scale_inv[0]), float(mw.scale_inv[0]), with_abs=False)
    my.record_amax(np.float32(np.abs(y).max()))
    D8 = orc.cast(dy, float(md.scale[0]), E5)
    md.record_amax(orc.amax(dy))
    dx, _ = orc.gemm_ref(D8, E5, orc.transpose_u8(W8), E4, float(md.scale_inv[0]), float(mw.scale_inv[0]),
                         with_abs=False)
    dw, _ = orc.gemm_ref(orc.transpose_u8(D8), E5, orc.transpose_u8(X8), E4, float(md.scale_inv[0]),
                         float(mx.scale_inv[0]), with_abs=False)
    for m, f in zip(metas, (E4, E4, E4, E5)):
        orc.scale_update(m, f, orc.AMAX_MOST_RECENT, 0)
    g = torch.from_numpy(dw.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    st = orc.LossScaleState(S0)
    orc.master_step(g.reshape(-1), w.reshape(-1), mom.reshape(-1), w8.reshape(-1), float(mw.scale[0]),
                    mw.cur_amax, st, LR, MU)


def oracle_initial_weight_copy(orc, w, metas):
    """The weight's first E4M3 copy, cast once before the first step."""
    mw = metas[1]
    w8 = orc.cast(w, float(mw.scale[0]), orc.E4M3).reshape(-1).copy()
    mw.record_amax(orc.amax(w))
    return w8


def cpu_baseline(tokens: int):
    import numpy as np

    import oracle as orc

    orc.build()
    x, dy, w = oracle_step_sample(tokens)
    mom = np.zeros_like(w)
    metas = [orc.Meta(HIST_LEN) for _ in range(4)]
    w8 = oracle_initial_weight_copy(orc, w, metas)
    t0 = time.perf_counter()
    oracle_step(orc, x, dy, w, mom, w8, metas)
    dt = time.perf_counter() - t0
    fl = flops_per_step(m=tokens)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
            "sample": (f"one full step of the whole {M_TOK}-token workload" if tokens == M_TOK
                       else f"one full step on a {tokens}-token sample of the {M_TOK}-token workload")
                      + f" (x {tokens}x{K_IN}, dY {tokens}x{N_OUT}, full {N_OUT}x{K_IN} weight, three GEMMs in fp64, "
                        f"casts, scale update and master step), {dt:.2f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    import numpy as np

    import oracle as orc

    orc.build()
    x, dy, w = oracle_step_sample(args.cpu_tokens)
    mom = np.zeros_like(w)
    metas = [orc.Meta(HIST_LEN) for _ in range(4)]
    w8 = oracle_initial_weight_copy(orc, w, metas)
    for _ in range(args.warmup):
        oracle_step(orc, x, dy, w.copy(), mom.copy(), w8.copy(), [m.copy() for m in metas])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(orc, x, dy, w, mom, w8, metas)
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    fl = flops_per_step(m=args.cpu_tokens)
    value = fl / (ms * 1e-3) / 1e12
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp64 accumulate over decoded fp8 codes; fp32 casts and master step",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "M": M_TOK, "K": K_IN, "N": N_OUT, "history_len": HIST_LEN,
                   "parallelism": "host cores", "sample_tokens": args.cpu_tokens},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
                         "sample": f"each step: the full step on a {args.cpu_tokens}-token sample of the "
                                   f"{M_TOK}-token workload"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------ kernel table


GEMM_SHAPES = (  # (name, M, K, N): the transformer block's and the MLP's linears
    ("proj", 8192, 4096, 4096), ("qkv", 8192, 4096, 12288),
    ("mlp_up", 16384, 4096, 14336), ("mlp_down", 16384, 14336, 4096))
MASTER_PARAMS = 10 ** 9  # the optimizer-state workload


def kernel_table(args):
    """--kernels: every kernel of the path on its own, at the sizes of the
    other workloads (the transformer block's and the MLP's GEMM shapes and
    casts, the master step on 1e9 parameters), each against its roofline:
    device time of one launch (the mean of the middle 80 % of the timed
    launches) with L2 flushed before it (3 warm-up
    launches; the flush's own dirty lines are written back before the
    launch), one JSON line per measurement, the clocks last. Inputs are
    seeded and synthetic. cuBLASLt's FP8 GEMMs (torch._scaled_mm, E4M3/E5M2
    in, bf16 out; the backward as its two launches on the transposed copies
    they need) are timed the same way beside ours, as context."""
    import torch

    import fp8_mixed_precision_reduce_gb300 as fp8mp
    import workloads

    fp8mp.load()
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    fp8_peak = float(peaks["bf16_tflops"]) * FP8_OVER_BF16
    flush = torch.empty(int(2 * 129e6 // 4) + 1, dtype=torch.float32, device="cuda")
    evict = torch.zeros_like(flush)
    reps = max(3, args.steps)

    def timed(fn, n=reps):
        ts = []
        for i in range(n + 3):
            # L2 flushed by a 2x-L2 write, then that write's dirty lines
            # evicted by a 2x-L2 read, so the timed launch starts from DRAM
            # and pays for its own traffic only (as ncu's cache flush does)
            flush.fill_(float(i))
            evict.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b) * 1e3)
        if fp8mp.fp8mp_check() != 0:
            raise RuntimeError("a kernel's bounded wait ran out")
        # the mean of the middle 80 %: the event durations of a ~20 us launch
        # cluster at a few values about 1 us apart, so their median jumps
        # between those values; the trimmed mean resolves finer and still
        # drops the outliers
        ts.sort()
        cut = len(ts) // 10
        return statistics.mean(ts[cut:len(ts) - cut])

    def emit(kernel, workload, us, work, bound, **extra):
        if bound == "tensor":
            achieved, peak, unit = work / us / 1e6, fp8_peak, "TFLOP/s"
        else:
            achieved, peak, unit = work / us / 1e3, hbm, "GB/s"
        line = {"kernel": kernel, "workload": workload, "us": round(us, 2), "value": round(achieved, 1),
                "unit": unit, "roofline": {"bound": bound, "achieved": round(achieved, 1), "peak": round(peak, 1),
                                           "unit": unit, "frac": round(achieved / peak, 4), "of": peak_kind}}
        line.update(extra)
        print(json.dumps(line), flush=True)

    one = torch.ones(1, device="cuda")
    one0 = torch.ones((), device="cuda")
    g = workloads.gen(7, "cuda")
    only = args.only or ""
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clocks:
        # ---- GEMMs: forward, fused backward (ours) and cuBLASLt's
        for name, M, K, N in GEMM_SHAPES:
            if only not in f"{name} M={M} K={K} N={N}":
                continue
            xf = (torch.randn(M, K, generator=g, device="cuda") * 4).to(torch.float8_e4m3fn)
            wf = (torch.randn(N, K, generator=g, device="cuda") * 0.1).to(torch.float8_e4m3fn)
            df = (torch.randn(M, N, generator=g, device="cuda") * 1e3).to(torch.float8_e5m2)
            x8, w8, d8 = xf.view(torch.uint8), wf.view(torch.uint8), df.view(torch.uint8)
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            dx = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
            dw = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
            am = torch.zeros(1, device="cuda")
            flag = torch.zeros(1, dtype=torch.int32, device="cuda")
            fl = 2.0 * M * N * K
            wl = f"{name} M={M} K={K} N={N}"
            lt_f = timed(lambda: torch._scaled_mm(xf, wf.t(), scale_a=one0, scale_b=one0, out_dtype=torch.bfloat16))
            us = timed(lambda: fp8mp.fp8_linear_fwd(x8, w8, one, one, y, y_amax=am))
            emit("gemm_fp8_kernel fwd (bf16 out, amax)", wl, us, fl, "tensor",
                 library={"cublaslt_us": round(lt_f, 2), "cublaslt_tflops": round(fl / lt_f / 1e6, 1)})
            if name == "proj":
                y8 = torch.empty(M, N, dtype=torch.uint8, device="cuda")
                us = timed(lambda: fp8mp.fp8_linear_fwd_fp8out(x8, w8, one, one, one, y8, y_amax=am))
                emit("gemm_fp8_kernel fwd (E4M3 out, amax)", wl, us, fl, "tensor")
                del y8
            wtf, dtf, xtf = wf.t().contiguous(), df.t().contiguous(), xf.t().contiguous()

            def lt_bwd():
                torch._scaled_mm(df, wtf.t(), scale_a=one0, scale_b=one0, out_dtype=torch.bfloat16)
                torch._scaled_mm(dtf, xtf.t(), scale_a=one0, scale_b=one0, out_dtype=torch.bfloat16)

            lt_b = timed(lt_bwd)
            us = timed(lambda: fp8mp.fp8_linear_bwd_rowmajor(d8, w8, x8, one, one, one, dx, dw, dw_nonfinite=flag))
            emit("gemm_fp8_kernel bwd (dgrad + wgrad, one launch, row-major copies)", wl, us, 2 * fl, "tensor",
                 library={"cublaslt_two_launches_us": round(lt_b, 2),
                          "cublaslt_tflops": round(2 * fl / lt_b / 1e6, 1)})
            del xf, wf, df, x8, w8, d8, y, dx, dw, wtf, dtf, xtf
            torch.cuda.empty_cache()
        # ---- casts (bytes per element: 2 in + 1 out, + 1 for the transposed copy)
        cast_wls = ("transformer x 8192x4096 bf16", "mlp down input 16384x14336 bf16", "transformer dY 8192x4096 bf16")
        blk = workloads.transformer_block(device="cuda") if any(only in w for w in cast_wls) else None
        mlp = workloads.mlp(device="cuda") if only in cast_wls[1] else None
        for wl, x in ((cast_wls[0], blk.x if blk else None), (cast_wls[1], mlp.x_down if mlp else None)):
            if x is None or only not in wl:
                continue
            rows, cols = x.shape
            sc = torch.full((1,), 64.0, device="cuda")
            am = torch.zeros(1, device="cuda")
            q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
            qt = torch.empty(cols, rows, dtype=torch.uint8, device="cuda")
            us = timed(lambda: fp8mp.fp8_quantize(x, fp8mp.E4M3, sc, q, None, am))
            emit("cast_rows_kernel (E4M3, amax)", wl, us, 3.0 * x.numel(), "hbm")
            us = timed(lambda: fp8mp.fp8_quantize(x, fp8mp.E4M3, sc, q, qt, am))
            emit("cast_rows_t_kernel (E4M3 + transposed copy, amax)", wl, us, 4.0 * x.numel(), "hbm")
            if rows == 8192:
                sinv = torch.ones(1, device="cuda")
                us = timed(lambda: fp8mp.fp8_quantize_current(x, fp8mp.E4M3, sc, sinv, am, q, None))
                # the operation reads x twice (amax pass, then the cast) and
                # writes the codes: 5 B/elem. It runs as one cooperative launch
                # whose second read of x comes from L2 when x fits there, so
                # the fraction of the 3 B/elem that must cross the DRAM
                # interface is reported beside it.
                emit("current scaling: amax, grid barrier, scale and cast in one launch", wl, us, 5.0 * x.numel(),
                     "hbm", dram_minimum_frac=round(3.0 * x.numel() / us / 1e3 / hbm, 4))
            del q, qt
        if blk is not None and only in cast_wls[2]:
            dy = blk.dy_proj
            rows, cols = dy.shape
            q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
            qt = torch.empty(cols, rows, dtype=torch.uint8, device="cuda")
            db = torch.empty(cols, dtype=torch.float32, device="cuda")
            ws = torch.zeros(fp8mp.fp8_quantize_dbias_workspace_bytes(rows, cols), dtype=torch.uint8, device="cuda")
            sc, am = torch.full((1,), 2.0 ** 10, device="cuda"), torch.zeros(1, device="cuda")
            us = timed(lambda: fp8mp.fp8_quantize_dbias(dy, fp8mp.E5M2, sc, q, qt, db, ws, am))
            emit("cast_dbias_kernel (E5M2 + transposed copy + bias gradient, one launch)",
                 cast_wls[2], us, 4.0 * dy.numel(), "hbm")
            us = timed(lambda: fp8mp.fp8_quantize_dbias(dy, fp8mp.E5M2, sc, q, None, db, ws, am))
            emit("cast_dbias_kernel (E5M2 + bias gradient, no transposed copy, one launch)",
                 cast_wls[2], us, 3.0 * dy.numel(), "hbm")
            del dy, q, qt, db, ws
        del blk, mlp
        torch.cuda.empty_cache()
        # ---- the master step on 1e9 parameters
        n = MASTER_PARAMS
        wl = f"optimizer state, {n:.0e} parameters"
        if only not in wl:
            n = 0
        if n > 0:
            w = workloads.master_weights(n, device="cuda")
            mom = torch.zeros(n, device="cuda")
            w8 = torch.empty(n, dtype=torch.uint8, device="cuda")
            grad = workloads.master_step(n, 0, device="cuda")
            sw, amw = torch.full((1,), 256.0, device="cuda"), torch.zeros(1, device="cuda")
            S, growth = torch.full((1,), S0, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
            found, flag = torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
            us = timed(lambda: fp8mp.mp_master_step(grad, w, mom, w8, sw, amw, S, growth, found, LR, MU,
                                                    grad_nonfinite=flag), n=5)
            emit("prescanned_step_kernel<SgdOpt> (flag from the gradients' producer)", wl, us, 19.0 * n, "hbm")
            us = timed(lambda: fp8mp.mp_master_step(grad, w, mom, w8, sw, amw, S, growth, found, LR, MU), n=5)
            emit("fused_step_kernel<SgdOpt> (scans the gradients itself)", wl, us, 21.0 * n, "hbm")
            bad = grad.clone()
            bad[12345] = float("inf")
            us = timed(lambda: fp8mp.mp_master_step(bad, w, mom, w8, sw, amw, S, growth, found, LR, MU), n=5)
            emit("fused_step_kernel<SgdOpt>, skipped step (an Inf in the gradients)", wl, us, 2.0 * n, "hbm")
            del bad
            S.fill_(S0)
            v2 = torch.zeros(n, device="cuda")
            bp = torch.ones(2, device="cuda")
            us = timed(lambda: fp8mp.mp_master_step_adam(grad, w, mom, v2, w8, sw, amw, S, growth, found, bp, LR,
                                                         grad_nonfinite=flag), n=5)
            emit("prescanned_step_kernel<AdamOpt>", wl, us, 27.0 * n, "hbm")
            us = timed(lambda: fp8mp.mp_master_step_adam(grad, w, mom, v2, w8, sw, amw, S, growth, found, bp, LR), n=5)
            emit("fused_step_kernel<AdamOpt>", wl, us, 29.0 * n, "hbm")
            del w, mom, w8, grad, v2
            torch.cuda.empty_cache()
        # ---- the scale update: latency only
        if only in f"4 metas, L={HIST_LEN}":
            metas = [fp8mp.Meta(HIST_LEN, f) for f in (fp8mp.E4M3, fp8mp.E4M3, fp8mp.E4M3, fp8mp.E5M2)]
            us = timed(lambda: fp8mp.delayed_scaling_update(metas, fp8mp.AMAX_MOST_RECENT))
            print(json.dumps({"kernel": "scale_update_kernel", "workload": f"4 metas, L={HIST_LEN}",
                              "us": round(us, 2), "roofline": None}), flush=True)
    print(json.dumps({"clocks": clocks.summary(),
                      "l2": "flushed (2x L2 write, then a 2x L2 read that evicts its dirty lines) before each timed launch",
                      "reps": reps, "warmup": 3}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=256,
                    help="tokens of the oracle's bounded sample per step of --impl reference")
    ap.add_argument("--baseline-tokens", type=int, default=8192,
                    help="tokens of the oracle step timed as cpu_baseline (8192: the full workload, about 20 s)")
    ap.add_argument("--repeat-seconds", type=float, default=1.0,
                    help="after the timed pass, repeat it for about this long to report the step time's spread")
    ap.add_argument("--max-repeats", type=int, default=400)
    ap.add_argument("--ingest-ncu", metavar="CSV", default=None,
                    help="record the GEMM launches' DRAM bytes from an ncu CSV export of the bench step "
                         "(first captured launch a forward one) for roofline.traffic, then exit")
    ap.add_argument("--ncu-command", default="",
                    help="with --ingest-ncu: the command line that made the capture, stored with the numbers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--master-scans-dw", action="store_true",
                    help="the master step scans dW for Inf/NaN itself instead of reading the wgrad epilogue's flag")
    ap.add_argument("--no-overlap", action="store_true",
                    help="the serial step: cast dY after the forward GEMM, one-launch backward, then the update "
                         "and the master step (no kernel runs beside a GEMM)")
    ap.add_argument("--eager", action="store_true",
                    help="launch every library call from Python in the timed steps instead of replaying graphs")
    ap.add_argument("--kernels", action="store_true",
                    help="instead of the step: each kernel alone at the other workloads' sizes against its "
                         "roofline (one JSON line each; --steps sets the timed launches per kernel)")
    ap.add_argument("--only", default=None,
                    help="with --kernels: only the workloads whose name contains this text (e.g. mlp_up)")
    args = ap.parse_args(argv)
    if args.ingest_ncu:
        rec = ingest_ncu(args.ingest_ncu, args.ncu_command)
        print(json.dumps({"wrote": os.path.relpath(TRAFFIC, ROOT), "dram_bytes_per_launch": rec["dram_bytes_per_launch"]}))
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        out = run_reference(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0

    import torch

    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}), flush=True)
        return 1
    import fp8_mixed_precision_reduce_gb300 as fp8mp

    fp8mp.load()  # raises when the library is missing: no fallback
    if args.kernels:
        # one GPU's table: under torchrun only rank 0 measures, the others exit
        if int(os.environ.get("RANK", "0")) == 0:
            kernel_table(args)
        return 0
    world, rank, local = dist_setup()
    out = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
