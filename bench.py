#!/usr/bin/env python
"""Benchmark: sparse multi-head attention forward on GB300.

One step = one call of ``gtattn_fwd`` (degree binning on the fly, the fused
row kernel, the split-row combine) over the whole R-MAT graph (2^20 nodes,
~17.1M entries, 4 heads x 32, bf16) with inputs resident in HBM.  Prints one
JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--path fwd|plan|probs|bias|weighted|bwd|bwd_plan|ndh|proj] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs its own replica of the workload
(weak scaling, no collective on the data path); the timed region is
bracketed by a barrier and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "sparse MHA fwd edge·heads/sec and achieved HBM GB/s (% of roofline), 1 GB300"
UNIT = "edge·heads/s"
L2_FLUSH_BYTES = 512 << 20


def compulsory_bytes(N, nnz, H, D, esize):
    """Algorithmic bytes of one forward: indptr + indices + Q + out + every
    K/V row gather (each edge reads one K row and one V row)."""
    row = H * D * esize
    return 4 * (N + 1) + 4 * nnz + 2 * N * row + 2 * nnz * row


def unique_bytes(N, nnz, H, D, esize):
    """Each array touched once: the DRAM floor when L2 holds every reuse."""
    row = H * D * esize
    return 4 * (N + 1) + 4 * nnz + 4 * N * row


def path_bytes(path, N, nnz, H, D, esize):
    """(compulsory, unique-floor) bytes of one call of `path`: the forward's
    figures plus what the variant reads or writes on top -- the fp32 bias
    [nnz, H], the fp32 adjacency values [nnz], the fp32 logits and
    probabilities [nnz, H] written by the unfused path; for the backward the
    dO rows read and the fp32 dQ, dK, dV rows written."""
    cb = compulsory_bytes(N, nnz, H, D, esize)
    ub = unique_bytes(N, nnz, H, D, esize)
    if path == "bias":
        cb += 4 * nnz * H
        ub += 4 * nnz * H
    elif path == "weighted":
        cb += 4 * nnz
        ub += 4 * nnz
    elif path == "probs":
        cb += 2 * 4 * nnz * H
        ub += 2 * 4 * nnz * H
    elif path in ("bwd", "bwd_plan"):
        extra = N * H * D * esize + 3 * 4 * N * H * D
        cb += extra
        ub += extra
    elif path in ("bwd_saved", "train"):
        # the backward given the forward's fp32 output and row statistics:
        # those read instead of the output written, dO read, dQ/dK/dV written;
        # the training step adds the forward that writes them
        nhd = N * H * D
        extra = -nhd * esize + 4 * nhd + 4 * N * H + nhd * esize + 3 * 4 * nhd
        if path == "train":
            fc, fu = compulsory_bytes(N, nnz, H, D, esize), unique_bytes(N, nnz, H, D, esize)
            cb += fc - nhd * esize + 4 * nhd + 4 * N * H
            ub += fu - nhd * esize + 4 * nhd + 4 * N * H
        cb += extra
        ub += extra
    elif path == "proj":   # hidden F = H*D in and out: X read, q/k/v and o written and read back, Y written
        F = H * D
        extra = N * F * esize + 2 * 3 * N * F * esize + 2 * N * F * esize + N * F * esize + 4 * F * F * esize
        cb += extra - 4 * N * H * D * esize   # (the attention's Q, K, V, out are the q/k/v/o counted here)
        ub += extra - 4 * N * H * D * esize
    return cb, ub


def proj_flops(N, H, D):
    """Multiply-add flops of the block's two linear maps (hidden H*D)."""
    F = H * D
    return 2.0 * N * F * 3 * F + 2.0 * N * F * F


def cpu_model():
    """The host CPU's model string (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def dense_flops(n_blocks, n, H, D):
    return 4.0 * n * n * D * H * n_blocks


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def ncu_traffic(kernel_tag: str, workload: str, src_name: str = "rows.cu"):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel source (`src_name`
    under csrc/) changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m_b or not m_h:
        return None
    src = os.path.join(ROOT, "graph_transformer_sparse_gb300", "csrc", src_name)
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != m_h.group(1):
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"gtattn_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, group=None) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def reduce_sum(value: float, group=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def job_throughput(local_units: float, local_ms: float, group=None):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    total_units = reduce_sum(local_units, group)
    worst_ms = reduce_max(local_ms, group)
    return total_units / (worst_ms / 1e3), worst_ms, total_units


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def device_inputs(w, dev):
    import torch
    d = dict(indptr=torch.from_numpy(w.indptr).to(dev), indices=torch.from_numpy(w.indices).to(dev))
    for name in ("Q", "K", "V"):
        if w.dtype == "bf16":
            d[name] = torch.from_numpy(w.bits[name].view(np.int16)).to(dev).view(torch.bfloat16)
        else:
            d[name] = torch.from_numpy(getattr(w, name)).to(dev)
    d["out"] = torch.empty_like(d["Q"])
    return d


def make_step(w, d, path, gt, plan=None, probs_bufs=None):
    dt = gt.GTATTN_BF16 if w.dtype == "bf16" else gt.GTATTN_F32
    if path == "fwd":
        return lambda: gt.gtattn_fwd(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz,
                                     w.H, w.D, w.scale, dt)
    if path == "plan":
        return lambda: gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"],
                                          w.H, w.D, w.scale, dt)
    if path == "probs":
        lg, pr = probs_bufs
        return lambda: gt.gtattn_fwd_probs(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], lg, pr,
                                           w.N, w.nnz, w.H, w.D, w.scale, dt)
    if path == "bias":
        (bias,) = probs_bufs
        return lambda: gt.gtattn_fwd_bias(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], bias, d["out"],
                                          w.N, w.nnz, w.H, w.D, w.scale, dt)
    if path == "weighted":
        (values,) = probs_bufs
        return lambda: gt.gtattn_fwd_weighted(d["indptr"], d["indices"], values, d["Q"], d["K"], d["V"], d["out"],
                                              w.N, w.nnz, w.H, w.D, w.scale, dt)
    if path == "ndh":   # the same synthetic rows read as [N, D, H] (head innermost)
        return lambda: gt.gtattn_fwd_ndh(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz,
                                         w.H, w.D, w.scale, dt)
    if path == "bwd":
        dO, dQ, dK, dV = probs_bufs
        return lambda: gt.gtattn_bwd(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], dO, dQ, dK, dV,
                                     w.N, w.nnz, w.H, w.D, w.scale, dt)
    if path == "bwd_plan":   # training on a fixed graph: the plan keeps the source-major pattern
        dO, dQ, dK, dV = probs_bufs
        return lambda: gt.gtattn_bwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], dO, dQ, dK, dV,
                                          w.H, w.D, w.scale, dt)
    if path in ("bwd_saved", "train"):   # the backward reusing the forward's output and row statistics
        dO, dQ, dK, dV, O, stats = probs_bufs
        fdt = gt.GTATTN_F32 if dt == gt.GTATTN_F32 else gt.GTATTN_BF16_OUT_F32

        def fwd():
            gt.gtattn_fwd_plan_stats(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], O, stats, w.H, w.D,
                                     w.scale, fdt)

        def bwd():
            gt.gtattn_bwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], dO, dQ, dK, dV, w.H, w.D,
                               w.scale, dt, O=O, stats=stats)

        if path == "bwd_saved":
            fwd()   # once, outside the timed steps
            return bwd
        return lambda: (fwd(), bwd())
    if path == "proj":   # the block with its projections (SparseMHA: biases, head-inner features)
        X, W, b, Wo, bo, Y = probs_bufs
        F = w.H * w.D
        return lambda: gt.gtattn_fwd_proj(d["indptr"], d["indices"], X, W, b, Wo, bo, Y, w.N, w.nnz, F, w.H, w.D, F,
                                          w.scale, dt, heads_inner=True)
    raise ValueError(path)


def time_steps(step, steps, flush):
    """Per-step CUDA-event times (ms) on the current stream, L2 flushed
    before every step (outside the events) unless `flush` is None."""
    import torch
    s = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        if flush is not None:
            flush.zero_()
        a.record(s)
        step()
        b.record(s)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def run_gpu_workload(w, path, steps, warmup, gt, dev, flush, want_profile=True, detect_dense=False,
                     soak_s=0.0):
    import torch
    d = device_inputs(w, dev)
    plan = None
    probs_bufs = None
    if path in ("plan", "bwd_plan", "bwd_saved", "train"):
        plan = gt.Plan(d["indptr"], d["indices"], detect_dense=detect_dense and path == "plan")
    if path == "probs":
        probs_bufs = (torch.empty(w.nnz, w.H, device=dev), torch.empty(w.nnz, w.H, device=dev))
    if path == "bias":   # per-edge, per-head additive bias: seeded N(0, 1), fp32 [nnz, H]
        gen = torch.Generator(device=dev)
        gen.manual_seed(12345)
        probs_bufs = (torch.randn(w.nnz, w.H, device=dev, generator=gen),)
    if path in ("bwd", "bwd_plan", "bwd_saved", "train"):
        # backward: seeded N(0, 1) output gradient in the input dtype, fp32 gradients
        gen = torch.Generator(device=dev)
        gen.manual_seed(34567)
        dO = torch.randn(w.N, w.H, w.D, device=dev, generator=gen).to(d["Q"].dtype)
        probs_bufs = (dO,) + tuple(torch.empty(w.N, w.H, w.D, device=dev) for _ in range(3))
        if path in ("bwd_saved", "train"):   # the forward's fp32 output and row statistics
            probs_bufs += (torch.empty(w.N, w.H, w.D, device=dev), torch.empty(w.N, w.H, device=dev))
    if path == "proj":   # X ~ N(0, 1), weights and biases ~ U(-1/sqrt(F), 1/sqrt(F)) (nn.Linear's init)
        gen = torch.Generator(device=dev)
        gen.manual_seed(45678)
        F = w.H * w.D
        a = 1.0 / math.sqrt(F)
        X = torch.randn(w.N, F, device=dev, generator=gen).to(d["Q"].dtype)
        W = ((torch.rand(3 * F, F, device=dev, generator=gen) * 2 - 1) * a).to(d["Q"].dtype)
        Wo = ((torch.rand(F, F, device=dev, generator=gen) * 2 - 1) * a).to(d["Q"].dtype)
        b = (torch.rand(3 * F, device=dev, generator=gen) * 2 - 1) * a
        bo = (torch.rand(F, device=dev, generator=gen) * 2 - 1) * a
        probs_bufs = (X, W, b, Wo, bo, torch.empty(w.N, F, dtype=d["Q"].dtype, device=dev))
    if path == "weighted":   # weighted adjacency: seeded U(0, 1) stored values, fp32 [nnz]
        gen = torch.Generator(device=dev)
        gen.manual_seed(23456)
        probs_bufs = (torch.rand(w.nnz, device=dev, generator=gen),)
    step = make_step(w, d, path, gt, plan, probs_bufs)
    if soak_s > 0:   # untimed load so the clock record covers a loaded GPU
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < soak_s:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    times = time_steps(step, steps, flush)
    prof = None
    if want_profile:
        gt.gtattn_profile_enable(True)
        gt.gtattn_profile_read(reset=True)
        time_steps(step, steps, flush)
        prof = gt.gtattn_profile_read(reset=True)
        gt.gtattn_profile_enable(False)
    info = plan.info() if plan is not None else None
    return w, d, step, times, prof, info, plan


def e2e_measure(w, gt, dev, steps, warmup):
    """Same metric end to end through the C ABI with host (pinned) buffers:
    every step one gtattn_fwd_host call, which copies the step's inputs to
    the device, runs the forward and copies the output back (the copies
    overlap the computation over row chunks)."""
    import torch
    host = {}
    host["indptr"] = torch.from_numpy(w.indptr).pin_memory()
    host["indices"] = torch.from_numpy(w.indices).pin_memory()
    for name in ("Q", "K", "V"):
        if w.dtype == "bf16":
            host[name] = torch.from_numpy(w.bits[name].view(np.int16)).view(torch.bfloat16).pin_memory()
        else:
            host[name] = torch.from_numpy(getattr(w, name)).pin_memory()
    host_out = torch.empty(host["Q"].shape, dtype=host["Q"].dtype).pin_memory()
    dt = gt.GTATTN_BF16 if w.dtype == "bf16" else gt.GTATTN_F32
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = host_out.numel() * host_out.element_size()

    def step():
        gt.gtattn_fwd_host(host["indptr"], host["indices"], host["Q"], host["K"], host["V"], host_out, w.N, w.nnz,
                           w.H, w.D, w.scale, dt)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # each step timed on its own (events around one call) and the median
    # reported: the host link is shared with other work on the machine, and
    # a median is not moved by one disturbed step
    s = torch.cuda.current_stream()
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        step()
        b.record(s)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times), h2d, d2h


def cpu_baseline(w, min_seconds=10.0, single_seconds=5.0):
    """The fp64 oracle as it stands, on the host cores: the whole workload,
    repeated until at least `min_seconds` of wall time with the rows split
    over every core; then single-threaded on a bounded random sample of rows
    (at least `single_seconds`)."""
    import oracle
    cores = os.cpu_count() or 1
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, threads=cores)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or reps >= 50:
            break
    eh = float(w.nnz) * w.H * reps
    # single thread: random rows (a fixed sample), repeated for the time budget
    rng = np.random.default_rng(0)
    deg = np.diff(w.indptr)
    rows = np.sort(rng.choice(w.N, size=min(w.N, max(1, w.N // 64)), replace=False))
    eh1, reps1 = float(deg[rows].sum()) * w.H, 0
    t1 = time.perf_counter()
    while True:
        oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, rows=rows, threads=1)
        reps1 += 1
        dt1 = time.perf_counter() - t1
        if dt1 >= single_seconds or reps1 >= 50:
            break
    return dict(value=round(eh / dt, 1), unit=UNIT, cores=cores, kind="oracle", cpu_model=cpu_model(),
                sample=f"whole workload x{reps} ({dt:.1f} s wall), fp64 C oracle, rows split over "
                       f"{cores} host threads",
                single_thread={"value": round(eh1 * reps1 / dt1, 1), "unit": UNIT, "cores": 1,
                               "sample": f"{len(rows)} random rows of {w.N} ({eh1 / (w.nnz * w.H):.2%} of the "
                                         f"edge-heads) x{reps1} ({dt1:.1f} s wall), one host thread"})


def link_rates(dev, nbytes=256 << 20):
    """Pinned host <-> device copy rates (GB/s) over `nbytes`, best of 5."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()
    res = {}
    for name, fn in (("h2d_gbs", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h_gbs", lambda: h.copy_(d, non_blocking=True))):
        best = None
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        res[name] = round(nbytes / (best / 1e3) / 1e9, 1)
    return res


def plan_build_ms(w, d, gt, reps=3):
    """Host wall time of gtattn_csr_build on the workload (it synchronises
    once), median of `reps`."""
    import torch
    ts = []
    for _ in range(reps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pl = gt.Plan(d["indptr"], d["indices"], detect_dense=(w.name == "dense_blocks"))
        torch.cuda.synchronize()
        ts.append((time.perf_counter() - t0) * 1e3)
        pl.close()
    return round(statistics.median(ts), 4)


def gpu_arm(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import graph_transformer_sparse_gb300 as gt
    gt.build()
    gt.load()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    peaks = measured_peaks()

    name = args.workload
    w = wl.make_workload(name)
    barrier()
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        w, d, step, times, prof, info, plan = run_gpu_workload(w, args.path, args.steps, args.warmup, gt, dev,
                                                               flush, detect_dense=(name == "dense_blocks"),
                                                               soak_s=args.soak)
        torch.cuda.synchronize()
        barrier()
    clocks = clk.summary()
    esize = 2 if w.dtype == "bf16" else 4
    local_ms = sum(times)
    units = float(w.nnz) * w.H * args.steps
    value, worst_ms, _ = job_throughput(units, local_ms)
    ms_per_step = worst_ms / args.steps
    cbytes, ubytes = path_bytes(args.path, w.N, w.nnz, w.H, w.D, esize)

    launches_per_step = sum(v["launches"] for v in prof.values()) / args.steps
    total_prof_ms = max(sum(x["ms"] for x in prof.values()), 1e-9)
    shares = {k: round(v["ms"] / total_prof_ms, 4) for k, v in prof.items() if v["launches"]}
    dominant = max(prof, key=lambda k: prof[k]["ms"])
    # the dominant kernel's time per step (the sum over its launches: one,
    # or one per head group when the forward runs the heads in groups)
    kern_ms = prof[dominant]["ms"] / args.steps
    kern_launches = prof[dominant]["launches"] / args.steps
    if dominant == "dense":
        flops = dense_flops(info["n_dense_blocks"], w.N // max(info["n_dense_blocks"], 1), w.H, w.D)
        achieved = flops / (kern_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": "k_dense_attn (tcgen05 dense-block kernel)",
                    "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "traffic": ncu_traffic("k_dense_attn", name, "dense.cu"),
                    "peak_source": f"{peaks['source']} bf16_tflops (burst: the kernel is timed per launch)",
                    "algorithmic_flops_per_launch": flops, "kernel_ms": round(kern_ms, 5),
                    "kernel_shares": shares}
    else:
        # achieved: the unique-bytes floor (each array crosses HBM once) over
        # the kernel's time; the compulsory figure (every K/V gather counted,
        # most served by the L2) and the ncu DRAM bytes sit beside it
        achieved = ubytes / (kern_ms / 1e3) / 1e9
        # (the capture is one launch: a step of head groups launches the kernel once per group)
        traffic = ncu_traffic("k_rows_vec", name) if args.path == "fwd" else None
        if traffic:
            traffic *= kern_launches
        roofline = {"bound": "hbm", "kernel": "k_rows_vec (fused row kernel)", "achieved": round(achieved, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": traffic,
                    "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)"
                    if peaks["source"] == "measured" else "fallback 6.8 TB/s",
                    "algorithmic_bytes_per_launch": ubytes,
                    "algorithmic_bytes": "unique floor: indptr, indices, Q, K, V and out once each",
                    "compulsory_bytes_per_launch": cbytes,
                    "frac_compulsory": round(cbytes / (kern_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                    "frac_dram": (round(traffic / (kern_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)
                                  if traffic else None),
                    "traffic_over_unique": round(traffic / ubytes, 3) if traffic else None,
                    "kernel_ms": round(kern_ms, 5), "kernel_launches_per_step": kern_launches,
                    "kernel_shares": shares}
    # the same step with a warm L2 (no flush between steps)
    warm = time_steps(step, args.steps, None)
    warm_ms = statistics.median(warm)
    build_ms = plan_build_ms(w, d, gt)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{name}: {w.desc}", "N": w.N, "nnz": w.nnz, "H": w.H, "D": w.D,
                   "path": {"fwd": "gtattn_fwd (binning on the fly + fused rows + combine)",
                            "plan": "gtattn_fwd_plan (prebuilt plan)",
                            "probs": "gtattn_fwd_probs (unfused SDDMM/softmax/SpMM)",
                            "bias": "gtattn_fwd_bias (fused, per-edge per-head additive bias, fp32 N(0,1))",
                            "weighted": "gtattn_fwd_weighted (fused, weighted adjacency, fp32 U(0,1))",
                            "bwd": "gtattn_bwd (dQ, dK, dV of sum(out * dO), dO ~ N(0,1))",
                            "bwd_plan": "gtattn_bwd_plan (as bwd, source-major pattern kept in the plan)",
                            "bwd_saved": "gtattn_bwd_plan given the fp32 output and row statistics of "
                                         "gtattn_fwd_plan_stats (no forward recompute)",
                            "train": "gtattn_fwd_plan_stats + gtattn_bwd_plan on its output and statistics "
                                     "(one training step of the attention)",
                            "ndh": "gtattn_fwd_ndh (head-innermost [N, D, H] rows, generic kernel)",
                            "proj": "gtattn_fwd_proj (q/k/v and output projections around the attention, "
                                    "hidden H*D, biases, head-inner features)"}[args.path],
                   "l2": "flushed before every timed step (512 MiB memset, outside the events)",
                   "clock_soak": f"{args.soak:g} s of untimed steps before the warm-up; clocks sampled from "
                                 f"then to the end",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "achieved_gbs_step": round(ubytes / (ms_per_step / 1e3) / 1e9, 1),
        "hbm_frac_step": round(ubytes / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
        "hbm_frac_step_compulsory": round(cbytes / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
        "ms_per_step_warm_l2": round(warm_ms, 5),
        "plan_build_ms": build_ms,
        "roofline": roofline,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clocks,
    }
    if info is not None:
        line["config"]["plan"] = {k: info[k] for k in ("n_long_rows", "n_chunks", "n_dense_blocks", "max_degree")}

    if rank == 0 and not args.no_e2e:
        e_ms, h2d, d2h = e2e_measure(w, gt, dev, max(3, min(args.steps, 9)), 2)
        line["e2e"] = {"value": round(w.nnz * w.H / (e_ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 4),
                       "link": link_rates(dev)}
        # the copies alone at the measured link rates (the two directions
        # overlap, so the longer one): the floor of the end-to-end step
        ln = line["e2e"]["link"]
        line["e2e"]["copy_floor_ms"] = round(max(h2d / (ln["h2d_gbs"] * 1e9), d2h / (ln["d2h_gbs"] * 1e9)) * 1e3, 4)
    if rank == 0 and not args.no_extra:
        extra = {}
        for other, pth in (("erdos_renyi", "fwd"), ("molecules", "fwd"), ("tiny_random", "fwd"),
                           ("dense_blocks", "plan"), ("dense_blocks_d32", "plan"), ("dense_blocks_d128", "plan"),
                           ("rmat", "probs"), ("rmat", "bias"), ("rmat", "weighted"),
                           ("rmat", "bwd"), ("rmat", "bwd_plan"), ("rmat", "bwd_saved"), ("rmat", "train"),
                           ("rmat", "ndh"), ("rmat", "proj"),
                           ("erdos_renyi", "proj"),
                           ("molecules", "proj")):
            if other == name and pth == args.path:
                continue
            # (microsecond-scale graphs: more steps for a stable median)
            n_o = 50 if other in ("tiny_random", "molecules") else max(3, args.steps // 2)
            try:
                if other.startswith("dense_blocks_d"):   # the dense-block graph with heads of another width
                    hd = int(other[len("dense_blocks_d"):])
                    w_o = wl.make_workload("dense_blocks", D=hd)
                    w_o.desc = f"64 disjoint complete graphs of 512 nodes, 8x{hd} bf16, 0.5*N(0,1)"
                else:
                    w_o = wl.make_workload(other)
                wo, _, _, t_o, p_o, inf_o, pl_o = run_gpu_workload(w_o, pth, n_o, 3, gt, dev, flush,
                                                                   detect_dense=True)
            except Exception as exc:  # report, do not hide
                extra[f"{other}/{pth}"] = {"error": str(exc)}
                continue
            ms = statistics.median(t_o)
            es = 2 if wo.dtype == "bf16" else 4
            cb, ub = path_bytes(pth, wo.N, wo.nnz, wo.H, wo.D, es)
            # per step (all of a category's launches in the step)
            kms = {k: round(v["ms"] / n_o, 5) for k, v in p_o.items() if v["groups"]}
            kl = {k: v["launches"] / n_o for k, v in p_o.items() if v["groups"]}
            ent = {"ms": round(ms, 5), "edge_heads_per_s": round(wo.nnz * wo.H / (ms / 1e3), 1),
                   "gbs_unique": round(ub / (ms / 1e3) / 1e9, 1),
                   "hbm_frac": round(ub / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                   "hbm_frac_compulsory": round(cb / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                   "kernel_ms": kms}
            if "rows" in kms and pth in ("fwd", "bias", "weighted"):
                ent["rows_kernel_hbm_frac"] = round(ub / (kms["rows"] / 1e3) / 1e9 / peaks["hbm_gbs"], 4)
                tr = ncu_traffic("k_rows_vec", other) if pth == "fwd" else None
                if tr:
                    tr *= kl["rows"]   # (one capture is one launch: per step, one per head group)
                    ent["rows_kernel_traffic"] = tr
                    ent["rows_kernel_frac_dram"] = round(tr / (kms["rows"] / 1e3) / 1e9 / peaks["hbm_gbs"], 4)
                    ent["traffic_over_unique"] = round(tr / ub, 3)
            if pth == "proj" and "gemm" in kms:
                # the two linear maps' launches (permutations of the weights included)
                tf = proj_flops(wo.N, wo.H, wo.D) / (kms["gemm"] / 1e3) / 1e12
                ent["gemm_ms_per_call"] = round(kms["gemm"], 5)
                ent["gemm_tflops"] = round(tf, 1)
                ent["gemm_tensor_frac"] = round(tf / peaks["bf16_tflops"], 4) if wo.dtype == "bf16" else None
            if other.startswith("dense_blocks") and inf_o and inf_o.get("n_dense_blocks"):
                tf = dense_flops(inf_o["n_dense_blocks"], 512, wo.H, wo.D) / (ms / 1e3) / 1e12
                ent["tflops"] = round(tf, 1)
                ent["tensor_frac"] = round(tf / peaks["bf16_tflops"], 4)
            extra[f"{other}/{pth}"] = ent
            if pl_o is not None:
                pl_o.close()
        line["per_workload"] = extra
    if rank == 0 and ws == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w)
    if plan is not None:
        plan.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def reference_arm(args):
    """The oracle as the reference arm: timed on the host cores on a bounded
    sample per step; rank 0 only."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.make_workload(args.workload)
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    deg = np.diff(w.indptr)
    rows = np.sort(rng.choice(w.N, size=min(w.N, max(1, w.N // 64)), replace=False))
    eh = float(deg[rows].sum()) * w.H
    for _ in range(args.warmup):
        oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, rows=rows[: len(rows) // 8 + 1],
                          threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, rows=rows, threads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    value = eh / dt
    sample = (f"{len(rows)} random rows of {w.N} per step ({eh / (w.nnz * w.H):.2%} of the edge-heads), "
              f"fp64 C oracle over {cores} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{args.workload}: {w.desc}", "N": w.N, "nnz": w.nnz,
                                             "H": w.H, "D": w.D, "path": "fp64 CPU oracle"},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="rmat", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--path", default="fwd", choices=["fwd", "plan", "probs", "bias", "weighted", "bwd", "bwd_plan",
                                                       "bwd_saved", "train", "ndh", "proj"])
    ap.add_argument("--soak", type=float, default=2.0,
                    help="seconds of untimed steps before the warm-up (clock record under load)")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
