"""Benchmark of the paged split-KV decode path on GB300.

One step = one decode pass of the whole path over one synthetic batch: host
planning (shared-prefix detection, split-KV work list, cascade plan), the upload of
the work lists, the split-KV partial kernel(s) and merge_states.  The headline
workload is the flat paged-decode batch (32 requests, Hq=32, Hkv=8, D=128, page 16,
lengths U[512,4096] with a partial last page, 16384-page pool, tile 512 tokens);
the metric is unique KV bytes per second.  The cascade workload (64 requests, 16
sharing an 8192-token prefix) is timed as a flat arm and a cascade arm on the same
inputs, and the MLA workload (128 heads over an fp8 576-wide latent) is timed too.

L2 is flushed before every timed step, outside the timed events: a 512 MB write,
then a 256 MB read of another buffer, so the step starts with a clean L2 holding none
of its inputs (see L2Flush; --l2-flush write keeps the write alone).  The flush also keeps the device busy while the host plans and enqueues the step, so
the events time the device path rather than the host's enqueue latency; the JSON
line reports both durations ("flush_us", "host_enqueue_us") so that this can be read
off each run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import os

# The oracle's CPU baseline runs one process per core on (request, KV head) tasks whose
# matmuls are small; a multi-threaded BLAS in each process would oversubscribe the
# cores (measured 30x slower), so numpy's BLAS keeps one thread per process.  Set
# before numpy is first imported.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")

import argparse
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "unique KV GB/s (flat paged decode; cascade and MLA arms alongside)"
L2_FLUSH_BYTES = 512 << 20
L2_FLUSH_READ_BYTES = 256 << 20
NOMINAL_HBM_GBS = 8000.0

# DRAM bytes (read + write) of one flat-decode launch of the partial kernel, from the
# ncu capture of the flat partial.  Reported only while the kernel source is the one
# the counters were taken on.
TRAFFIC_SOURCE = os.path.join(ROOT, "paged_split_kv_decode_gb300", "csrc", "partial_tcs.cu")
TRAFFIC_SHA256 = "65a307d5034b1e9069eaf9efeb0dcda8734670d0a38e66704fd89dfb81b7b1f6"
TRAFFIC_BYTES = 316089600 + 1150720

# DRAM bytes read per step by the partial kernels of each arm of the two cascade
# workloads (median over launches of a single-pass ncu capture of dram__bytes_read.sum,
# `bench.py --workload cascade`).  They let the criterion be read on the reads each arm
# makes from DRAM as well as on algorithmic reads.  Valid while the partial kernels'
# sources are unchanged.
CASCADE_DRAM_SOURCES = [os.path.join(ROOT, "paged_split_kv_decode_gb300", "csrc", f)
                        for f in ("partial_tcs.cu", "partial_l0.cu")]
CASCADE_DRAM_SHA256 = "601112f6e4e27371b7610a6355e90dc9931e2d3a0dbd4795aefb4a5b7d283b02"
CASCADE_DRAM_READ = {
    # 8192-token prefix: the flat arm's prefix re-reads hit the 129 MB L2
    "flat_vs_cascade": {"flat": 533349504, "cascade": 533303808,
                        "kernels": "flat: partial_tcs 523x8 CTAs; cascade: one partial_tcs launch, both levels"},
    # 65536-token prefix (268 MB): the flat arm re-reads part of the prefix from DRAM
    "flat_vs_cascade_prefix_beyond_l2": {"flat": 931388288, "cascade": 268661504 + 499737216,
                                         "kernels": "flat: partial_tcs 2315x8 CTAs; cascade: partial_l0 (level 0) "
                                                    "+ partial_tcs 267x8 (level 1)"},
}


def partial_traffic():
    import hashlib
    with open(TRAFFIC_SOURCE, "rb") as f:
        return TRAFFIC_BYTES if hashlib.sha256(f.read()).hexdigest() == TRAFFIC_SHA256 else None


def cascade_dram_reads(key):
    """The stored DRAM reads of both arms of a cascade workload, or None once the
    partial kernels' sources differ from those the counters were taken on."""
    import hashlib
    h = hashlib.sha256()
    for path in CASCADE_DRAM_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return CASCADE_DRAM_READ.get(key) if h.hexdigest() == CASCADE_DRAM_SHA256 else None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def unique_kv_bytes(w) -> int:
    """Bytes of K and V a decode step must read at least once: every distinct
    (page, slot) referenced by the page table, for all KV heads."""
    seen = set()
    tokens = 0
    for b in range(w.batch):
        ids = w.page_indices[w.page_indptr[b]:w.page_indptr[b + 1]]
        for k, pid in enumerate(ids):
            valid = w.page_size if k < len(ids) - 1 else int(w.last_page_len[b])
            key = int(pid)
            if key in seen:
                continue
            seen.add(key)
            tokens += valid
    return tokens * w.kv_bytes_per_token()


def flat_config(w, kv_bytes: int, l2_mode: str) -> dict:
    """The headline workload, as both arms of the bench name it."""
    return {"workload": "flat paged decode: B=32, Hq=32, Hkv=8, D=128, page 16, L~U[512,4096], "
                        "16384-page pool, tile 512, merge",
            "batch": w.batch, "unique_kv_bytes": int(kv_bytes),
            "l2": "flushed before every timed step: " + ("512 MB write, then 256 MB read of another buffer"
                                                         if l2_mode == "write+read" else "512 MB write"),
            "parallelism": "replicas"}


def flat_kv_bytes(w) -> int:
    return int(np.sum(w.lengths)) * w.kv_bytes_per_token()


# ----------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.text or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our kernels
class Arm:
    """One workload on the device, run through the library's public API."""

    def __init__(self, w, enable: int):
        import paged_split_kv_decode_gb300 as psd
        self.psd = psd
        self.w = w
        self.enable = enable
        self.ctx = psd.Context(torch.cuda.current_device())
        self.q = w.q.cuda()
        self.k = w.k_pool.cuda()
        self.v = self.k if w.v_pool is None else w.v_pool.cuda()
        self.indices = torch.from_numpy(np.ascontiguousarray(w.page_indices, dtype=np.int32)).cuda()
        self.table = psd.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
        self.args = psd.decode_args(self.q, self.k, self.v, self.indices, num_pages=w.num_pages,
                                    page_size=w.page_size, Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale,
                                    k_scale=w.k_scale, v_scale=w.v_scale)
        self.plan = psd.plan_decode(self.table, w.tile_tokens, enable, w.min_shared_pages, w.min_members)
        self.o = torch.empty((w.batch, w.Hq, w.Dv), dtype=torch.float32, device="cuda")
        self.lse = torch.empty((w.batch, w.Hq), dtype=torch.float32, device="cuda")
        # workspace sized for this page table's largest plan
        cap_items = int(w.page_indptr[-1])
        self.ws = torch.empty(psd.workspace_bytes(w.batch, cap_items, self.plan.num_rows + w.batch,
                                                  w.Hq, w.Dv), dtype=torch.uint8, device="cuda")
        self.stats = None

    def step(self):
        """Host planning + the device path, as a caller runs it each decode step."""
        psd, w = self.psd, self.w
        psd.plan_decode(self.table, w.tile_tokens, self.enable, w.min_shared_pages, w.min_members,
                        plan=self.plan)
        self.stats = psd.cascade_decode(self.ctx, self.args, self.plan, self.o, self.lse, self.ws)

    def launches_per_step(self) -> int:
        return (2 if self.plan.num_members > 0 else 1) + 1

    def check(self):
        assert self.psd.check_device_error(self.ctx, self.ws) == 0


class L2Flush:
    """Evicts the decode's inputs from L2 before a timed step, outside the events.

    'write' writes a 512 MB buffer (about 4x the 129 MB L2).  That leaves L2 full of
    dirty lines, and the next kernel's reads must first write them back to HBM, so a
    read-bound kernel timed right after it pays for the flush's write-backs too.
    'write+read' (the default) then reads a separate 256 MB buffer, which moves those
    write-backs before the timed region and leaves L2 holding only clean lines that the
    step never touches.  Either way the step starts with none of its inputs in L2."""

    def __init__(self, mode: str = "write+read"):
        self.mode = mode
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.rbuf = torch.ones(L2_FLUSH_READ_BYTES // 4, dtype=torch.float32, device="cuda") \
            if mode == "write+read" else None
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        self.buf.zero_()
        if self.rbuf is not None:
            torch.sum(self.rbuf, dim=0, out=self.sink)

    def describe(self) -> str:
        return ("512 MB write, then a 256 MB read of another buffer" if self.rbuf is not None
                else "512 MB write") + ", before every timed step"


def time_steps(fn, steps: int, warmup: int, flush: L2Flush, host_us: list | None = None):
    """Per-step CUDA-event times (ms) with an L2 flush before each step.  When
    `host_us` is given, the host time from the start event's record to the end
    event's record (planning, marshalling and launches) is appended to it per step."""
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        t0 = time.perf_counter()
        fn()
        e1.record(s)
        if host_us is not None:
            host_us.append((time.perf_counter() - t0) * 1e6)
        times.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def rep_stats(times, reps: int = 5) -> dict:
    """The K per-step times split into `reps` consecutive reps (fewer when K < reps):
    each rep's median step time, then the median, minimum and maximum over reps, in
    ms (the per-arm median/min/max over reps of the mlxcel PR #1004 bench harness,
    How to run the benchmarks section)."""
    n = max(1, min(reps, len(times)))
    per = [statistics.median(times[i * len(times) // n:(i + 1) * len(times) // n]) for i in range(n)]
    return {"reps": n, "steps_per_rep": len(times) // n, "median_ms": round(statistics.median(per), 5),
            "min_ms": round(min(per), 5), "max_ms": round(max(per), 5)}


def flush_us(flush: L2Flush, reps: int = 5) -> float:
    """Device time of one L2 flush (µs), CUDA events on the current stream."""
    s = torch.cuda.current_stream()
    flush()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(reps):
        flush()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def kernel_timing(arm: Arm, steps: int, warmup: int, flush, kind: str = "auto"):
    """Per-kernel device times of the decode step, from the CUDA events the library
    records around each kernel on the stream it launches on ('auto' = the
    16-row-group tensor-core partial kernel, 'cuda_core' = the CUDA-core one)."""
    arm.ctx.set_partial_kernel(kind)
    arm.ctx.set_timing(True)
    for _ in range(warmup):
        flush()
        arm.step()
    torch.cuda.synchronize()
    out = {"level0_ms": [], "partial_ms": [], "merge_ms": []}
    for _ in range(steps):
        flush()
        arm.step()
        for k, v in arm.ctx.kernel_times().items():
            out[k].append(v)
    arm.ctx.set_timing(False)
    arm.ctx.set_partial_kernel("auto")
    return {k: statistics.mean(v) for k, v in out.items()}


def partial_algorithmic_bytes(arm: Arm) -> int:
    """Bytes the split-KV partial kernel must move: every K/V token of every work item
    (all KV heads), the query rows, and the partial rows it writes."""
    w = arm.w
    n_rows = arm.plan.num_rows
    return flat_kv_bytes(w) + w.q.numel() * 2 + n_rows * w.Hq * (w.Dv + 1) * 4


def merge_algorithmic_bytes(arm: Arm) -> int:
    w = arm.w
    return (arm.plan.num_rows + w.batch) * w.Hq * (w.Dv + 1) * 4


def e2e_timing(arm: Arm, steps: int, warmup: int, flush):
    """Same decode step through the public API with host buffers.  The step's query
    rows and page table sit in one pinned host buffer that the partial kernel reads
    over the host link as it runs (no staging copy); the plan reaches the kernels in
    their launch parameters; the merge kernel stores the output rows and LSE straight
    into pinned host memory (no separate copy)."""
    psd, w = arm.psd, arm.w
    q_bytes = w.q.numel() * 2
    idx = np.ascontiguousarray(w.page_indices, dtype=np.int32)
    off_idx = (q_bytes + 255) // 256 * 256
    in_bytes = off_idx + idx.nbytes
    host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    host_in[:q_bytes].copy_(w.q.contiguous().view(torch.uint8).reshape(-1))
    host_in[off_idx:].copy_(torch.from_numpy(idx).view(torch.uint8))
    q_host = host_in[:q_bytes].view(torch.bfloat16).view(w.q.shape)
    idx_host = host_in[off_idx:].view(torch.int32)
    o_elems, l_elems = arm.o.numel(), arm.lse.numel()
    host_out = torch.empty(o_elems + l_elems, dtype=torch.float32).pin_memory()
    o_host, l_host = host_out[:o_elems].view(arm.o.shape), host_out[o_elems:].view(arm.lse.shape)
    args = psd.decode_args(q_host, arm.k, arm.v, idx_host, num_pages=w.num_pages, page_size=w.page_size,
                           Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale, k_scale=w.k_scale, v_scale=w.v_scale)

    def step():
        psd.plan_decode(arm.table, w.tile_tokens, arm.enable, w.min_shared_pages, w.min_members, plan=arm.plan)
        psd.cascade_decode(arm.ctx, args, arm.plan, o_host, l_host, arm.ws)

    times = time_steps(step, steps, warmup, flush)
    # Host-observed latency of the same step: from the call's start, with the device
    # idle and L2 flushed, until the host holds the outputs (stream synchronize).
    wall = []
    s = torch.cuda.current_stream()
    for _ in range(steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step()
        s.synchronize()
        wall.append((time.perf_counter() - t0) * 1e3)
    torch.cuda.synchronize()
    arm.step()
    torch.cuda.synchronize()
    assert torch.equal(o_host, arm.o.cpu()) and torch.equal(l_host, arm.lse.cpu()), \
        "end-to-end outputs differ from the device-resident step"
    plan_bytes = (arm.plan.num_items * 16 + (w.batch * 3 + 1) * 4 + 256)
    h2d = in_bytes + plan_bytes
    d2h = (o_elems + l_elems) * 4
    return times, h2d, d2h, wall


def no_sharing_gate(arm, steps: int, warmup: int, flush) -> dict:
    """The flat workload (no two requests share a page) with and without shared-prefix
    detection in front of the flat launch: the no-sharing overhead gate of the mlxcel
    PR #1004 bench harness (How to run the benchmarks).  Host time per planning call
    with detection (psd_plan_decode enable=1: the scan runs and declines) and without
    it (enable=0: the split work list alone), and the device time of the step each way
    (CUDA events, medians over steps)."""
    psd, w = arm.psd, arm.w

    def plan(enable):
        psd.plan_decode(arm.table, w.tile_tokens, enable, w.min_shared_pages, w.min_members, plan=arm.plan)

    def host_us(enable, reps=400):
        plan(enable)
        t0 = time.perf_counter()
        for _ in range(reps):
            plan(enable)
        return (time.perf_counter() - t0) / reps * 1e6

    def step(enable):
        plan(enable)
        psd.cascade_decode(arm.ctx, arm.args, arm.plan, arm.o, arm.lse, arm.ws)

    h_det, h_flat = host_us(1), host_us(0)
    assert arm.plan.num_members == 0
    d_det = statistics.median(time_steps(lambda: step(1), steps, warmup, flush))
    d_flat = statistics.median(time_steps(lambda: step(0), steps, warmup, flush))
    return {"workload": "the flat workload (nothing shared)",
            "host_plan_us_with_detection": round(h_det, 2), "host_plan_us_without_detection": round(h_flat, 2),
            "detection_host_us": round(h_det - h_flat, 2),
            "device_step_ms_with_detection": round(d_det, 5),
            "device_step_ms_without_detection": round(d_flat, 5),
            "note": "host time per call through the Python binding; the device step is timed after an L2 "
                    "flush that outlasts the host's planning, so detection shows up in host time only"}


def merge_sweep(ctx, steps: int, warmup: int, flush, hbm: float, sizes=(1024, 16384, 262144, 1048576)):
    """merge_states alone over the sweep's sizes (H=32, D=128, log2 LSE ~ U(-5,20),
    groups U[1,16] with a group of one), inputs drawn on the device."""
    import paged_split_kv_decode_gb300 as psd
    out = []
    for M in sizes:
        v_in, lse_in, o_indptr = synth.merge_inputs_device(0, M)
        ind = torch.from_numpy(o_indptr).cuda()
        N = int(o_indptr[-1])
        H, D = v_in.shape[1], v_in.shape[2]
        v_out = torch.empty((M, H, D), dtype=torch.float32, device="cuda")
        l_out = torch.empty((M, H), dtype=torch.float32, device="cuda")
        n = max(3, steps // 4) if M >= 262144 else steps
        t = statistics.mean(time_steps(lambda: psd.merge_states(ctx, v_in, lse_in, ind, v_out, l_out),
                                       n, min(warmup, 3), flush))
        nbytes = (N + M) * H * (D + 1) * 4 + (M + 1) * 4
        gbs = nbytes / (t * 1e-3) / 1e9
        out.append({"rows": M, "input_rows": N, "ms": round(t, 4), "gbs": round(gbs, 1),
                    "frac_of_measured_hbm": round(gbs / hbm, 4)})
        del v_in, lse_in, v_out, l_out, ind
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------- oracle
# The float64 oracle, as it stands, timed on the host cores: one task is one
# (request, KV head) pair (the oracle's gather over that head's slice of the pools,
# then its softmax attention for the head's G query rows).  The tasks run on every
# core the process may use, through a pool of forked workers that inherit the
# workload's arrays; the pool is forked before this process touches CUDA (a process
# forked after CUDA is initialised must not use it, and these never do).
_ORACLE = {}


def _oracle_task(task) -> int:
    from oracle import attention as A
    a, q, G = _ORACLE["a"], _ORACLE["q"], _ORACLE["G"]
    b, kv = task
    head = dict(a, k_raw=a["k_raw"][:, :, kv:kv + 1],
                v_raw=None if a["v_raw"] is None else a["v_raw"][:, :, kv:kv + 1])
    K, V = A.gather_kv(head, b)
    A.attend(q[b, kv * G:(kv + 1) * G], K, V, a["sm_scale"])
    return K.shape[0]


class OraclePool:
    """The oracle over (request, KV head) tasks of one workload, on all host cores
    (a forked process pool) or on one (this process)."""

    def __init__(self, w):
        import multiprocessing as mp
        from oracle import attention as A
        a = A.workload_arrays(w)
        _ORACLE.update(a=a, q=A.bf16_bits_to_f64(a["q_raw"]), G=w.Hq // w.Hkv)
        self.w = w
        self.tasks = [(b, kv) for b in range(w.batch) for kv in range(w.Hkv)]
        self.head_bytes = w.kv_bytes_per_token() // w.Hkv
        self.cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        self.pool = mp.get_context("fork").Pool(self.cores)

    def pass_all_cores(self) -> int:
        """One pass over every task on all cores; returns the K/V bytes attended."""
        return sum(self.pool.imap_unordered(_oracle_task, self.tasks, chunksize=2)) * self.head_bytes

    def pass_one_core(self, tasks) -> int:
        return sum(_oracle_task(t) for t in tasks) * self.head_bytes

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_baseline(w, budget_all_s: float = 8.0, budget_one_s: float = 6.0):
    """cpu_baseline: the oracle on all host cores (whole passes over the batch for about
    budget_all_s) and on one core (tasks in batch order for about budget_one_s)."""
    op = OraclePool(w)
    try:
        op.pass_all_cores()                                   # warm the workers
        t0, nbytes, passes = time.perf_counter(), 0, 0
        while passes == 0 or time.perf_counter() - t0 < budget_all_s:
            nbytes += op.pass_all_cores()
            passes += 1
        all_gbs = nbytes / (time.perf_counter() - t0) / 1e9
    finally:
        op.close()
    t0, nbytes1, ntask = time.perf_counter(), 0, 0
    while ntask == 0 or time.perf_counter() - t0 < budget_one_s:
        nbytes1 += op.pass_one_core([op.tasks[ntask % len(op.tasks)]])
        ntask += 1
    one_gbs = nbytes1 / (time.perf_counter() - t0) / 1e9
    return {"value": round(all_gbs, 4), "unit": "GB/s", "cores": op.cores, "kind": "oracle",
            "value_all_cores": round(all_gbs, 4), "cores_all": op.cores, "value_1_core": round(one_gbs, 4),
            "sample": f"all cores: {passes} whole passes over the {w.name} batch ({len(op.tasks)} "
                      f"(request, KV head) tasks each); 1 core: {ntask} tasks; float64 numpy oracle"}


# ------------------------------------------------------------------- main paths
def dist_setup(n):
    """Replicas under torchrun: one process per GPU over NCCL (gloo without a GPU, as
    in the CPU tests).  Returns (rank, world, local_rank)."""
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, int(os.environ.get("LOCAL_RANK", 0))
    import torch.distributed as dist
    dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return dist.get_rank(), dist.get_world_size(), int(os.environ.get("LOCAL_RANK", 0))


def dist_max(x: float, world: int) -> float:
    """The maximum of x over the ranks (the slowest replica sets the job's time)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def replica_throughput(bytes_per_rank: int, ms_local: float, world: int) -> tuple:
    """Whole-job GB/s of `world` replicas that each process bytes_per_rank per step:
    all ranks' bytes over the slowest rank's step time.  Returns (GB/s, max ms)."""
    ms_max = dist_max(ms_local, world)
    return world * bytes_per_rank / (ms_max * 1e-3) / 1e9, ms_max


def autotune_report(arm, reps):
    """psd_autotune_tile on the flat batch: cold-L2 step time per candidate tile (the
    headline keeps the configured 512-token tile)."""
    import paged_split_kv_decode_gb300 as psd
    w = arm.w
    tiles = [256, 384, 512, 768, 1024, 2048]
    items, o_indptr = psd.split_plan(arm.table, min(tiles))
    ws = torch.empty(psd.workspace_bytes(w.batch, max(len(items), 1), int(o_indptr[-1]), w.Hq, w.Dv),
                     dtype=torch.uint8, device="cuda")
    best, ms = arm.ctx.autotune_tile(arm.args, arm.table, tiles, arm.o, arm.lse, ws, 1, w.min_shared_pages,
                                     w.min_members, reps=reps)
    return {"tiles": tiles, "step_ms": [round(x, 5) for x in ms], "best_tile": best,
            "method": "psd_autotune_tile: cascade_decode per tile, cold clean L2 before each timed call (256 MB write, then 256 MB read of another region)"}


def nested_timing(steps, warmup, flush):
    """System prompt + two tenant sub-prefixes: flat arm, two-level cascade (the
    system prompt once) and nested cascade (the tenant sub-prefixes once as well)."""
    import paged_split_kv_decode_gb300 as psd
    w = synth.nested_decode(seed=0, canary=False)
    flat_arm, casc_arm = Arm(w, enable=0), Arm(w, enable=1)
    nest = Arm(w, enable=1)
    plan = psd.plan_nested(nest.table, w.tile_tokens, 1, w.min_shared_pages, w.min_members, 2)
    ws = psd.nested_workspace_for(plan, w.Hq, w.Dv, "cuda")

    def nested_step():
        psd.cascade_decode_nested(nest.ctx, nest.args, plan, nest.o, nest.lse, ws)
    nested_step()
    torch.cuda.synchronize()
    err = np.abs(nest.o.cpu().double().numpy() - flat_arm_outputs(flat_arm)).max()
    tf = statistics.mean(time_steps(flat_arm.step, steps, warmup, flush))
    tc = statistics.mean(time_steps(casc_arm.step, steps, warmup, flush))
    tn = statistics.mean(time_steps(nested_step, steps, warmup, flush))
    uniq = unique_kv_bytes(w)
    return {"workload": "nested decode: 32 requests; a 4096-token system prompt for two tenants of 8, "
                        "each with a 2048-token sub-prefix and suffixes U[64,1024]; 16 independent "
                        "U[512,4096]; Hq=32, Hkv=8, D=128, page 16, tile 512",
            "flat_ms": round(tf, 4), "two_level_ms": round(tc, 4), "nested_ms": round(tn, 4),
            "segments": [list(x) for x in plan.segments], "flat_bytes": int(flat_kv_bytes(w)),
            "unique_bytes": int(uniq), "nested_unique_kv_gbs": round(uniq / (tn * 1e-3) / 1e9, 1),
            "max_abs_diff_vs_flat": float(err)}


def flat_arm_outputs(arm):
    arm.step()
    torch.cuda.synchronize()
    return arm.o.cpu().double().numpy()


def rope_append_timing(ctx, steps, warmup, flush):
    """The RoPE + KV-append step before decode: one launch per step, CUDA events."""
    import paged_split_kv_decode_gb300 as psd
    out = {}
    for kind, T, kv in (("gqa", 32, "bf16"), ("mla", 128, "fp8_e4m3"), ("gqa", 4096, "bf16")):
        st = synth.append_step(seed=0, kind=kind, T=T, kv_dtype=kv, num_pages=max(1024, T // 8))
        dev = lambda t: None if t is None else t.cuda().contiguous()
        q, kn, kr, v, kp, vp = dev(st.q), dev(st.k_nope), dev(st.k_rope), dev(st.v), dev(st.k_pool), dev(st.v_pool)
        cs = torch.from_numpy(st.cos_sin).cuda()
        pos, slots = torch.from_numpy(st.positions).cuda(), torch.from_numpy(st.slot_mapping).cuda()
        fault = torch.zeros(1, dtype=torch.int32, device="cuda")

        def step():
            psd.rope_append_kv(ctx, q, kn, kr, v, cs, pos, slots, kp, vp, rot_dim=st.rot_dim, neox=st.neox,
                               q_rope_col=st.q_rope_col, page_size=st.page_size, k_scale=st.k_scale,
                               v_scale=st.v_scale, fault=fault)
        ms = statistics.mean(time_steps(step, steps, warmup, flush))
        assert int(fault.item()) == 0
        esz = 1 if kv == "fp8_e4m3" else 2
        Hq, Dq = st.q.shape[1], st.q.shape[2]
        Hkv = st.k_rope.shape[1]
        Dk = st.k_rope.shape[2] + (st.k_nope.shape[2] if st.k_nope is not None else 0)
        Dv = st.v.shape[2] if st.v is not None else 0
        # algorithmic bytes: q rope columns read + written, new K/V read, pool rows written,
        # cos/sin rows and the two int32 per token
        b = T * (2 * Hq * st.rot_dim * 2 + Hkv * (Dk + Dv) * 2 + Hkv * (Dk + Dv) * esz
                 + st.rot_dim * 4 + 8)
        out[f"{kind}_{kv}_T{T}"] = {"us": round(ms * 1e3, 2), "gbs": round(b / (ms * 1e-3) / 1e9, 1),
                                    "algorithmic_bytes": int(b)}
    return out


def host_plan_us(w, reps=200):
    """Host detection + cascade planning per call: from scratch (psd_plan_decode) and
    as a plan-cache hit (the same table on the next layer)."""
    import paged_split_kv_decode_gb300 as psd
    t = psd.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
    plan = psd.plan_decode(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    t0 = time.perf_counter()
    for _ in range(reps):
        psd.plan_decode(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members, plan)
    scratch = (time.perf_counter() - t0) / reps
    cache = psd.PlanCache(4)
    cache.lookup(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    t0 = time.perf_counter()
    for _ in range(reps):
        cache.lookup(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    hit = (time.perf_counter() - t0) / reps
    cache.lookup(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members, generation=1)
    t0 = time.perf_counter()
    for _ in range(reps):
        cache.lookup(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members, generation=1)
    gen_hit = (time.perf_counter() - t0) / reps
    return {"plan_decode": round(scratch * 1e6, 1), "plan_cache_hit": round(hit * 1e6, 1),
            "plan_cache_generation_hit": round(gen_hit * 1e6, 1), "page_ids": int(w.page_indptr[-1]),
            "note": "per call, through the Python binding"}


def large_flat_timing(args, flush, hbm: float):
    """The flat workload's shapes with four times the requests (128, 1.2 GB of K/V):
    the partial kernel's rate when a launch's fixed ramp and tail weigh less."""
    w = synth.flat_decode(seed=0, canary=False, batch=128, num_pages=65536)
    arm = Arm(w, enable=0)
    arm.step()
    arm.check()
    t = statistics.mean(time_steps(arm.step, args.steps, args.warmup, flush))
    kt = kernel_timing(arm, args.steps, args.warmup, flush)
    algo = partial_algorithmic_bytes(arm)
    uniq = unique_kv_bytes(w)
    out = {"workload": "flat paged decode, 128 requests (otherwise the flat workload), 65536-page pool",
           "ms": round(t, 5), "unique_kv_gbs": round(uniq / (t * 1e-3) / 1e9, 1),
           "frac_of_measured_hbm": round(uniq / (t * 1e-3) / 1e9 / hbm, 4),
           "partial_ms": round(kt["partial_ms"], 5),
           "partial_gbs": round(algo / (kt["partial_ms"] * 1e-3) / 1e9, 1),
           "partial_frac_of_measured_hbm": round(algo / (kt["partial_ms"] * 1e-3) / 1e9 / hbm, 4),
           "algorithmic_bytes_per_launch": int(algo)}
    del arm
    return out


def cascade_comparison(wc, label, args, flush, plan_us=False, key=None):
    """Flat arm vs cascade arm on one batch: step times, per-kernel times and the
    criterion (T_flat - T_casc) / T_flat >= 0.7 x the fraction of K/V reads removed."""
    flat_arm, casc_arm = Arm(wc, enable=0), Arm(wc, enable=1)
    casc_arm.step()
    casc_arm.check()
    st = casc_arm.stats
    tfs = time_steps(flat_arm.step, args.steps, args.warmup, flush)
    tcs = time_steps(casc_arm.step, args.steps, args.warmup, flush)
    tf, tc = statistics.mean(tfs), statistics.mean(tcs)
    kf = kernel_timing(flat_arm, args.steps, args.warmup, flush)
    kc = kernel_timing(casc_arm, args.steps, args.warmup, flush)
    # each level-0 kernel forced on the same batch (the default picks one by the size
    # of level 0)
    level0 = {}
    for kind in ("mma_sync", "tcgen05"):
        casc_arm.ctx.set_level0_kernel(kind)
        tk = time_steps(casc_arm.step, args.steps, args.warmup, flush)
        kk = kernel_timing(casc_arm, args.steps, args.warmup, flush)
        level0[kind] = {"rep_stats": rep_stats(tk), "kernels_ms": {k: round(v, 5) for k, v in kk.items()}}
    casc_arm.ctx.set_level0_kernel("auto")
    casc_arm.step()
    casc_arm.check()
    flat_arm.check()
    flat_b, uniq_b = flat_kv_bytes(wc), unique_kv_bytes(wc)
    removed = (flat_b - uniq_b) / flat_b
    reduction = (tf - tc) / tf
    out = {
        "workload": label,
        "flat_ms": round(tf, 4), "cascade_ms": round(tc, 4),
        "flat_rep_stats": rep_stats(tfs), "cascade_rep_stats": rep_stats(tcs),
        "flat_tokens_per_s": round(wc.batch / (tf * 1e-3), 1),
        "cascade_tokens_per_s": round(wc.batch / (tc * 1e-3), 1),
        "flat_kv_bytes": int(flat_b), "unique_kv_bytes": int(uniq_b),
        "flat_unique_kv_gbs": round(uniq_b / (tf * 1e-3) / 1e9, 1),
        "cascade_unique_kv_gbs": round(uniq_b / (tc * 1e-3) / 1e9, 1),
        "flat_arm_algorithmic_gbs": round(flat_b / (kf["partial_ms"] * 1e-3) / 1e9, 1),
        "removed_read_fraction": round(removed, 4), "wall_time_reduction": round(reduction, 4),
        "criterion_reduction_ge_0.7x_removed": bool(reduction >= 0.7 * removed),
        "criterion_on_dram_bytes": None,
        "flat_kernels_ms": {k: round(v, 5) for k, v in kf.items()},
        "cascade_kernels_ms": {k: round(v, 5) for k, v in kc.items()},
        "level0_kernels": dict(level0, note="mma_sync: level 0 in 16-row groups (or 64-row blocks) of the "
                                               "mma.sync kernel, in one launch with level 1; tcgen05: the persistent "
                                               "tcgen05 kernel over (chunk, KV head) tasks, on a second stream; the "
                                               "headline arm takes the default choice"),
        "stats": st,
    }
    dram = cascade_dram_reads(key)
    if dram is not None:
        removed_dram = (dram["flat"] - dram["cascade"]) / dram["flat"]
        out["criterion_on_dram_bytes"] = {
            "flat_arm_dram_read": dram["flat"], "cascade_arm_dram_read": dram["cascade"],
            "removed_dram_fraction": round(removed_dram, 4),
            "met": bool(reduction >= 0.7 * removed_dram), "kernels": dram["kernels"],
            "source": "ncu dram__bytes_read.sum per launch (single pass), median over launches"}
    if plan_us:
        out["host_plan_us"] = host_plan_us(wc)
    del flat_arm, casc_arm
    return out


def headline_summary(line: dict) -> dict:
    """The figures a reader checks first, repeated compactly at the end of the line."""
    out = {"flat_step_ms": line["rep_stats"], "flat_partial_frac": line["roofline"]["frac"],
           "e2e_gbs": line["e2e"]["value"], "e2e_wall_ms": line["e2e"]["wall_ms_median"],
           "detection_host_us": line["no_sharing_gate"]["detection_host_us"]}
    for key, short in (("flat_vs_cascade", "cascade"), ("flat_vs_cascade_prefix_beyond_l2", "beyond_l2")):
        c = line.get(key)
        if c:
            out[short] = {"flat_ms": c["flat_rep_stats"]["median_ms"], "cascade_ms": c["cascade_rep_stats"]["median_ms"],
                          "cascade_level0_ms": c["cascade_kernels_ms"]["level0_ms"],
                          "cascade_partial_ms": c["cascade_kernels_ms"]["partial_ms"],
                          "cascade_ms_level0_mma_sync": c["level0_kernels"]["mma_sync"]["rep_stats"]["median_ms"],
                          "cascade_ms_level0_tcgen05": c["level0_kernels"]["tcgen05"]["rep_stats"]["median_ms"],
                          "reduction": c["wall_time_reduction"], "removed": c["removed_read_fraction"],
                          "criterion": c["criterion_reduction_ge_0.7x_removed"]}
            if c.get("criterion_on_dram_bytes"):
                out[short]["criterion_dram"] = {k: c["criterion_on_dram_bytes"][k] for k in ("removed_dram_fraction", "met")}
    m = line.get("mla")
    if m:
        out["mla"] = {"ms": m["rep_stats"], "partial_tflops": m["partial_kernel_tflops"],
                      "partial_frac_bf16_burst": m["partial_kernel_frac_of_burst_bf16"]}
    c = line.get("cpu_baseline")
    if c:
        out["cpu"] = {"all_cores_gbs": c["value_all_cores"], "cores": c["cores_all"], "one_core_gbs": c["value_1_core"]}
    return out


def run_ours(args):
    rank, world, local = dist_setup(args.gpus)
    w = synth.flat_decode(seed=0, canary=False)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(w)          # its worker pool forks before CUDA is initialised
    torch.cuda.set_device(local)
    hbm, bf16, bf16s, peak_src = measured_peaks()
    flush = L2Flush(args.l2_flush)

    arm = Arm(w, enable=1)
    arm.step()
    arm.check()
    kv_bytes = unique_kv_bytes(w)

    barrier(world)
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        host_us = []
        times = time_steps(arm.step, args.steps, args.warmup, flush, host_us)
        barrier(world)
        t_wall = time.perf_counter() - t_wall0
        kt = kernel_timing(arm, args.steps, args.warmup, flush)
        kt_cc = kernel_timing(arm, args.steps, args.warmup, flush, "cuda_core")
    arm.check()
    algo = partial_algorithmic_bytes(arm)
    merge_bytes = merge_algorithmic_bytes(arm)
    ms = statistics.mean(times)
    value, ms_max = replica_throughput(kv_bytes, ms, world)
    k_ms = kt["partial_ms"]
    achieved = algo / (k_ms * 1e-3) / 1e9
    k_ms_cc = kt_cc["partial_ms"]
    achieved_cc = algo / (k_ms_cc * 1e-3) / 1e9
    merge_gbs = merge_bytes / (kt["merge_ms"] * 1e-3) / 1e9

    et, h2d, d2h, wall = e2e_timing(arm, args.steps, args.warmup, flush)
    e2e_ms = dist_max(statistics.mean(et), world)
    gate = no_sharing_gate(arm, args.steps, args.warmup, flush)

    extra = {}
    if not args.quick and args.workload in ("all", "cascade"):
        # cascade workload: flat arm vs cascade arm on the same inputs
        wc = synth.cascade_decode(seed=0, canary=False)
        extra["flat_vs_cascade"] = cascade_comparison(
            wc, "cascade decode: 64 requests, 16 share an 8192-token prefix (suffix U[64,1024]), "
                "48 independent U[512,4096]; Hq=32, Hkv=8, D=128, page 16, tile 512", args, flush, plan_us=True,
            key="flat_vs_cascade")
    if not args.quick and args.workload in ("all", "cascade", "cascade_l2"):
        # The same batch with a 65536-token shared prefix (268 MB of K/V, more than the
        # 129 MB L2), so the flat arm's re-reads of the prefix go to DRAM.
        wl = synth.cascade_decode(seed=0, canary=False, shared_tokens=65536)
        extra["flat_vs_cascade_prefix_beyond_l2"] = cascade_comparison(
            wl, "cascade decode, prefix larger than L2: 64 requests, 16 share a 65536-token prefix "
                "(suffix U[64,1024]), 48 independent U[512,4096]; Hq=32, Hkv=8, D=128, page 16, tile 512",
            args, flush, key="flat_vs_cascade_prefix_beyond_l2")
    if not args.quick and args.workload in ("all", "mla"):
        wm = synth.mla_decode(seed=0, canary=False, batch=args.mla_batch)
        marm = Arm(wm, enable=1)
        marm.step()
        marm.check()
        tms = time_steps(marm.step, max(5, args.steps // 2), args.warmup, flush)
        tm = statistics.mean(tms)
        km = kernel_timing(marm, max(3, args.steps // 2), 1, flush)
        mb = unique_kv_bytes(wm)
        flops = float(np.sum(wm.lengths)) * wm.Hq * (wm.Dqk + wm.Dv) * 2
        extra["mla"] = {
            "workload": f"MLA decode: {wm.batch} requests U[4096,32768], 128 heads, latent 576 fp8-e4m3 "
                        "(V = first 512), page 64, tile 2048",
            "ms": round(tm, 4), "rep_stats": rep_stats(tms), "tokens_per_s": round(wm.batch / (tm * 1e-3), 1),
            "unique_kv_gbs": round(mb / (tm * 1e-3) / 1e9, 1),
            "tflops": round(flops / (tm * 1e-3) / 1e12, 1),
            "tensor_frac_of_sustained_bf16": round(flops / (tm * 1e-3) / 1e12 / bf16s, 4) if bf16s else None,
            "kernels_ms": {k: round(v, 4) for k, v in km.items()},
            "partial_kernel_tflops": round(flops / (km["partial_ms"] * 1e-3) / 1e12, 1),
            "partial_kernel_frac_of_burst_bf16": round(flops / (km["partial_ms"] * 1e-3) / 1e12 / bf16, 4),
        }
        del marm
    if not args.quick and args.workload in ("all", "merge"):
        sizes = tuple(int(x) for x in args.merge_rows.split(",")) if args.merge_rows else \
            (1024, 16384, 262144, 1048576)
        extra["merge_sweep"] = merge_sweep(arm.ctx, args.steps, args.warmup, flush, hbm, sizes)
    if not args.quick and args.workload in ("all", "cascade", "nested"):
        extra["nested"] = nested_timing(args.steps, args.warmup, flush)
    if not args.quick and args.workload in ("all", "large"):
        extra["flat_decode_128_requests"] = large_flat_timing(args, flush, hbm)
    if not args.quick and args.workload in ("all", "tune"):
        extra["autotune"] = autotune_report(arm, max(3, args.steps // 4))
    if not args.quick and args.workload in ("all", "append"):
        extra["rope_append"] = rope_append_timing(arm.ctx, args.steps, args.warmup, flush)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_max, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": flat_config(w, kv_bytes, args.l2_flush),
            "rep_stats": rep_stats(times),
            "timing_notes": {"flush_us": round(flush_us(flush), 1),
                             "host_enqueue_us": round(statistics.mean(host_us), 1),
                             "replicas": world,
                             "lengths": "L~U[512,4096] with a partial last page (no multiple of 16)"},
            "decode_tokens_per_s": round(world * w.batch / (ms_max * 1e-3), 1),
            "pct_of_nominal_8TBs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "pct_of_measured_hbm": round(100 * value / world / hbm, 2),
            "roofline": {"bound": "hbm",
                         "kernel": "partial_tcs_kernel<128> (split-KV partial, 16-row-group tensor cores)",
                         "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "peak_source": peak_src + " copy bandwidth",
                         "traffic": partial_traffic(), "algorithmic_bytes_per_launch": algo,
                         "launch_ms": round(k_ms, 5)},
            "merge_kernel": {"kernel": "merge_states_kernel<1>", "achieved": round(merge_gbs, 1),
                             "unit": "GB/s", "frac": round(merge_gbs / hbm, 4),
                             "launch_ms": round(kt["merge_ms"], 5), "algorithmic_bytes": merge_bytes,
                             "note": "3.3 MB per launch on this batch, so latency sets its time; "
                                     "merge_sweep measures its bandwidth"},
            "partial_cuda_core": {"kernel": "partial_cc_kernel<128,4> (split-KV partial, CUDA cores)",
                                  "achieved": round(achieved_cc, 1), "unit": "GB/s",
                                  "frac": round(achieved_cc / hbm, 4), "launch_ms": round(k_ms_cc, 5)},
            "e2e": {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h),
                    "wall_ms_median": round(statistics.median(wall), 5),
                    "wall_gbs": round(world * kv_bytes / (statistics.median(wall) * 1e-3) / 1e9, 1),
                    "transfers": "inputs: query rows and page ids read by the partial kernel from "
                                 "pinned host memory (no staging copy); plan: launch parameters; "
                                 "outputs: merge-kernel stores into pinned host memory"},
            "gpu_launches": arm.launches_per_step() * args.steps,
            "wall_s": round(t_wall, 3),
            "clocks": clk.summary(),
        }
        line["no_sharing_gate"] = gate
        line.update(extra)
        if cpu is not None:
            line["cpu_baseline"] = cpu
        line["summary"] = headline_summary(line)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The oracle timed on the host cores on the flat workload (rank 0 only): each step
    is one pass over the whole batch, its (request, KV head) tasks spread over every
    core this process may use."""
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return
    w = synth.flat_decode(seed=0, canary=False)
    kv_bytes = unique_kv_bytes(w)
    op = OraclePool(w)
    try:
        for _ in range(args.warmup):
            op.pass_all_cores()
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            nbytes = op.pass_all_cores()
            times.append((time.perf_counter() - t0) * 1e3)
    finally:
        op.close()
    dt = statistics.mean(times)
    value = nbytes / (dt * 1e-3) / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": flat_config(w, kv_bytes, args.l2_flush),
        "rep_stats": rep_stats(times),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": op.cores, "kind": "oracle",
                         "sample": f"whole {w.name} batch per step: {len(op.tasks)} (request, KV head) "
                                   "tasks of the float64 numpy oracle on all cores; no GPU, so the "
                                   "L2 flush of the config does not apply"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--quick", action="store_true", help="flat workload only")
    p.add_argument("--workload", choices=["all", "cascade", "cascade_l2", "mla", "merge", "append", "nested", "tune",
                                          "large"],
                   default="all",
                   help="which workloads run after the flat headline")
    p.add_argument("--mla-batch", type=int, default=128, help="requests in the MLA workload")
    p.add_argument("--merge-rows", default="", help="merge sweep sizes, comma-separated (default 1K,16K,256K,1M)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--l2-flush", choices=["write+read", "write"], default="write+read",
                   help="L2 flush before each timed step (see L2Flush)")
    args = p.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
