#!/usr/bin/env python3
"""Benchmark of the FlashAttention-2 forward pass on GB300.

One step = one forward pass (the whole path: tile scheduling, Q/K/V tile
loads, S = Q K^T, masking, online softmax, O += P V, epilogue) over the
headline workload, bf16 B=4 H=16 N=4096 d=128 causal, with Q, K, V resident
in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With --pass bwd a step is one backward pass instead (fa_bwd: D = rowsum(dO*O),
the dK/dV kernel and the dQ kernel, with Q, K, V, O, L and dO resident), and
the line reports TFLOP/s over 2.5x the forward's algorithmic FLOPs.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas: the path needs no exchange between GPUs), the timed
region is bracketed by a barrier and a synchronize on both sides, the time
is the max over ranks, and `value` counts the work of all ranks.
"""
from __future__ import annotations

import os

# The CPU oracle (baseline and reference legs) runs one head per worker
# process; each worker's BLAS is single-threaded.  Must be set before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import csv
import hashlib
import io
import json
import multiprocessing as mp
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FA2 fwd TFLOP/s, bf16 B4 H16 N4096 d128 causal; % of GB300 dense peak"
FP8_METRIC = "FA2 fwd TFLOP/s, fp8 (e4m3) inputs, bf16 output; % of GB300 dense fp8 peak"
FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)
BWD_METRIC = "FA2 bwd TFLOP/s (2.5x the forward's algorithmic FLOPs), bf16; % of GB300 dense peak"
BWD_FLOP_FACTOR = 2.5  # dV = P^T dO, dP = dO V^T, dQ = dS K, dK = dS^T Q, plus S = Q K^T recomputed
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20  # larger than the 129 MB L2
KERNEL_SOURCES = ["tiled_attention_fwd_gb300/csrc/fa_fwd_tc.cuh", "tiled_attention_fwd_gb300/csrc/ptx.cuh",
                  "tiled_attention_fwd_gb300/csrc/fa_tc_launch.cuh"]
BWD_KERNEL_SOURCES = ["tiled_attention_fwd_gb300/csrc/fa_bwd_tc.cuh", "tiled_attention_fwd_gb300/csrc/ptx.cuh",
                      "tiled_attention_fwd_gb300/csrc/fa_bwd_launch.cuh"]


# ------------------------------------------------------------------ helpers
def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for p in (KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str, prefix: str = "traffic", sources=None):
    """dram bytes per launch from a committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", f"{prefix}_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, one sample every `period_ms`, each
    stamped on arrival with the host clock (time.perf_counter) by a reader
    thread, so that the samples can be binned against the timed region.

    The benchmark keeps the GPU under the same load (the same L2 flush + step
    sequence, untimed) for a while before and after its timed steps; `sm_mhz`
    is the median over that whole load window, which contains the timed
    region, and the samples that fall inside the timed region itself are
    reported separately."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.thread = None
        self.samples = []  # (perf_counter seconds, csv row)
        self.marks = {}

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line))

    def __enter__(self):
        import threading

        exe = shutil.which("nvidia-smi")
        if exe is not None:
            self.proc = subprocess.Popen([exe, f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        return self

    def mark(self, name: str):
        self.marks[name] = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    @staticmethod
    def _parse(rows):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in rows:
            r = next(csv.reader(io.StringIO(line)), [])
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return sm, smax, reasons

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        lo, hi = self.marks.get("load_start", 0.0), self.marks.get("load_end", float("inf"))
        t0, t1 = self.marks.get("timed_start", lo), self.marks.get("timed_end", hi)
        load = [line for t, line in self.samples if lo <= t <= hi]
        timed = [line for t, line in self.samples if t0 <= t <= t1]
        sm, smax, reasons = self._parse(load)
        sm_t, _, reasons_t = self._parse(timed)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons | reasons_t), "samples": len(sm),
                "samples_in_timed_region": len(sm_t),
                "sm_mhz_timed_region": statistics.median(sm_t) if sm_t else None,
                "period_ms": self.period_ms,
                "load_window_s": (hi - lo) if hi != float("inf") else None,
                "timed_region_s": (t1 - t0) if t1 != float("inf") else None,
                "note": "sm_mhz: median over a window of identical load (untimed flush + step sequences before "
                        "and after the timed steps) that contains the timed region"}


def soak(step_fn, seconds: float, sync):
    """Run `step_fn` back to back for about `seconds` (untimed; keeps the GPU
    under the timed region's load while the clock sampler runs)."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        for _ in range(8):
            step_fn()
        sync()


MUFU_EX2_PER_CLK_PER_SM = 32  # ex2.approx.ftz.f32 results per clock per SM, measured on GB300


def exp_rate(w, kernel_ms: float, sms: int, sm_mhz):
    """Exponentials of the softmax (one per unmasked score: B*H*N^2, halved when
    causal) per second, against the MUFU rate at the sampled SM clock."""
    n = float(w.B * w.H * w.N * w.N) / (2.0 if w.causal else 1.0)
    per_s = n / (kernel_ms / 1e3)
    mhz = sm_mhz if sm_mhz else 2070.0
    peak = MUFU_EX2_PER_CLK_PER_SM * sms * mhz * 1e6
    return {"per_launch": n, "per_s": per_s, "peak_per_s": peak, "frac": per_s / peak,
            "peak_basis": f"{MUFU_EX2_PER_CLK_PER_SM} ex2/clk/SM x {sms} SMs x {mhz:.0f} MHz"}


def aggregate_ranks(local_seconds: float, world: int, reduce_max=None) -> float:
    """Max over ranks of the timed-region duration (identity on one rank)."""
    if world <= 1 or reduce_max is None:
        return local_seconds
    return reduce_max(local_seconds)


def make_reduce_max(dist, device):
    """All-reduce(MAX) of one float over the default process group."""
    import torch

    def reduce_max(x: float) -> float:
        t = torch.tensor([x], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return reduce_max


def job_throughput(world: int, steps: int, flops_per_step: float, seconds: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of `flops_per_step` in `seconds` (max over ranks)."""
    return world * steps * flops_per_step / seconds / 1e12


# ------------------------------------------------------------------ CPU oracle legs
def _oracle_head(args):
    import numpy as np  # noqa: F401  (worker process: BLAS single-threaded by env)

    import oracle
    q, k, v, scale, causal = args
    t0 = time.perf_counter()
    oracle.attention_head(q, k, v, scale, causal)
    return time.perf_counter() - t0


def _oracle_bwd_head(args):
    import oracle
    q, k, v, do, scale, causal = args
    t0 = time.perf_counter()
    oracle.attention_backward_head(q, k, v, do, scale, causal)
    return time.perf_counter() - t0


def oracle_sample(w, budget_s: float, pool, cores: int, inputs=None, backward=False):
    """Run the fp64 oracle (forward, or backward given dO) on whole heads of
    workload `w` for about `budget_s` seconds on `cores` worker processes;
    returns (TFLOP/s, heads, seconds), counting the algorithmic FLOPs."""
    from tiled_attention_fwd_gb300.inputs import as_f64_numpy, make_dout, make_qkv

    q, k, v = make_qkv(w) if inputs is None else inputs
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    per_head = w.flops / len(heads) * (BWD_FLOP_FACTOR if backward else 1.0)
    qn, kn, vn = as_f64_numpy(q), as_f64_numpy(k), as_f64_numpy(v)
    don = as_f64_numpy(make_dout(w)) if backward else None
    t0 = time.perf_counter()

    def submit(i):
        b, h = heads[i]
        if backward:
            return pool.apply_async(_oracle_bwd_head, ((qn[b, h], kn[b, h], vn[b, h], don[b, h], w.scale, w.causal),))
        return pool.apply_async(_oracle_head, ((qn[b, h], kn[b, h], vn[b, h], w.scale, w.causal),))

    pending = [submit(i) for i in range(min(cores, len(heads)))]
    nxt, done = len(pending), 0
    while pending:
        pending.pop(0).get()
        done += 1
        if nxt < len(heads) and time.perf_counter() - t0 < budget_s:
            pending.append(submit(nxt))
            nxt += 1
    dt = time.perf_counter() - t0
    return done * per_head / dt / 1e12, done, dt


def make_pool(cores: int):
    ctx = mp.get_context("spawn")
    return ctx.Pool(cores)


def workload_inputs(w):
    """Host inputs of workload w: (q, k, v) in its dtype, plus the three
    dequantisation factors for e4m3 workloads (None otherwise)."""
    from tiled_attention_fwd_gb300.inputs import make_qkv, make_qkv_fp8

    if w.dtype == "fp8":
        return make_qkv_fp8(w)
    return make_qkv(w), None


def oracle_inputs(w, qkv, factors):
    """The real-valued inputs the oracle takes: e4m3 values times their factors
    (exact in fp32 for the power-of-two factors of the synthetic inputs)."""
    if factors is None:
        return qkv
    return tuple(x.float() * f for x, f in zip(qkv, factors))


# ------------------------------------------------------------------ reference arm
def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    pool = make_pool(cores)
    inputs = oracle_inputs(w, *workload_inputs(w))
    bwd = args.pass_ == "bwd"
    budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, budget, pool, cores, inputs, backward=bwd)
    vals, heads, secs = [], 0, 0.0
    for _ in range(args.steps):
        v, h, s = oracle_sample(w, budget, pool, cores, inputs, backward=bwd)
        vals.append(v)
        heads += h
        secs += s
    pool.close()
    value = heads * (w.flops / (w.B * w.H)) * (BWD_FLOP_FACTOR if bwd else 1.0) / secs / 1e12
    sample = (f"whole heads of the workload, as many as fit in ~{budget:.0f} s per step on {cores} worker "
              f"processes (one head each, fp64 {'backward' if bwd else 'forward'}, BLAS single-threaded); "
              f"{heads} heads in {args.steps} steps")
    line = {
        "impl": "reference", "metric": BWD_METRIC if bwd else (FP8_METRIC if w.dtype == "fp8" else METRIC),
        "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w):
    inputs = f"seeded iid normal (seed {w.seed}, Q/K std {w.qk_std})"
    if w.dtype == "fp8":
        inputs += ", quantised to e4m3 with one power-of-two factor per tensor; O bf16"
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "dtype": w.dtype, "inputs": inputs,
            "l2": "flushed (256 MB write) between timed steps", "layout": "[B,H,N,d] contiguous"}


# ------------------------------------------------------------------ our arm
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import tiled_attention_fwd_gb300 as fa

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    want_cpu = (not args.no_cpu_baseline) and rank == 0 and world == 1
    cores = os.cpu_count() or 1
    pool = make_pool(cores) if want_cpu else None  # spawn before the first GPU call

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    reduce_max = None
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
        reduce_max = make_reduce_max(dist, dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    (q, k, v), factors = workload_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty(q.shape, device=dev, dtype=torch.bfloat16 if w.dtype == "fp8" else q.dtype)
    lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    fn = {"bf16": fa.fa_fwd, "f32": fa.fa_fwd_f32, "fp8": fa.fa_fwd_fp8}[w.dtype]
    extra = tuple(factors) if factors is not None else ()

    def step():
        rc = fn(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N, w.d,
                w.scale, *extra, w.causal, sh)
        if rc != 0:
            raise fa.FAError(rc, fn.__name__)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    fa.check_status(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]

    def load_step():
        flush.zero_()
        step()

    with ClockSampler(local) as clocks:
        clocks.mark("load_start")
        soak(load_step, args.clock_soak_s, torch.cuda.synchronize)
        barrier()
        clocks.mark("timed_start")
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()  # outside the events: L2 holds no inputs when each step starts
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        barrier()
        t_wall = time.perf_counter() - t_wall
        clocks.mark("timed_end")
        soak(load_step, args.clock_soak_s / 4, torch.cuda.synchronize)
        clocks.mark("load_end")
    fa.check_status(dev)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    local_s = sum(step_ms) / 1e3
    total_s = aggregate_ranks(local_s, world, reduce_max)
    value = job_throughput(world, args.steps, w.flops, total_s)
    kernel_ms = statistics.mean(step_ms)

    # End to end through the C ABI on HOST buffers: H2D of Q, K, V from pinned
    # memory, the forward pass, D2H of O and L, every step.
    e2e = None
    if not args.no_e2e and w.dtype == "bf16":
        qp, kp, vp = (t.pin_memory() for t in (q, k, v))
        op = torch.empty_like(qp).pin_memory()
        lp = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
        nbytes = fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.N, w.d)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def host_step():
            rc = fa.fa_fwd_host(qp.data_ptr(), kp.data_ptr(), vp.data_ptr(), op.data_ptr(), lp.data_ptr(),
                                ws.data_ptr(), nbytes, w.B, w.H, w.N, w.d, w.scale, w.causal, sh)
            if rc != 0:
                raise fa.FAError(rc, "fa_fwd_host")

        for _ in range(max(1, args.warmup)):
            host_step()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            host_step()
        e1.record(stream)
        barrier()
        e2e_s = aggregate_ranks(e0.elapsed_time(e1) / 1e3, world, reduce_max)
        tb = w.B * w.H * w.N * w.d * 2
        e2e = {"value": job_throughput(world, args.steps, w.flops, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": 3 * tb, "d2h_bytes_per_step": tb + w.B * w.H * w.N * 4,
               "ms_per_step": e2e_s / args.steps * 1e3, "api": "fa_fwd_host (C ABI, pinned host buffers)"}
        fa.check_status(dev)
    if not args.no_e2e and w.dtype == "fp8":
        # e4m3 inputs: the public Python API on pinned host tensors (H2D of the
        # three e4m3 tensors, fa_fwd_fp8, D2H of O and L), every step.
        hq, hk, hv = (t.pin_memory() for t in (q, k, v))
        ho = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        hl = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
        dq8, dk8, dv8 = (torch.empty_like(qd) for _ in range(3))

        def host_step():
            for src, dst in zip((hq, hk, hv), (dq8, dk8, dv8)):
                dst.copy_(src, non_blocking=True)
            fa.forward_fp8(dq8, dk8, dv8, factors, causal=w.causal, scale=w.scale, out=o, lse=lse)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            host_step()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            host_step()
        e1.record(stream)
        barrier()
        e2e_s = aggregate_ranks(e0.elapsed_time(e1) / 1e3, world, reduce_max)
        n = w.B * w.H * w.N * w.d
        e2e = {"value": job_throughput(world, args.steps, w.flops, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": 3 * n, "d2h_bytes_per_step": 2 * n + w.B * w.H * w.N * 4,
               "ms_per_step": e2e_s / args.steps * 1e3,
               "api": "tiled_attention_fwd_gb300.forward_fp8 (pinned host tensors, copies on the stream)"}
        fa.check_status(dev)

    cpu = None
    if want_cpu:
        tflops, heads, secs = oracle_sample(w, args.cpu_seconds, pool, cores, oracle_inputs(w, (q, k, v), factors))
        cpu = {"value": tflops, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{heads} whole heads of the workload (fp64 standard attention, one head per worker "
                         f"process, {cores} processes, BLAS single-threaded) in {secs:.1f} s"}
    if pool is not None:
        pool.close()

    peaks, src = load_peaks()
    peak = peaks["bf16_tflops"] * (FP8_OVER_BF16 if w.dtype == "fp8" else 1.0)
    achieved = w.flops / (kernel_ms / 1e3) / 1e12
    clock_rec = clocks.summary()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    exps = exp_rate(w, kernel_ms, sms, clock_rec.get("sm_mhz"))
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": load_traffic(w.name),
            "peak_source": (f"fp8 dense = bf16 dense burst ({src}) x {FP8_OVER_BF16:g}, the nominal fp8/bf16 ratio"
                            if w.dtype == "fp8" else f"bf16 dense burst, {src}"),
            "kernel": {"bf16": f"fa_fwd_tc_kernel<{w.d},{str(w.causal).lower()}>",
                       "fp8": f"fa_fwd_tc_kernel<{w.d},{str(w.causal).lower()},e4m3>",
                       "f32": "fa_fwd_simt_kernel"}[w.dtype],
            "flops_per_launch": w.flops}
    if rank == 0:
        line = {
            "metric": FP8_METRIC if w.dtype == "fp8" else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": config_of(w), "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": clock_rec, "exp": exps,
            "kernel_ms": {"mean": kernel_ms, "min": min(step_ms), "max": max(step_ms),
                          "median": statistics.median(step_ms)},
            "wall_s_timed_region": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_ours_bwd(args, w):
    """The backward pass (fa_bwd: preprocessing + dK/dV + dQ kernels) of workload `w`."""
    import torch
    import torch.distributed as dist

    import tiled_attention_fwd_gb300 as fa
    from tiled_attention_fwd_gb300.inputs import make_dout, make_qkv

    if w.dtype != "bf16" or w.d not in (32, 64, 128, 256):
        raise SystemExit(f"the backward pass covers bf16 with d in (32, 64, 128, 256), not {w.name}")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    want_cpu = (not args.no_cpu_baseline) and rank == 0 and world == 1
    cores = os.cpu_count() or 1
    pool = make_pool(cores) if want_cpu else None  # spawn before the first GPU call

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    reduce_max = None
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
        reduce_max = make_reduce_max(dist, dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    q, k, v = make_qkv(w)
    do = make_dout(w)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    nws = fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flops = BWD_FLOP_FACTOR * w.flops

    def step():
        rc = fa.fa_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), dod.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N, w.d, w.scale, w.causal,
                       ws.data_ptr(), nws, sh)
        if rc != 0:
            raise fa.FAError(rc, "fa_bwd")

    for _ in range(args.warmup):
        flush.zero_()
        step()
    fa.check_status(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]

    def load_step():
        flush.zero_()
        step()

    with ClockSampler(local) as clocks:
        clocks.mark("load_start")
        soak(load_step, args.clock_soak_s, torch.cuda.synchronize)
        barrier()
        clocks.mark("timed_start")
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        barrier()
        t_wall = time.perf_counter() - t_wall
        clocks.mark("timed_end")
        soak(load_step, args.clock_soak_s / 4, torch.cuda.synchronize)
        clocks.mark("load_end")
    fa.check_status(dev)
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_s = aggregate_ranks(sum(step_ms) / 1e3, world, reduce_max)
    value = job_throughput(world, args.steps, flops, total_s)
    kernel_ms = statistics.mean(step_ms)

    # End to end through the public Python API on HOST tensors: copies of Q, K,
    # V, O, L and dO from pinned memory, backward(), copies of dQ, dK, dV back.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
        ho, hl = o.cpu().pin_memory(), lse.cpu().pin_memory()
        outs = [torch.empty_like(hq).pin_memory() for _ in range(3)]
        dev_in = [torch.empty_like(qd) for _ in range(5)]
        dev_l = torch.empty_like(lse)

        def host_step():
            for src, dst in zip((hq, hk, hv, ho, hdo), dev_in):
                dst.copy_(src, non_blocking=True)
            dev_l.copy_(hl, non_blocking=True)
            grads = fa.backward(*dev_in[:4], dev_l, dev_in[4], causal=w.causal, scale=w.scale, workspace=ws)
            for src, dst in zip(grads, outs):
                dst.copy_(src, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            host_step()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            host_step()
        e1.record(stream)
        barrier()
        e2e_s = aggregate_ranks(e0.elapsed_time(e1) / 1e3, world, reduce_max)
        tb = w.B * w.H * w.N * w.d * 2
        e2e = {"value": job_throughput(world, args.steps, flops, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": 5 * tb + w.B * w.H * w.N * 4, "d2h_bytes_per_step": 3 * tb,
               "ms_per_step": e2e_s / args.steps * 1e3, "api": "tiled_attention_fwd_gb300.backward (pinned host tensors)"}
        fa.check_status(dev)

    cpu = None
    if want_cpu:
        tflops, heads, secs = oracle_sample(w, args.cpu_seconds, pool, cores, (q, k, v), backward=True)
        cpu = {"value": tflops, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{heads} whole heads of the workload (fp64 backward, one head per worker process, "
                         f"{cores} processes, BLAS single-threaded) in {secs:.1f} s"}
    if pool is not None:
        pool.close()

    peaks, src = load_peaks()
    peak = peaks["bf16_tflops"]
    achieved = flops / (kernel_ms / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": load_traffic(w.name, "traffic_bwd", BWD_KERNEL_SOURCES),
            "peak_source": f"bf16 dense burst, {src}",
            "kernel": f"fa_bwd_prep_kernel<{w.d}> + fa_bwd_tc_kernel<{w.d},0,{str(w.causal).lower()}> + "
                      f"fa_bwd_tc_kernel<{w.d},1,{str(w.causal).lower()}>",
            "flops_per_launch": flops,
            "note": "achieved counts 2.5x the forward's FLOPs over the three kernels' time; the split "
                    "dK/dV + dQ kernels execute 3.5x (S and dP are recomputed in both)"}
    if rank == 0:
        line = {
            "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(config_of(w), **{"pass": "backward", "dO": f"seeded iid normal (seed {w.seed + 1000})"}),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 3 * args.steps, "clocks": clocks.summary(),
            "kernel_ms": {"mean": kernel_ms, "min": min(step_ms), "max": max(step_ms),
                          "median": statistics.median(step_ms)},
            "wall_s_timed_region": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ per-config report
REPORT_WORKLOADS = [
    "f32_b1h1n128d16", "f32_b1h1n128d16_causal", "bf16_b8h1n1024d64", "bf16_b8h1n1024d64_causal",
    "bf16_b4h16n4096d128_causal", "bf16_b1h32n16384d128_causal", "bf16_b2h16n8192d32_qk3",
    "bf16_b2h16n8192d64_qk3", "bf16_b2h16n8192d128_qk3", "bf16_b2h16n8192d256_qk3",
    "fp8_b4h16n4096d128_causal", "fp8_b2h16n8192d128_qk3",
]


def run_report(args):
    """Every config once: the forward's CUDA-event time over >= 20 launches (L2
    flushed before each; median, min, max), its TFLOP/s and fraction of the
    dense bf16 peak, beside the fp64 oracle timed in the same run on the host
    cores (whole heads for about --report-cpu-seconds each; heads cost the same,
    so the full config's oracle time is that rate scaled to all heads)."""
    import torch

    from tiled_attention_fwd_gb300 import check_status, fa_fwd, fa_fwd_f32, fa_fwd_fp8
    from tiled_attention_fwd_gb300.inputs import WORKLOADS

    cores = os.cpu_count() or 1
    pool = make_pool(cores)  # spawned before the first GPU call
    peaks, peak_src = load_peaks()
    peak = peaks["bf16_tflops"]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    runs = max(20, args.steps)
    rows = []
    for name in REPORT_WORKLOADS:
        w = WORKLOADS[name]
        host, factors = workload_inputs(w)
        q, k, v = (t.to(dev) for t in host)
        o = torch.empty(q.shape, device=dev, dtype=torch.bfloat16 if w.dtype == "fp8" else q.dtype)
        lse = torch.empty(q.shape[:-1], device=dev, dtype=torch.float32)

        fn = {"bf16": fa_fwd, "f32": fa_fwd_f32, "fp8": fa_fwd_fp8}[w.dtype]
        extra = tuple(float(f) for f in factors) if factors is not None else ()
        call = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N, w.d,
                float(w.scale), *extra, int(w.causal), torch.cuda.current_stream(dev).cuda_stream)

        def launch():  # the C ABI directly, so that no host work sits between the events
            rc = fn(*call)
            if rc != 0:
                raise RuntimeError(f"{fn.__name__} returned {rc}")

        for _ in range(max(3, args.warmup)):
            flush.zero_()
            launch()
        check_status(dev)
        times = []
        for _ in range(runs):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            launch()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        check_status(dev)
        med = statistics.median(times)
        tflops = w.flops / (med * 1e-3) / 1e12
        exps = exp_rate(w, med, torch.cuda.get_device_properties(dev).multi_processor_count, None)
        ora, heads, secs = oracle_sample(w, args.report_cpu_seconds, pool, cores, oracle_inputs(w, host, factors))
        own_peak = peak * (FP8_OVER_BF16 if w.dtype == "fp8" else 1.0)
        row = {"workload": name, "dtype": w.dtype, "causal": w.causal, "gflop": w.flops / 1e9,
               "gpu_ms_median": med, "gpu_ms_min": min(times), "gpu_ms_max": max(times), "runs": runs,
               "tflops": tflops, "frac_of_bf16_peak": tflops / peak, "frac_of_own_peak": tflops / own_peak,
               "peak_tflops": own_peak, "peak_source": peak_src,
               "exp_per_s": exps["per_s"], "exp_frac_of_mufu": exps["frac"],
               "oracle_tflops": ora, "oracle_heads": heads, "oracle_s": secs,
               "oracle_full_s": w.flops / (ora * 1e12), "oracle_cores": cores}
        rows.append(row)
        print(json.dumps(row), flush=True)
    pool.close()
    print(f"\n| config | GFLOP | GPU median / min / max (ms, {runs} runs) | TFLOP/s | of bf16 peak | "
          f"of own dtype's peak | exp/s (of MUFU at 2070 MHz) | CPU oracle ({cores} cores): TFLOP/s | "
          f"oracle s, full config |")
    print("|---|---|---|---|---|---|---|---|---|")
    for r in rows:
        print(f"| `{r['workload']}` | {r['gflop']:.3g} | {r['gpu_ms_median']:.4f} / {r['gpu_ms_min']:.4f} / "
              f"{r['gpu_ms_max']:.4f} | {r['tflops']:.4g} | {r['frac_of_bf16_peak']:.3g} | "
              f"{r['frac_of_own_peak']:.3g} | "
              f"{r['exp_per_s']:.3g} ({r['exp_frac_of_mufu']:.3g}) | "
              f"{r['oracle_tflops']:.3g} | {r['oracle_full_s']:.3g} |")
    return 0


def main(argv=None):
    from tiled_attention_fwd_gb300.inputs import HEADLINE, WORKLOADS

    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU oracle sample budget")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="forward pass (the headline) or backward pass (fa_bwd)")
    ap.add_argument("--report", action="store_true",
                    help="time the forward on every config beside the CPU oracle and print a table")
    ap.add_argument("--report-cpu-seconds", type=float, default=8.0, help="CPU oracle budget per config in --report")
    ap.add_argument("--clock-soak-s", type=float, default=0.3,
                    help="seconds of identical untimed load before the timed steps (a quarter of it after), "
                         "so that the clock samples bracket the timed region")
    args = ap.parse_args(argv)
    if args.report:
        return run_report(args)
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.pass_ == "bwd":
        return run_ours_bwd(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
