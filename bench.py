"""Benchmark of the FlashAttention-2 forward pass on GB300.

One step = one forward pass (the whole hot path: tile loads, S = Q K^T,
masking, online softmax, P V, normalisation, LSE) over one batch of seeded
synthetic bf16 inputs already resident in HBM.  The default workload is
B=1, H=32, Nq=Nk=16384, d=128, causal -- the head count, head dimension and
long-sequence regime of the FlashAttention-2 utilisation table in
"FlashAttention-2 算法架构升级" (section 四).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                        [--impl reference]
For N > 1 launch one process per GPU with torch.distributed.run; every rank
runs an independent replica (the pass has no exchange step) and rank 0
prints one JSON line with the whole-job throughput.

``--impl reference`` times the fp64 CPU oracle on this arm's workload (a
bounded row sample per step) on the host cores and prints the same JSON
line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from exact_attention_17_gb300 import inputs  # noqa: E402

METRIC = "FA2 fwd TFLOP/s (causal-halved) and % of GB300 dense-BF16 tensor peak"
METRIC_BWD = "FA2 bwd TFLOP/s (5 GEMMs = 2.5x fwd FLOPs, causal-halved) and % of GB300 dense-BF16 tensor peak"
DEFAULT_WORKLOAD = "b1_h32_n16384_d128_causal"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
BWD_KERNEL_SOURCES = ["exact_attention_17_gb300/csrc/fa2_bwd_sm103.cuh",
                      "exact_attention_17_gb300/csrc/ptx.cuh",
                      "exact_attention_17_gb300/csrc/fa2_bwd.cu"]
KERNEL_SOURCES = ["exact_attention_17_gb300/csrc/fa2_fwd_sm103.cuh",
                  "exact_attention_17_gb300/csrc/ptx.cuh",
                  "exact_attention_17_gb300/csrc/fa2_tc_d128_bf16.cu"]


def fwd_kernel_sources(d: int, fp16: bool = False):
    """Sources of the forward kernel a workload runs (head dimension, element type)."""
    return KERNEL_SOURCES[:2] + [f"exact_attention_17_gb300/csrc/fa2_tc_d{d}_{'f16' if fp16 else 'bf16'}.cu"]


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_bytes_backward(w) -> float:
    """Q, K, V and dO read once as bf16, O (fp32) and LSE read once; dQ, dK and
    dV written once as fp32."""
    return w.B * w.H * (2.0 * w.Nq * w.d + 4.0 * w.Nk * w.d + 2.0 * w.Nq * w.d + 4.0 * w.Nq * w.d
                        + 4.0 * w.Nq + 4.0 * w.Nq * w.d + 8.0 * w.Nk * w.d)


def algorithmic_bytes(w, o_bytes: int = 4) -> float:
    """Q, K, V read once as 16-bit values; O written once (fp32 unless
    `o_bytes` says otherwise) and the fp32 LSE written once."""
    return w.B * w.H * (2.0 * w.Nq * w.d + 4.0 * w.Nk * w.d + o_bytes * w.Nq * w.d + 4.0 * w.Nq)


def recorded_traffic(workload: str, sources=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples taken during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
            self.thread.join(timeout=5)

    def summary(self):
        if self.proc is None or not self.lines:
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- multi-rank aggregation

def job_time_ms(local_ms: float, dist=None, device=None) -> float:
    """Elapsed time of the whole job: the slowest replica's timed region."""
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step: float, steps: int, world: int, job_ms: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of the workload."""
    return flops_per_step * steps * world / (job_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- oracle (CPU) timing

def oracle_sample_rate(w, Q, K, V, budget_s: float, seed: int = 0):
    """Time the fp64 oracle on random rows of the workload for about budget_s.

    Returns (TFLOP/s, cores, rows, seconds); FLOPs per row are the algorithmic
    4 * |J_i| * d of that row (|J_i| = kept keys)."""
    import oracle

    qb, kb, vb = (inputs.bf16_bits(t) for t in (Q, K, V))
    cores = oracle.default_threads()
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.H * w.Nq
    flops = 0.0
    rows_done = 0
    batch = max(cores, 16)
    t0 = time.perf_counter()
    while True:
        rows = rng.integers(0, total_rows, size=batch)
        oracle.attention_rows(qb, kb, vb, w.causal, w.scale, rows, nthreads=cores)
        i = rows % w.Nq
        kept = np.minimum(i + 1, w.Nk) if w.causal else np.full_like(i, w.Nk)
        flops += float(np.sum(4.0 * kept * w.d))
        rows_done += batch
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
        batch = int(min(batch * 2, max(batch, rows_done * (budget_s - el) / max(el, 1e-3))))
        batch = max(batch, cores)
    return flops / el / 1e12, cores, rows_done, el


def backward_sample_shape(w, budget_s: float):
    """The oracle's backward on one head costs about 9 d flops per kept (query,
    key) pair and phase at roughly 4 Gflop/s per core: the largest leading
    square of one head that fits the budget (the whole head when it does)."""
    rate = 4e9 * (os.cpu_count() or 1)
    n = min(w.Nq, w.Nk)
    while n > 128:
        pairs = n * n / (2 if w.causal else 1)
        if 2 * 9 * w.d * pairs / rate <= budget_s:
            break
        n //= 2
    return n


def oracle_backward_rate(w, Q, K, V, G, budget_s: float):
    """Time the fp64 oracle's backward on one head (truncated to its leading
    n x n block when the whole head would exceed the budget).  Returns
    (TFLOP/s, cores, n, seconds) with the algorithmic 2.5x forward FLOPs of
    the timed problem."""
    import oracle

    n = backward_sample_shape(w, budget_s)
    qb, kb, vb, gb = (np.ascontiguousarray(inputs.bf16_bits(t)[:1, :1, :n]) for t in (Q, K, V, G))
    cores = oracle.default_threads()
    t0 = time.perf_counter()
    dtype = "fp16" if Q.dtype == torch.float16 else "bf16"
    oracle.attention_backward(qb, kb, vb, gb, w.causal, w.scale, nthreads=cores, dtype=dtype)
    el = time.perf_counter() - t0
    flops = 2.5 * 4.0 * n * n * w.d / (2 if w.causal else 1)
    return flops / el / 1e12, cores, n, el


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    Q, K, V = inputs.workload_inputs(w)
    if args.pass_ == "backward":
        return run_reference_backward(args, w, Q, K, V)
    per_step = []
    rows_total = 0
    cores = 0
    for s in range(args.warmup + args.steps):
        budget = 1.0 if s < args.warmup else args.reference_step_s
        tf, cores, rows, el = oracle_sample_rate(w, Q, K, V, budget, seed=s)
        if s >= args.warmup:
            per_step.append((tf, rows, el))
            rows_total += rows
    secs = sum(e for _, _, e in per_step)
    value = sum(tf * e for tf, _, e in per_step) / secs
    sample = (f"{rows_total} uniformly drawn query rows of {w.name} over {args.steps} steps "
              f"(~{args.reference_step_s:.0f} s each), fp64 three-pass oracle, FLOPs = 4*|J_i|*d per row")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1000 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": forward_config(w, args),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_backward(args, w, Q, K, V):
    G = inputs.draw_bf16((w.B, w.H, w.Nq, w.d), w.seed, 3)
    per_step = []
    cores, n = 0, 0
    for s in range(args.warmup + args.steps):
        budget = 1.0 if s < args.warmup else args.reference_step_s
        tf, cores, n, el = oracle_backward_rate(w, Q, K, V, G, budget)
        if s >= args.warmup:
            per_step.append((tf, el))
    secs = sum(e for _, e in per_step)
    value = sum(tf * e for tf, e in per_step) / secs
    sample = (f"head 0 of {w.name} truncated to its leading {n} queries and keys, once per step, "
              f"fp64 oracle backward, FLOPs = 2.5 x the forward's")
    line = {
        "impl": "reference", "metric": METRIC_BWD, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1000 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": backward_config(w, args),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129 * 1024 * 1024


def forward_l2_note(w):
    """Whether the forward arm flushes L2 between steps (inputs that would fit
    twice in L2 are flushed), as the note the config carries."""
    in_bytes = 2 * w.B * w.H * (w.Nq + 2 * w.Nk) * w.d
    if in_bytes <= 2 * L2_BYTES:
        return True, "L2 flushed between steps (256 MiB write, outside the kernel events)"
    return False, f"inputs {in_bytes / 2**20:.0f} MiB > 129 MiB L2, no flush"


def backward_l2_note(w):
    in_bytes = algorithmic_bytes_backward(w)
    if in_bytes <= 2 * L2_BYTES:
        return True, "L2 flushed between steps (256 MiB write, outside the kernel events)"
    return False, f"operands {in_bytes / 2**20:.0f} MiB > 129 MiB L2, no flush"


def forward_config(w, args):
    """The config object of the forward arms (the same for the GPU arm and the
    reference arm, so that the two lines describe one workload)."""
    return dict(workload_config(w, forward_l2_note(w)[1]), num_splits=args.num_splits,
                inputs=f"{args.dtype} BHSD",
                outputs=f"{'fp32' if args.out_dtype == 'fp32' else args.dtype} O, fp32 LSE")


def backward_config(w, args):
    return dict(workload_config(w, backward_l2_note(w)[1]), **{
        "pass": "backward", "inputs": f"{args.dtype} Q, K, V, dO; fp32 O, LSE",
        "outputs": "fp32 dQ, dK, dV"})


def workload_config(w, l2_note):
    return {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
            "causal": w.causal, "scale": w.scale, "qk_dist": f"{w.qk_dist}(std {w.qk_std})",
            "v_dist": w.v_dist, "seed": w.seed, "inputs": "bf16 BHSD", "outputs": "fp32 O, fp32 LSE",
            "l2": l2_note, "parallelism": "replicas"}


# ---------------------------------------------------------------- GPU arm

def roofline_entry(hbm_bound, achieved_tflops, peak_tflops, peak_src, peaks, traffic, flops,
                   algo_bytes, mean_launch_ms, kernel="fa2dev::fa2_fwd_tc_kernel"):
    """The roofline object for the forward kernel: against the measured HBM
    copy bandwidth when the workload sits below the machine balance, else
    against the measured bf16 tensor throughput."""
    common = {
        "traffic": traffic,
        "kernel": kernel,
        "flops_per_launch": flops,
        "algorithmic_bytes_per_launch": algo_bytes,
        "mean_launch_ms": round(mean_launch_ms, 4),
        "tensor_frac": round(achieved_tflops / peak_tflops, 4),
    }
    if hbm_bound:
        hbm = float(peaks["hbm_gbs"])
        gbs = algo_bytes / (mean_launch_ms * 1e-3) / 1e9
        return dict({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 4), "peak_kind": f"HBM copy ({peak_src})"}, **common)
    return dict({"bound": "tensor", "achieved": round(achieved_tflops, 2), "peak": peak_tflops,
                 "unit": "TFLOP/s", "frac": round(achieved_tflops / peak_tflops, 4),
                 "peak_kind": f"bf16 dense burst ({peak_src})",
                 "frac_of_sustained": round(achieved_tflops / float(peaks["bf16_tflops_sustained"]), 4)},
                **common)


def relaunch_distributed(n: int) -> int:
    """Run this same command as n ranks (one process per GPU) under
    torch.distributed.run on 127.0.0.1 and return its exit status."""
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.run(cmd).returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-baseline-s", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline field (0 = skip)")
    ap.add_argument("--reference-step-s", type=float, default=None,
                    help="oracle seconds per reference step (default: ~120 s over all steps)")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp16"], help="Q/K/V element type")
    ap.add_argument("--out-dtype", default="fp32", choices=["fp32", "same"],
                    help="O element type: fp32, or the Q/K/V type")
    ap.add_argument("--num-splits", type=int, default=1,
                    help="split the keys into this many ranges (split-KV forward + merge)")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the workload's head count (smaller profiling captures)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="groups of heads the end-to-end call pipelines its copies over")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads measured beside the headline one")
    ap.add_argument("--pass", dest="pass_", default="forward", choices=["forward", "backward"],
                    help="time the forward pass (default) or the backward pass")
    args = ap.parse_args()
    w = inputs.workload(args.workload)
    if args.heads is not None:
        import dataclasses
        w = dataclasses.replace(w, H=args.heads, name=f"{w.name}_heads{args.heads}")
    if args.reference_step_s is None:
        args.reference_step_s = max(1.0, min(10.0, 120.0 / max(1, args.steps)))

    world_env = os.environ.get("WORLD_SIZE")
    if world_env is None and args.gpus > 1:
        return relaunch_distributed(args.gpus)
    if world_env is not None and int(world_env) != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world_env}", file=sys.stderr)
        return 2
    if args.gpus < 1:
        print("bench.py: --gpus must be >= 1", file=sys.stderr)
        return 2

    if args.impl == "reference":
        return run_reference(args, w)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)

    import exact_attention_17_gb300 as fa2

    if args.pass_ == "backward":
        return run_backward(args, w, fa2, dev, dist, world, rank)

    # seeded inputs, generated on the host (same bits the oracle sees)
    in_dtype = torch.float16 if args.dtype == "fp16" else torch.bfloat16
    out_dtype = torch.float32 if args.out_dtype == "fp32" else in_dtype
    Qh, Kh, Vh = inputs.make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.seed, w.qk_dist, w.qk_std, w.v_dist,
                                 dtype=in_dtype)
    Q, K, V = Qh.to(dev), Kh.to(dev), Vh.to(dev)
    O = torch.empty(w.B, w.H, w.Nq, w.d, device=dev, dtype=out_dtype)
    L = torch.empty(w.B, w.H, w.Nq, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = None
    if forward_l2_note(w)[0]:
        flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)

    workspace = None
    if args.num_splits > 1:
        need = fa2.fa2_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.d, args.num_splits)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)

    def step(s):
        fa2.forward(Q, K, V, causal=w.causal, scale=w.scale, out=O, lse=L, stream=s,
                    num_splits=args.num_splits, workspace=workspace, out_dtype=out_dtype)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(stream)
    torch.cuda.synchronize(dev)
    if fa2.fa2_device_status(None, reset=True) != fa2.FA2_OK:
        raise SystemExit("device status error during warm-up")

    # timed region: K steps, per-launch events on the launching stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clocks:
        with torch.cuda.stream(stream):
            t_begin.record(stream)
            for i in range(args.steps):
                if flush is not None:
                    flush.zero_()
                starts[i].record(stream)
                step(stream)
                ends[i].record(stream)
            t_end.record(stream)
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    status = fa2.fa2_device_status(None, reset=True)
    if status != fa2.FA2_OK:
        raise SystemExit(f"device status error in the timed region: {status}")
    launch_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    kernel_ms = sum(launch_ms)
    total_ms = t_begin.elapsed_time(t_end)
    timed_ms = kernel_ms if flush is not None else total_ms
    job_ms = job_time_ms(timed_ms, dist, dev)

    # End to end through the public call with host buffers: pinned host
    # inputs -> device -> forward -> host result.  With bf16 inputs, fp32 O
    # and no split this is fa2_forward_host, which overlaps the copies of one
    # group of heads with the computation of another; otherwise the copies
    # and the forward run one after another on the stream.
    Qp, Kp, Vp = Qh.pin_memory(), Kh.pin_memory(), Vh.pin_memory()
    Op = torch.empty(O.shape, dtype=out_dtype).pin_memory()
    Lp = torch.empty(L.shape, dtype=torch.float32).pin_memory()
    pipelined = args.dtype == "bf16" and args.out_dtype == "fp32" and args.num_splits == 1
    e2e_kind = (f"fa2_forward_host, {args.e2e_chunks} head groups pipelined over copy/compute streams"
                if pipelined else "copies and forward in order on one stream")

    def e2e_step():
        if pipelined:
            fa2.forward_host(Qp, Kp, Vp, causal=w.causal, scale=w.scale, out=Op, lse=Lp,
                             device_buffers=(Q, K, V, O, L), chunks=args.e2e_chunks, stream=stream)
            return
        Q.copy_(Qp, non_blocking=True)
        K.copy_(Kp, non_blocking=True)
        V.copy_(Vp, non_blocking=True)
        fa2.forward(Q, K, V, causal=w.causal, scale=w.scale, out=O, lse=L, stream=stream,
                    num_splits=args.num_splits, workspace=workspace, out_dtype=out_dtype)
        Op.copy_(O, non_blocking=True)
        Lp.copy_(L, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    e2e_ms = job_time_ms(e0.elapsed_time(e1), dist, dev)
    h2d = (Qp.numel() + Kp.numel() + Vp.numel()) * 2
    d2h = Op.numel() * Op.element_size() + Lp.numel() * 4

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    mean_launch_ms = statistics.mean(launch_ms)
    achieved = w.flops / (mean_launch_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    value = job_tflops(w.flops, args.steps, world, job_ms)
    # Which roof bounds the kernel: tensor throughput when the workload's
    # FLOPs per algorithmic byte are above the machine balance, else HBM.
    algo_bytes = algorithmic_bytes(w, 2 if args.out_dtype == "same" else 4)
    balance = peak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    hbm_bound = w.flops / algo_bytes < balance
    traffic = recorded_traffic(w.name, fwd_kernel_sources(w.d, args.dtype == "fp16"))

    cpu = None
    if args.cpu_baseline_s > 0:
        tf, cores, rows, el = oracle_sample_rate(w, Qh, Kh, Vh, args.cpu_baseline_s)
        cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{rows} uniformly drawn query rows of {w.name} in {el:.1f} s "
                         f"(fp64 three-pass oracle, FLOPs = 4*|J_i|*d per row)"}

    clk = clocks.summary()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(job_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": args.dtype,
        "data": "synthetic",
        "config": forward_config(w, args),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "roofline": roofline_entry(hbm_bound, achieved, peak, peak_src, peaks, traffic, w.flops,
                                   algo_bytes, mean_launch_ms),
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_tflops(w.flops, args.e2e_steps, world, e2e_ms), 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms / args.e2e_steps, 4), "how": e2e_kind},
        "gpu_launches": args.steps * (2 if args.num_splits > 1 else 1),
        "clocks": clk,
    }
    if not args.no_workloads and args.heads is None:
        line["workloads"] = other_workloads(fa2, dev, w.name, peaks, peak_src)
        if w.d in (64, 128) and args.dtype == "bf16":
            line["backward"] = backward_entry(fa2, dev, w, peaks, peak_src)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0



# Measured beside the headline workload, each with its own roof.  The
# 4096-length causal case and the cross-length case are two of the five
# workloads; the non-causal 16384-length case is the same shape as the
# headline without the mask; the 1000-length case runs split-KV with the
# library's recommended split count; the one-tile case reports the host cost
# of a call next to its device time.
OTHER_WORKLOADS = ["b4_h16_n4096_d128_causal", "b16_h32_nq128_nk8192_d128", "b1_h32_n16384_d128",
                   "b2_h8_n1000_d64", "b1_h1_n128_d64"]


def measure_launches(fa2, dev, w, steps=10, warmup=3, num_splits=1):
    """Mean CUDA-event time of one forward call of workload w on its own
    stream (inputs resident; L2 flushed between launches when the inputs
    would fit in it)."""
    Qh, Kh, Vh = inputs.workload_inputs(w)
    Q, K, V = Qh.to(dev), Kh.to(dev), Vh.to(dev)
    del Qh, Kh, Vh
    O = torch.empty(w.B, w.H, w.Nq, w.d, device=dev)
    L = torch.empty(w.B, w.H, w.Nq, device=dev)
    stream = torch.cuda.Stream(device=dev)
    in_bytes = (Q.numel() + K.numel() + V.numel()) * 2
    flush = None
    if in_bytes <= 2 * 129 * 1024 * 1024:
        flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)
    workspace = None
    if num_splits > 1:
        need = fa2.fa2_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.d, num_splits)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)

    def call():
        fa2.forward(Q, K, V, causal=w.causal, scale=w.scale, out=O, lse=L, stream=stream,
                    num_splits=num_splits, workspace=workspace)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
        torch.cuda.synchronize(dev)
        ms = []
        for _ in range(steps):
            if flush is not None:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
    if fa2.fa2_device_status(None, reset=True) != fa2.FA2_OK:
        raise SystemExit(f"device status error while timing {w.name}")
    note = ("L2 flushed between launches (256 MiB write, outside the events)" if flush is not None
            else f"inputs {in_bytes / 2**20:.0f} MiB > 129 MiB L2, no flush")
    extra = {}
    if w.B * w.H * w.Nq <= 128:
        # host cost of one call: back-to-back calls without synchronisation
        n = 200
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            t0 = time.perf_counter()
            for _ in range(n):
                call()
            t1 = time.perf_counter()
            b.record(stream)
            b.synchronize()
        args = (Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), L.data_ptr(), w.B, w.H, w.Nq,
                w.Nk, w.d, int(w.causal), w.scale, stream.cuda_stream)
        t2 = time.perf_counter()
        for _ in range(n):
            fa2.fa2_forward(*args)
        t3 = time.perf_counter()
        torch.cuda.synchronize(dev)
        extra = {"host_us_per_call_python": round(1e6 * (t1 - t0) / n, 2),
                 "host_us_per_call_c_abi": round(1e6 * (t3 - t2) / n, 2),
                 "device_us_per_call_back_to_back": round(1000 * a.elapsed_time(b) / n, 2)}
    del Q, K, V, O, L, flush, workspace
    torch.cuda.empty_cache()
    return statistics.mean(ms), note, extra


def backward_entry(fa2, dev, w, peaks, peak_src, steps=5, warmup=3):
    """The backward pass of the headline workload (pre-pass and tensor-core
    kernel, one call per step) measured beside the forward: mean CUDA-event
    time of a call, TFLOP/s at 2.5x the forward's FLOPs, and its roofline."""
    Qh, Kh, Vh = inputs.workload_inputs(w)
    Gh = inputs.draw_bf16((w.B, w.H, w.Nq, w.d), w.seed, 3)
    Q, K, V, G = (t.to(dev) for t in (Qh, Kh, Vh, Gh))
    del Qh, Kh, Vh, Gh
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, device=dev) if backward_l2_note(w)[0] else None
    with torch.cuda.stream(stream):
        O, L = fa2.forward(Q, K, V, causal=w.causal, scale=w.scale, stream=stream)
        dQ = torch.empty(w.B, w.H, w.Nq, w.d, device=dev)
        dK = torch.empty(w.B, w.H, w.Nk, w.d, device=dev)
        dV = torch.empty(w.B, w.H, w.Nk, w.d, device=dev)
        ws = torch.empty(max(fa2.fa2_backward_workspace_bytes(w.B, w.H, w.Nq), 1), dtype=torch.uint8,
                         device=dev)

        def call():
            fa2.backward(Q, K, V, O, L, G, causal=w.causal, scale=w.scale, dq=dQ, dk=dK, dv=dV,
                         workspace=ws, stream=stream)

        for _ in range(warmup):
            call()
        torch.cuda.synchronize(dev)
        ms = []
        for _ in range(steps):
            if flush is not None:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
    if fa2.fa2_device_status(None, reset=True) != fa2.FA2_OK:
        raise SystemExit("device status error while timing the backward pass")
    mean_ms = statistics.mean(ms)
    flops = 2.5 * w.flops
    tf = flops / (mean_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    algo = algorithmic_bytes_backward(w)
    hbm_bound = flops / algo < peak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    del Q, K, V, G, O, L, dQ, dK, dV, ws, flush
    torch.cuda.empty_cache()
    return {"metric": METRIC_BWD, "config": {"workload": w.name, "l2": backward_l2_note(w)[1]},
            "mean_call_ms": round(mean_ms, 4), "tflops": round(tf, 2), "pct_of_peak": round(100 * tf / peak, 2),
            "kernels_per_call": 2,
            "roofline": roofline_entry(hbm_bound, tf, peak, peak_src, peaks,
                                       recorded_traffic(w.name + ":backward", BWD_KERNEL_SOURCES), flops, algo,
                                       mean_ms, kernel="fa2dev::fa2_bwd_tc_kernel")}


def other_workloads(fa2, dev, headline, peaks, peak_src):
    out = {}
    peak = float(peaks["bf16_tflops"])
    balance = peak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    for name in OTHER_WORKLOADS:
        if name == headline:
            continue
        w = inputs.workload(name)
        splits = 1
        if name == "b2_h8_n1000_d64":
            splits = fa2.fa2_splitkv_recommended_splits(w.B, w.H, w.Nq, w.Nk, 0)
        ms, note, extra = measure_launches(fa2, dev, w, num_splits=splits)
        tf = w.flops / (ms * 1e-3) / 1e12
        algo = algorithmic_bytes(w)
        hbm_bound = w.flops / algo < balance
        entry = {"config": {"B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
                            "num_splits": splits, "l2": note},
                 "mean_launch_ms": round(ms, 4), "tflops": round(tf, 2),
                 "pct_of_peak": round(100 * tf / peak, 2),
                 "kernels_per_call": 2 if splits > 1 else 1,
                 "roofline": roofline_entry(hbm_bound, tf, peak, peak_src, peaks,
                                            recorded_traffic(name, fwd_kernel_sources(w.d)), w.flops,
                                            algo, ms)}
        entry.update(extra)
        out[name] = entry
    return out


def run_backward(args, w, fa2, dev, dist, world, rank):
    """One step = one backward pass (pre-pass + tensor-core kernel) of the
    workload, with O and LSE from one forward pass before the timed region."""
    if args.num_splits != 1 or args.out_dtype != "fp32":
        raise SystemExit("--pass backward takes fp32 O and no split")
    in_dtype = torch.float16 if args.dtype == "fp16" else torch.bfloat16
    Qh, Kh, Vh = inputs.make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.seed, w.qk_dist, w.qk_std, w.v_dist,
                                 dtype=in_dtype)
    Gh = inputs.draw_bf16((w.B, w.H, w.Nq, w.d), w.seed, 3, dtype=in_dtype)
    Q, K, V, G = (t.to(dev) for t in (Qh, Kh, Vh, Gh))
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        O, L = fa2.forward(Q, K, V, causal=w.causal, scale=w.scale, stream=stream)
        dQ = torch.empty(w.B, w.H, w.Nq, w.d, device=dev)
        dK = torch.empty(w.B, w.H, w.Nk, w.d, device=dev)
        dV = torch.empty(w.B, w.H, w.Nk, w.d, device=dev)
        ws = torch.empty(max(fa2.fa2_backward_workspace_bytes(w.B, w.H, w.Nq), 1), dtype=torch.uint8,
                         device=dev)
    flush = None
    if backward_l2_note(w)[0]:
        flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)

    def step(s):
        fa2.backward(Q, K, V, O, L, G, causal=w.causal, scale=w.scale, dq=dQ, dk=dK, dv=dV,
                     workspace=ws, stream=s)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(stream)
    torch.cuda.synchronize(dev)
    if fa2.fa2_device_status(None, reset=True) != fa2.FA2_OK:
        raise SystemExit("device status error during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clocks:
        with torch.cuda.stream(stream):
            t_begin.record(stream)
            for i in range(args.steps):
                if flush is not None:
                    flush.zero_()
                starts[i].record(stream)
                step(stream)
                ends[i].record(stream)
            t_end.record(stream)
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    if fa2.fa2_device_status(None, reset=True) != fa2.FA2_OK:
        raise SystemExit("device status error in the timed region")
    launch_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    timed_ms = sum(launch_ms) if flush is not None else t_begin.elapsed_time(t_end)
    job_ms = job_time_ms(timed_ms, dist, dev)
    flops = 2.5 * w.flops

    # end to end through the public calls: pinned inputs in, gradients out, every step
    pins = [t.pin_memory() for t in (Qh, Kh, Vh, Gh)]
    Oh, Lh = O.cpu().pin_memory(), L.cpu().pin_memory()
    outs = [torch.empty(t.shape, dtype=torch.float32).pin_memory() for t in (dQ, dK, dV)]

    def e2e_step():
        for dst, src in zip((Q, K, V, G, O, L), pins + [Oh, Lh]):
            dst.copy_(src, non_blocking=True)
        step(stream)
        for dst, src in zip(outs, (dQ, dK, dV)):
            dst.copy_(src, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    e2e_ms = job_time_ms(e0.elapsed_time(e1), dist, dev)
    h2d = sum(t.numel() * t.element_size() for t in pins + [Oh, Lh])
    d2h = sum(t.numel() * 4 for t in outs)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    mean_launch_ms = statistics.mean(launch_ms)
    achieved = flops / (mean_launch_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    algo = algorithmic_bytes_backward(w)
    hbm_bound = flops / algo < peak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    cpu = None
    if args.cpu_baseline_s > 0:
        tf, cores, n, el = oracle_backward_rate(w, Qh, Kh, Vh, Gh, args.cpu_baseline_s)
        cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"head 0 of {w.name} truncated to its leading {n} queries and keys in "
                         f"{el:.1f} s (fp64 oracle backward, FLOPs = 2.5 x the forward's)"}
    value = job_tflops(flops, args.steps, world, job_ms)
    line = {
        "metric": METRIC_BWD,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(job_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": args.dtype,
        "data": "synthetic",
        "config": backward_config(w, args),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "roofline": roofline_entry(hbm_bound, achieved, peak, peak_src, peaks,
                                   recorded_traffic(w.name + ":backward" + (":fp16" if args.dtype == "fp16" else ""),
                                                    BWD_KERNEL_SOURCES),
                                   flops, algo, mean_launch_ms, kernel="fa2dev::fa2_bwd_tc_kernel"),
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_tflops(flops, args.e2e_steps, world, e2e_ms), 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * 2,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
