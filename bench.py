#!/usr/bin/env python
"""Attention-forward benchmark on GB300.

One step = one fa_fwd call over the whole workload (every batch, head and
query tile): O = softmax(scale QK^T [+mask]) V and LSE.  Default workload:
B=8, H=16, Sq=Sk=2048, D=128, bf16, non-causal.  Metric: forward TFLOP/s
(4*B*H*Sq*Sk*D, halved when causal) and its fraction of the measured dense
bf16 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 it runs one rank per GPU under torch.distributed.run (started by
the caller, or by bench.py itself when --gpus N > 1 is given without a
WORLD_SIZE in the environment).  By default every rank processes its own full
workload (independent problems, no data-path collective: weak scaling); with
--split heads the B*H heads of ONE workload are dealt out to the ranks in
contiguous blocks, each rank writing only its heads' rows of O and LSE (strong
scaling).  Either way value = all ranks' FLOPs / the slowest rank's time.
`--impl reference` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd attention TFLOP/s & % of GB300 dense BF16 peak (causal FLOPs halved)"
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
_CSRC = "exact_attention_82_gb300/csrc/"
# the sources each path's kernels are built from (a recorded DRAM-traffic figure is
# valid only while they are unchanged)
KERNEL_SOURCES = {
    "fwd": [_CSRC + "fa_fwd_kernel.cu", _CSRC + "sm103_ptx.cuh", _CSRC + "fa_internal.h"],
    "bwd": [_CSRC + "fa_bwd.cu", _CSRC + "sm103_ptx.cuh", _CSRC + "fa_internal.h"],
    "splitkv": [_CSRC + "fa_splitkv.cu", _CSRC + "sm103_ptx.cuh", _CSRC + "fa_internal.h"],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=1, help="index into the workload table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target seconds of oracle work for the CPU baseline")
    ap.add_argument("--split", choices=["none", "heads"], default="none",
                    help="none: every rank runs the whole workload (weak scaling); heads: the "
                         "B*H heads of one workload are split across the ranks (strong scaling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


def source_group(path: str) -> str:
    """Which kernel sources serve a workload path ("fp8" and "fwd" share one kernel)."""
    return path if path in ("bwd", "splitkv") else "fwd"


def _strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (string and character
    literals are kept as they are), so that a comment edit leaves the key of
    the kernel's DRAM record unchanged while any code change alters it."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash(group: str = "fwd") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[group]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_strip_comments(f.read()).encode("utf-8"))
    return h.hexdigest()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return None, "fallback"


def traffic_per_launch(w):
    """DRAM bytes per launch (per step, both kernels, for the backward) from a
    committed ncu capture, if it still describes the current kernel sources;
    else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(w.name)
    if not entry or entry.get("kernel_sha256") != kernel_source_hash(source_group(w.path)):
        return None
    return entry.get("dram_bytes_per_launch")


# ----------------------------------------------------- rank aggregation
def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the slowest rank's step time); x itself at N=1."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Every rank processes its own full workload: all ranks' FLOPs / the slowest time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def rank_workload(w, world: int, rank: int, split: str):
    """The part of workload `w` this rank runs, and the heads it owns:
    (workload, start, count).  With split "heads" the rank runs heads
    [start, start + count) of the flattened B*H axis as a B = 1, H = count
    workload; otherwise the whole workload (start 0, count B*H)."""
    import dataclasses

    from exact_attention_82_gb300.shard import head_range

    if split != "heads":
        return w, 0, w.B * w.H
    start, count = head_range(w.B * w.H, world, rank)
    return dataclasses.replace(w, B=1, H=count), start, count


def spawn_command(argv, nproc: int, port: int):
    """The command that runs this script as `nproc` ranks on this node under
    torch.distributed.run (rendezvous on 127.0.0.1), with the same arguments."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={nproc}", "--master-addr=127.0.0.1", f"--master-port={port}",
            os.path.abspath(__file__), *argv]


def _free_port() -> int:
    import socket

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [ln.strip().split(",") for ln in self.out.read().splitlines() if ln.strip()]
        self.out.close()
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- our arm
def run_path(fa, w, q, k, v, o, lse, ws, stream):
    """One step of workload `w` through the library's public call for its path.
    For the backward, `ws` holds (forward O, forward LSE, dO, dQ, dK, dV, Delta)."""
    if w.path == "bwd":
        fo, flse, dout, dq, dk, dv, delta = ws
        fa.fa_bwd(q, k, v, fo, flse, dout, dq=dq, dk=dk, dv=dv, delta=delta, scale=w.scale,
                  causal=w.causal, stream=stream)
    elif w.path == "splitkv":
        fa.fa_fwd_splitkv(q, k, v, o=o, lse=lse, scale=w.scale, workspace=ws, stream=stream)
    elif w.path == "fp8":
        fa.fa_fwd_fp8(q, k, v, *ws, o=o, lse=lse, scale=w.scale, causal=w.causal, stream=stream)
    elif w.path == "blockmask":
        fa.fa_fwd_blockmask(q, k, v, ws, w.window[0], w.window[1], o=o, lse=lse, scale=w.scale,
                            pair_stride=w.dilation, stream=stream)
    elif w.window_left >= 0:
        fa.fa_fwd_window(q, k, v, w.window[0], w.window[1], o=o, lse=lse, scale=w.scale,
                         stream=stream)
    else:
        fa.fa_fwd(q, k, v, o=o, lse=lse, scale=w.scale, causal=w.causal, stream=stream)


def workload_inputs(index):
    """CPU inputs of workload `index`: (q, k, v, descales); descales is None except
    on the 8-bit path, whose q, k, v are e4m3 codes (uint8)."""
    from exact_attention_82_gb300.inputs import WORKLOADS, workload_qkv, workload_qkv_fp8

    if WORKLOADS[index].path == "fp8":
        (q, k, v), ds = workload_qkv_fp8(index)
        return q, k, v, ds
    q, k, v = workload_qkv(index)
    return q, k, v, None


def make_workspace(fa, w, q, k, v, dev, descales=None):
    """Per-path extra buffers (the descales on the 8-bit path), made once outside
    the timed region."""
    import torch

    if w.path == "fp8":
        return descales
    if w.path == "blockmask":  # the pattern: a fixed input, on the device before timing
        return w.block_mask.to(dev)
    if w.path == "splitkv":
        return torch.empty(fa.fa_fwd_splitkv_workspace_bytes(w.B, w.H, w.Sq, w.Sk, w.D),
                           dtype=torch.uint8, device=dev)
    if w.path == "bwd":
        from exact_attention_82_gb300.inputs import SEED_BASE, make_qkv

        fo, flse = fa.fa_fwd(q, k, v, scale=w.scale, causal=w.causal)
        dout = make_qkv(w.B, w.H, w.Sq, w.Sk, w.D, SEED_BASE + 999)[0].to(dev)
        return (fo, flse, dout, torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev))
    return None


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import exact_attention_82_gb300 as fa
    from exact_attention_82_gb300.inputs import WORKLOADS

    from exact_attention_82_gb300.shard import head_slice

    w_full = WORKLOADS[args.workload]
    # this rank's part: the whole workload, or (--split heads) its block of heads
    w, h0, nh = rank_workload(w_full, world, rank, args.split)
    if args.split == "heads" and w_full.path not in ("fwd", "fp8", "blockmask"):
        raise SystemExit("--split heads applies to the forward workloads")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    q, k, v, descales = workload_inputs(args.workload)
    if args.split == "heads":
        q, k, v = (head_slice(t, h0, nh).contiguous() for t in (q, k, v))
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty((w.B, w.H, w.Sq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    ws = make_workspace(fa, w, dq, dk, dv, dev, descales)

    def step():
        if nh > 0:  # a rank beyond the head count has nothing to do
            run_path(fa, w, dq, dk, dv, o, lse, ws, stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local_rank).start()
    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    st = fa.fa_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after warm-up: {fa.fa_strerror(st)}")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))           # evict the previous step's data from L2
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = sum(times) / len(times)
    ms = max_over_ranks(ms_local, world, dev)
    st = fa.fa_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status after timing: {fa.fa_strerror(st)}")

    strong = args.split == "heads"
    e2e = None if args.no_e2e else run_e2e(args, w, q, k, v, dev, world, descales,
                                           job_flops=w_full.flops if strong else None)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q, k, v, args.cpu_seconds, descales)
    if rank != 0:
        return None
    peaks, which = measured_peaks()
    peak = float(peaks["bf16_tflops"]) if peaks else FALLBACK_PEAK_TFLOPS
    tflops_launch = w.flops / (ms_local * 1e-3) / 1e12
    # strong: the ranks share one workload; weak: each runs a whole one
    value = (w_full.flops / (ms * 1e-3) / 1e12) if strong else whole_job_tflops(w.flops, world, ms)
    if strong:
        parallelism = (f"B*H = {w_full.B * w_full.H} heads of one workload split across {world} "
                       f"GPU(s) in contiguous blocks (rank 0: heads [{h0}, {h0 + nh})), each "
                       f"writing only its heads' O and LSE; no data-path collective")
    else:
        parallelism = f"independent workload per GPU x{world}"
    traffic = traffic_per_launch(w)
    if traffic is not None and strong:  # recorded for the whole workload; this rank runs nh heads
        traffic = traffic * nh / (w_full.B * w_full.H)
    if w.path == "splitkv":
        # decode reads each key and value once: bound by HBM bandwidth
        hbm_peak = float(peaks["hbm_gbs"]) if peaks else FALLBACK_HBM_GBS
        gbs = w.hbm_bytes / (ms_local * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(gbs / hbm_peak, 4),
                    "peak_source": f"{which}: hbm_gbs (copy bandwidth)" if peaks
                    else "fallback: 6.8 TB/s", "traffic": traffic}
    elif w.path == "fp8":
        # e4m3 contractions: the measured bf16 peak times the nominal 8-bit : 16-bit
        # dense ratio (4.5 : 2.25 PFLOP/s)
        peak8 = 2.0 * peak
        roofline = {"bound": "tensor", "achieved": round(tflops_launch, 2), "peak": peak8,
                    "unit": "TFLOP/s", "frac": round(tflops_launch / peak8, 4),
                    "peak_source": (f"{which}: bf16_tflops (burst, cuBLAS bf16 GEMM)" if peaks
                                    else "fallback: 1.9 PFLOP/s bf16")
                    + " x 2, the nominal fp8/bf16 dense ratio", "traffic": traffic}
    else:
        roofline = {"bound": "tensor", "achieved": round(tflops_launch, 2), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(tflops_launch / peak, 4),
                    "peak_source": f"{which}: bf16_tflops (burst, cuBLAS bf16 GEMM)"
                    if peaks else "fallback: 1.9 PFLOP/s bf16", "traffic": traffic}
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "strong" if strong else "weak", "vs_baseline": None,
        "dtype": "e4m3" if w.path == "fp8" else "bf16", "data": "synthetic",
        "config": {"workload": w_full.name, "desc": w_full.describe(), "B": w_full.B,
                   "H": w_full.H, "Sq": w.Sq, "Sk": w.Sk, "D": w.D, "causal": w.causal,
                   "window": list(w.window), "parallelism": parallelism,
                   "l2": "flushed before every step (256 MiB write outside the timed events)",
                   "pct_of_bf16_peak": round(100.0 * tflops_launch / peak, 2),
                   "ms_median": round(statistics.median(times), 5), "ms_min": round(min(times), 5),
                   "hbm_gbs_algorithmic": round(w.hbm_bytes / (ms_local * 1e-3) / 1e9, 1)
                   if w.path != "bwd" else None,
                   "wall_s_timed_region": round(t_wall, 4)},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (2 if w.path in ("splitkv", "bwd") else 1) * (nh > 0),
        "clocks": clk,
        "impl": "ours",
    }


def _pipelined_e2e(args, host_in, host_out, launch, dev, world, flops, job_flops=None):
    """End-to-end steps through the public call: step i copies `host_in` (pinned)
    to the device, calls `launch(dev_in, dev_out, stream)` and reads `dev_out`
    back into `host_out` (pinned).  Steps are pipelined as a serving loop runs
    them, with two sets of device buffers: the input copy of step i+1 (its own
    stream) overlaps step i's call, and step i's read-back (a third stream)
    overlaps step i+1.  Every step's copies lie inside the timed region, which
    starts before the first input copy and ends after the last read-back."""
    import torch
    import torch.distributed as dist

    dev_in = [[torch.empty_like(h, device=dev) for h in host_in] for _ in range(2)]
    dev_out = [[torch.empty_like(h, device=dev) for h in host_out] for _ in range(2)]
    compute = torch.cuda.current_stream(dev)
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(steps):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(compute)
        h2d.wait_stream(compute)
        ready, used, read = [None, None], [None, None], [None, None]

        def load(i):
            b = i & 1
            if used[b] is not None:  # step i-2's call is done with these inputs
                h2d.wait_event(used[b])
            with torch.cuda.stream(h2d):
                for d, h in zip(dev_in[b], host_in):
                    d.copy_(h, non_blocking=True)
            ready[b] = torch.cuda.Event()
            ready[b].record(h2d)

        load(0)
        for i in range(steps):
            b = i & 1
            if i + 1 < steps:
                load(i + 1)
            compute.wait_event(ready[b])
            if read[b] is not None:  # step i-2's outputs have been read back
                compute.wait_event(read[b])
            launch(dev_in[b], dev_out[b], compute)
            used[b] = torch.cuda.Event()
            used[b].record(compute)
            d2h.wait_event(used[b])
            with torch.cuda.stream(d2h):
                for h, d in zip(host_out, dev_out[b]):
                    h.copy_(d, non_blocking=True)
            read[b] = torch.cuda.Event()
            read[b].record(d2h)
        compute.wait_stream(h2d)
        compute.wait_stream(d2h)
        end.record(compute)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    run(3)
    if world > 1:
        dist.barrier()
    steps = max(3, min(args.steps, 50))
    ms = max_over_ranks(run(steps) / steps, world, dev)
    value = job_flops / (ms * 1e-3) / 1e12 if job_flops else whole_job_tflops(flops, world, ms)
    return {"value": round(value, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": steps,
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in),
            "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out),
            "overlap": "step i+1's input copy and step i's read-back run beside step i's call "
                       "(three streams, two device buffer sets)"}


def run_e2e(args, w, q, k, v, dev, world, descales=None, job_flops=None):
    """Same metric through the public call with host buffers: every step copies
    Q, K, V from pinned host memory, runs the attention call and reads O and LSE
    back (pipelined across steps, see _pipelined_e2e).  With `job_flops` (a head
    split) the ranks share one workload of that many FLOPs."""
    import torch

    import exact_attention_82_gb300 as fa

    if w.path == "bwd":
        return run_e2e_bwd(args, w, q, k, v, dev, world)
    host_in = [t.pin_memory() for t in (q, k, v)]
    host_out = [torch.empty((w.B, w.H, w.Sq, w.D), dtype=torch.bfloat16).pin_memory(),
                torch.empty((w.B, w.H, w.Sq), dtype=torch.float32).pin_memory()]
    ws = make_workspace(fa, w, *host_in, dev, descales)  # (Q, K, V only matter on the backward path)

    def launch(din, dout, stream):
        if w.B * w.H > 0:
            run_path(fa, w, *din, *dout, ws, stream)

    return _pipelined_e2e(args, host_in, host_out, launch, dev, world, w.flops, job_flops)


def run_e2e_bwd(args, w, q, k, v, dev, world):
    """The backward end to end: every step copies Q, K, V, the forward's O and LSE
    and dO from pinned host memory, runs fa_bwd and reads dQ, dK, dV back
    (pipelined across steps, see _pipelined_e2e)."""
    import torch

    import exact_attention_82_gb300 as fa

    dq_, dk_, dv_ = (t.to(dev) for t in (q, k, v))
    fo, flse, dout = make_workspace(fa, w, dq_, dk_, dv_, dev)[:3]
    host_in = [t.pin_memory() for t in (q, k, v)] + [t.cpu().pin_memory() for t in (fo, flse, dout)]
    host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in (dq_, dk_, dv_)]
    delta = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)
    del dq_, dk_, dv_, fo, flse, dout

    def launch(din, dout, stream):
        fa.fa_bwd(*din, dq=dout[0], dk=dout[1], dv=dout[2], delta=delta, scale=w.scale,
                  causal=w.causal, stream=stream)

    return _pipelined_e2e(args, host_in, host_out, launch, dev, world, w.flops)


# ------------------------------------------------------- CPU (oracle) legs
def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_sample(w, qb, kb, vb, heads, descales=None, gb=None):
    """Oracle over the first `heads` (b,h) pairs, all rows; returns (seconds, flops).
    qb, kb, vb: bf16 bit patterns, or e4m3 codes when `descales` is given; for the
    backward `gb` holds dO's bf16 bits and the oracle's backward is timed."""
    import oracle

    BH = w.B * w.H
    qs = qb.reshape(BH, w.Sq, w.D)[:heads][None]
    ks = kb.reshape(BH, w.Sk, w.D)[:heads][None]
    vs = vb.reshape(BH, w.Sk, w.D)[:heads][None]
    t0 = time.perf_counter()
    if w.path == "bwd":
        gs = gb.reshape(BH, w.Sq, w.D)[:heads][None]
        oracle.attn_bwd(qs, ks, vs, gs, w.scale, w.causal, nthreads=_host_cores())
    elif descales is not None:
        oracle.attn_fwd_fp8(qs, ks, vs, *descales, w.scale, w.causal, nthreads=_host_cores())
    else:
        oracle.attn_fwd(qs, ks, vs, w.scale, w.causal, w.window, nthreads=_host_cores())
    dt = time.perf_counter() - t0
    return dt, w.flops / BH * heads


def _dout_bits(w):
    """dO of the backward workloads (the draw bench.py's own leg uses), as bf16 bits."""
    from exact_attention_82_gb300.inputs import SEED_BASE, bf16_bits, make_qkv

    return bf16_bits(make_qkv(w.B, w.H, w.Sq, w.Sk, w.D, SEED_BASE + 999)[0])


def _oracle_inputs(q, k, v, descales):
    from exact_attention_82_gb300.inputs import bf16_bits, u8_codes

    conv = u8_codes if descales is not None else bf16_bits
    return conv(q), conv(k), conv(v)


def cpu_baseline(w, q, k, v, target_s, descales=None):
    """The oracle as it stands, on the host cores, over a bounded sample of the
    same workload: whole heads, grown until about `target_s` seconds (block-mask
    path: whole query blocks from the middle of as many heads as there are cores)."""
    if w.path == "blockmask":
        from exact_attention_82_gb300.inputs import BLOCK

        cores = _host_cores()
        BH = w.B * w.H
        rows = min(w.Sq, 8 * BLOCK)  # (the oracle holds rows x Sk fp64 arrays per head)
        r0 = max(0, (w.Sq // 2 - rows // 2) // BLOCK * BLOCK)
        nh = min(BH, cores)
        dt, fl = _RowSampler(w, q, k, v, None, nh).run(r0, rows)
        if dt < target_s / 4 and nh < BH:
            nh = min(BH, max(nh + 1, int(nh * target_s / max(dt, 1e-3) * 0.8)))
            dt, fl = _RowSampler(w, q, k, v, None, nh).run(r0, rows)
        return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
                "kind": "oracle", "seconds": round(dt, 2),
                "sample": f"query rows {r0}..{min(w.Sq, r0 + rows) - 1} of {nh} of {BH} (batch,head) pairs of "
                          f"{w.name}, with every key; fp64 numpy block-mask oracle forward with S and P "
                          f"materialised (numpy's matmul threads)"}
    qb, kb, vb = _oracle_inputs(q, k, v, descales)
    gb = _dout_bits(w) if w.path == "bwd" else None
    cores = _host_cores()
    BH = w.B * w.H
    heads = min(BH, cores)
    dt, fl = _oracle_sample(w, qb, kb, vb, heads, descales, gb)
    if dt < target_s / 4 and heads < BH:
        heads = min(BH, max(heads + 1, int(heads * target_s / max(dt, 1e-3) * 0.8)))
        dt, fl = _oracle_sample(w, qb, kb, vb, heads, descales, gb)
    what = "backward (dQ, dK, dV)" if w.path == "bwd" else "forward"
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{heads} of {BH} (batch,head) pairs of {w.name}, every query row; "
                      f"fp64 C oracle {what} with S and P materialised"}


REFERENCE_BUDGET_S = 120.0  # host time of a whole --impl reference run (warm-up + timed steps)


class _RowSampler:
    """Samples of a workload for the reference arm: `rows` consecutive query rows
    of each of the first `nh` heads (one oracle call, which runs a thread per
    head), evaluated on exactly the keys those rows may see (the key range and
    band are re-expressed in the slice's own indices), so a sample's work is
    exactly that of those rows in the full workload."""

    def __init__(self, w, q, k, v, descales, nh):
        import oracle

        self.w, self.nh = w, nh
        BH = w.B * w.H

        def heads(t, d=None):
            t = t.reshape(BH, -1, w.D)[:nh].contiguous()
            if d is not None:
                return oracle.e4m3_to_f64(t.numpy()) * float(np.float32(d))
            return oracle.bf16_bits_to_f64(t.view(torch_int16()).numpy().view(np.uint16))

        ds = descales if descales is not None else (None, None, None)
        self.q, self.k, self.v = (heads(t, d) for t, d in zip((q, k, v), ds))
        self.mask = w.block_mask.numpy() if w.path == "blockmask" else None
        self.g = None
        if w.path == "bwd":
            from exact_attention_82_gb300.inputs import SEED_BASE, make_qkv

            self.g = heads(make_qkv(w.B, w.H, w.Sq, w.Sk, w.D, SEED_BASE + 999)[0])

    def run(self, r0, rows):
        """Time the oracle on rows r0 .. r0 + rows - 1 of the sampled heads; (seconds, flops)."""
        import oracle

        w = self.w
        if w.path == "blockmask":
            return self._run_blockmask(r0, rows)
        wl, wr = w.window
        r1 = min(w.Sq, r0 + rows)
        k0 = max(0, r0 - wl) if wl >= 0 else 0
        k1 = min(w.Sk, r1 + wr) if wr >= 0 else w.Sk
        shift = r0 - k0
        win = (wl - shift if wl >= 0 else -1, wr + shift if wr >= 0 else -1)
        i = np.arange(r0, r1)
        lo = np.maximum(0, i - wl) if wl >= 0 else np.zeros_like(i)
        hi = np.minimum(w.Sk - 1, i + wr) if wr >= 0 else np.full_like(i, w.Sk - 1)
        pairs = float(np.maximum(hi - lo + 1, 0).sum()) * self.nh
        flops = 4.0 * w.D * pairs * (2.5 if w.path == "bwd" else 1.0)
        qa = self.q[None, :, r0:r1]
        ka, va = self.k[None, :, k0:k1], self.v[None, :, k0:k1]
        t0 = time.perf_counter()
        if w.path == "bwd":
            oracle.attn_bwd(qa, ka, va, self.g[None, :, r0:r1], w.scale, False, win, nthreads=_host_cores())
        else:
            oracle.attn_fwd(qa, ka, va, w.scale, False, win, nthreads=_host_cores())
        return time.perf_counter() - t0, flops


    def _run_blockmask(self, r0, rows):
        """Whole query blocks covering rows r0 .. r0 + rows - 1, against every key:
        the block-mask oracle on those rows, with the causal bound shifted to the
        slice's row indices."""
        import oracle
        from exact_attention_82_gb300.inputs import BLOCK

        w = self.w
        a0 = r0 // BLOCK
        a1 = -(-min(w.Sq, r0 + rows) // BLOCK)
        rb0, rb1 = a0 * BLOCK, min(w.Sq, a1 * BLOCK)
        kept = self.mask[0] != 0
        i = np.arange(rb0, rb1)[:, None]
        j = np.arange(w.Sk)[None, :]
        allowed = kept[i // BLOCK, j // BLOCK]
        if w.causal:
            allowed &= j <= i
        flops = 4.0 * w.D * float(allowed.sum()) * self.nh
        win = (-1, rb0) if w.causal else (-1, -1)
        qa = self.q[None, :, rb0:rb1]
        t0 = time.perf_counter()
        oracle.attn_fwd_blockmask(qa, self.k[None], self.v[None], w.scale, self.mask[:, a0:a1],
                                  window=win, block=(BLOCK, BLOCK))
        return time.perf_counter() - t0, flops


def torch_int16():
    import torch

    return torch.int16


def run_reference(args):
    """Reference arm: the fp64 oracle on the host cores, each step a bounded
    sample (consecutive query rows of as many heads as there are cores, rows
    advancing from step to step) of the same workload, sized so that the whole
    run takes about REFERENCE_BUDGET_S seconds whatever --steps and --warmup are."""
    from exact_attention_82_gb300.inputs import WORKLOADS

    w = WORKLOADS[args.workload]
    q, k, v, descales = workload_inputs(args.workload)
    cores = _host_cores()
    BH = w.B * w.H
    nh = min(BH, cores)
    sampler = _RowSampler(w, q, k, v, descales, nh)
    per_step = max(0.002, REFERENCE_BUDGET_S / (args.steps + args.warmup))
    # calibrate the rows per step on a middle block
    rows = min(w.Sq, 32)
    dt, _ = sampler.run(max(0, w.Sq // 2 - rows // 2), rows)
    rows = max(1, min(w.Sq, int(rows * per_step / max(dt, 1e-6))))
    pos = [0]

    def step(i):
        r0 = (pos[0] * rows) % max(1, w.Sq - rows + 1) if rows < w.Sq else 0
        pos[0] += 1
        return sampler.run(r0, rows)

    for i in range(args.warmup):
        step(i)
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = step(args.warmup + i)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    what = "backward (dQ, dK, dV)" if w.path == "bwd" else "forward"
    sample = (f"{rows} consecutive query rows of each of {nh} (batch, head) pairs of {w.name} per "
              f"step (of {w.Sq} rows x {BH} heads), rows advancing per step, with exactly the "
              f"keys they may see; fp64 C oracle {what}, a thread per head, S and P "
              f"materialised; {REFERENCE_BUDGET_S:.0f} s budget for the whole run")
    if w.path == "blockmask":
        sample = (f"whole 128-row query blocks covering {rows} rows of each of {nh} (batch, head) pairs "
                  f"of {w.name} per step, rows advancing per step, with every key; fp64 numpy "
                  f"block-mask oracle forward, S and P materialised; {REFERENCE_BUDGET_S:.0f} s budget "
                  f"for the whole run")
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "desc": w.describe()},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # asked for N GPUs without a launcher: start the N ranks here
        return subprocess.call(spawn_command(sys.argv[1:] if argv is None else list(argv),
                                             args.gpus, _free_port()))
    if world != args.gpus:
        print(f"error: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        return 2
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    try:
        res = run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
