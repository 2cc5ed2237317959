#!/usr/bin/env python3
"""Benchmark of the GB300 draft-head path (prints one JSON line on rank 0).

A step is one pass of the draft head over one batch: dh_draft_head (projection, vocabulary-wide
low-rank scores, exact top-K, gathered full-rank logits and their softmax), on the workload's
synthetic inputs already resident in HBM.  The headline workload is ``batch1`` (B=1, d=5120,
vocab=151936, r=128, K=64, bf16), timed for exactly ``--steps`` steps.  The same line carries a
``workloads`` object with the other workloads (moderate, high, the draft level, tree acceptance),
each timed for at least 100 ms.

* value: rows per second over the whole job (sum over ranks / slowest rank's time); steps run as
  CUDA-graph replays; input sets rotate over enough independent copies that the bytes touched
  between two uses of one copy exceed twice the L2 size.
* path_roofline: the path's ideal time per the hot-path measurement rule (per stage, the larger of
  its HBM bytes over the measured copy bandwidth and its FLOPs over the peak of the unit that runs
  it; stage 2 charged at the distinct W rows the step gathers) over the measured time.
* roofline: one named kernel per workload, its algorithmic bytes (or FLOPs) per launch over its
  CUDA-event duration (a separate pass with per-kernel events on the launch stream).
* e2e: the same metric through the public API with each step's input h copied from pinned host
  memory and the step's results copied back, all in stream order (one graph replay per step); the
  per-step synchronised form and the eager Python-level form are reported beside it.
* cpu_baseline: the CPU oracle timed on host cores on a bounded sample of the same workload.
* ``--impl reference``: the CPU oracle as the reference arm (rank 0 only).
* ``--gpus N`` without a launcher: spawns N ranks (one per GPU) on this node; replicas need no
  collective in the data path, only the barrier and the max over ranks of the timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import socket
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_draft_dh_gb300 import inputs  # noqa: E402

METRIC = "draft-head rows/sec and µs per call (low-rank top-K + rescore); % of HBM roofline"
TREE_METRIC = "tree-acceptance requests/sec and µs per call (per-node argmax + tree walk); % of HBM roofline"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp32 FMA peak of the CUDA cores: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz
FP32_CORE_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
DEFAULT_STEPS = {"batch1": 20000, "moderate": 5000, "high": 500, "tree": 200, "level": 10000, "verify": 2000}
DEFAULT_WARMUP = {"batch1": 200, "moderate": 50, "high": 10, "tree": 5, "level": 100, "verify": 10}
EXTRA_WORKLOADS = ["moderate", "high", "level", "tree", "verify"]
MIN_TIMED_S = 0.1  # every added workload's timed region
EXPAND_W = {"level": 4}  # children per frontier node in the draft-level workload
# the draft level then sizes the next level: requests (the frontier nodes split evenly), width limit,
# threshold in accepted tokens per microsecond of the synthetic latency table
SIZE_LEVEL = {"level": {"requests": 2, "wmax": 8, "theta": 0.002}}
# the kernel each workload's `roofline` reports (the one that moves the step's bytes)
ROOFLINE_KERNEL = {"batch1": "scores_lsu", "moderate": "rescore_ring", "high": "rescore_ring",
                   "level": "lowrank_mma", "tree": "tree_argmax"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="batch1",
                    choices=["batch1", "moderate", "high", "tree", "level", "verify"])
    ap.add_argument("--only", action="store_true", help="time the named workload alone (no `workloads`)")
    ap.add_argument("--api", default="head", choices=["head", "split"],
                    help="head: dh_draft_head (both stages in one call); split: dh_lowrank_topk + "
                         "dh_exact_rescore")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--dry-run", action="store_true",
                    help="no GPU: the ranks meet over gloo, time a host loop and report (tests the "
                         "multi-rank plumbing)")
    ap.add_argument("--profile-run", action="store_true",
                    help="for profilers: one input copy, eager launches of warmup+steps steps, "
                         "no graphs, e2e, CPU baseline or clock sampling; prints a short line")
    a = ap.parse_args(argv)
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.workload]
    if a.warmup is None:
        a.warmup = DEFAULT_WARMUP[a.workload]
    a.warmup = max(3, a.warmup)
    return a


# ------------------------------------------------------------------------------------------ env

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, local, backend=None):
    if world > 1:
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's value (max) on every rank."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processed units_per_step per step; time = slowest rank."""
    return units_per_step * steps * world / (max_ms / 1e3)


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def spawn_ranks(n: int, argv) -> int:
    """Runs this script as n ranks on this node (RANK / LOCAL_RANK / WORLD_SIZE / MASTER_* set as a
    launcher would, rendezvous on 127.0.0.1); returns the worst exit code."""
    port = free_port()
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n), LOCAL_WORLD_SIZE=str(n),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *argv], env=env))
    rcs = [p.wait() for p in procs]
    return max(rcs, key=abs)


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background (every 50 ms)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={device_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [s for t, s in self.samples if t0 - 0.1 <= t <= t1 + 0.1]
        where = "timed region"
        if len(win) < 2:
            win = [s for _, s in self.samples]
            where = "whole run (timed region shorter than the sampling interval)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in win if num(s[0]) is not None]
        mx = [num(s[1]) for s in win if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4)
                          if len(s) > 4 + i and s[4 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(win), "window": where,
                "power_w_max": max([num(s[2]) for s in win if num(s[2]) is not None], default=None)}


def kernel_source_digest(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "speculative_decoding_draft_dh_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str, workload: str, files):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if the kernel source is
    unchanged since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(f"{workload}:{kernel}")
        if e and e.get("source_digest") == kernel_source_digest(files):
            return e.get("dram_bytes_per_launch")
    except (ValueError, OSError):
        return None
    return None


# ------------------------------------------------------------------------------------- head

KERNEL_FILES = {"scores_summary": ["gemv_topk.cu", "dh_internal.cuh"],
                "scores_small": ["small_b.cu", "sm100.cuh", "dh_internal.cuh"],
                "scores_lsu": ["small_b.cu", "sm100.cuh", "dh_internal.cuh"],
                "proj_small": ["small_b.cu", "dh_internal.cuh"],
                "lowrank_mma": ["mma_topk.cu", "sm100.cuh", "dh_internal.cuh"],
                "select": ["select.cu", "select.cuh", "dh_internal.cuh"],
                "rescore": ["rescore.cu", "dh_internal.cuh"],
                "rescore_ring": ["rescore.cu", "sm100.cuh", "dh_internal.cuh"],
                "rescore_cluster": ["rescore.cu", "sm100.cuh", "dh_internal.cuh"],
                "head_cluster": ["head_cl.cu", "select.cuh", "dh_internal.cuh"],
                "expand": ["expand.cu", "dh_internal.cuh"],
                "proj_partial": ["proj.cu", "dh_internal.cuh"],
                "proj_mma": ["mma_topk.cu", "sm100.cuh", "dh_internal.cuh"],
                "proj_reduce_mma": ["mma_topk.cu", "sm100.cuh", "dh_internal.cuh"],
                "tree_argmax": ["tree.cu", "dh_internal.cuh"],
                "tree_walk": ["tree.cu", "dh_internal.cuh"],
                "size_level": ["sizing.cu", "dh_internal.cuh"],
                "verify_stats": ["verify.cu", "dh_internal.cuh"],
                "verify_walk": ["verify.cu", "dh_internal.cuh"]}


def head_bytes(cfg):
    """HBM bytes of one call: U, V, h once and the B*K gathered rows of W."""
    e = 2 if cfg.dtype == "bf16" else 4
    return {"U": cfg.d * cfg.r * e, "V": cfg.r * cfg.vocab * e, "h": cfg.B * cfg.d * e,
            "W_rows": cfg.B * cfg.K * cfg.d * e}


def stage1_on_tensor_cores(cfg) -> bool:
    """The library runs stage 1 on the tensor cores for bf16 batches above four rows."""
    return cfg.dtype == "bf16" and cfg.B > 4


def path_ideal(cfg, unique_rows, peaks):
    """Ideal time of one call per the measurement rule: per stage max(bytes / copy bandwidth,
    FLOPs / peak of the unit that runs it), summed; stage 2 reads each distinct W row once."""
    e = 2 if cfg.dtype == "bf16" else 4
    bw = peaks["hbm_gbs"] * 1e9
    s1_bytes = cfg.d * cfg.r * e + cfg.r * cfg.vocab * e + cfg.B * cfg.d * e
    s1_flops = 2.0 * cfg.B * (cfg.d * cfg.r + cfg.r * cfg.vocab)
    s1_peak = (peaks["bf16_tflops"] if stage1_on_tensor_cores(cfg) else FP32_CORE_TFLOPS) * 1e12
    s2_bytes = unique_rows * cfg.d * e + cfg.B * cfg.d * e
    s2_flops = 2.0 * cfg.B * cfg.K * cfg.d
    s2_peak = FP32_CORE_TFLOPS * 1e12
    t1 = max(s1_bytes / bw, s1_flops / s1_peak)
    t2 = max(s2_bytes / bw, s2_flops / s2_peak)
    return {"stage1_us": t1 * 1e6, "stage1_bound": "hbm" if s1_bytes / bw >= s1_flops / s1_peak else
            ("tensor" if stage1_on_tensor_cores(cfg) else "alu"),
            "stage1_bytes": s1_bytes, "stage1_flops": s1_flops,
            "stage2_us": t2 * 1e6, "stage2_bound": "hbm" if s2_bytes / bw >= s2_flops / s2_peak else "alu",
            "stage2_bytes_unique_rows": s2_bytes, "ideal_us": (t1 + t2) * 1e6}


def kernel_algo(cfg, name, peaks, unique_rows=None):
    """(bound, algorithmic work per launch, unit) of a head kernel: HBM bytes the step must move,
    or tensor FLOPs of the dense contraction when those take longer at the peaks.  The rescoring
    kernels are charged at the distinct W rows of the step (unique_rows; all B*K when not given)."""
    e = 2 if cfg.dtype == "bf16" else 4
    if name in ("scores_small", "scores_lsu", "scores_summary"):
        return "hbm", cfg.r * cfg.vocab * e + cfg.B * cfg.r * e, "GB/s"
    if name in ("proj_small", "proj_partial"):
        return "hbm", cfg.d * cfg.r * e + cfg.B * cfg.d * e, "GB/s"
    if name in ("lowrank_mma", "proj_mma"):
        flops = 2.0 * cfg.B * cfg.r * (cfg.vocab if name == "lowrank_mma" else cfg.d)
        nbytes = cfg.r * (cfg.vocab if name == "lowrank_mma" else cfg.d) * e + cfg.B * cfg.r * e
        if flops / (peaks["bf16_tflops"] * 1e12) > nbytes / (peaks["hbm_gbs"] * 1e9):
            return "tensor", flops, "TFLOP/s"
        return "hbm", nbytes, "GB/s"
    if name == "expand":  # candidates' probabilities and ids in, children out
        return "hbm", cfg.B * cfg.K * 8 + cfg.B * 4 * 8 + cfg.B * 8, "GB/s"
    if name == "head_cluster":  # records read once, the candidates' W rows, h
        return "hbm", cfg.B * ((cfg.vocab + 63) // 64) * 16 + cfg.B * cfg.K * cfg.d * e + cfg.B * cfg.d * e, "GB/s"
    if name in ("rescore", "rescore_ring", "rescore_cluster"):
        rows = cfg.B * cfg.K if unique_rows is None else unique_rows
        return "hbm", rows * cfg.d * e + cfg.B * cfg.d * e, "GB/s"
    if name == "select":
        return "hbm", cfg.B * ((cfg.vocab + 63) // 64) * 16, "GB/s"
    if name == "size_level":  # the children in, the next frontier out
        sz = SIZE_LEVEL.get(cfg.name, {"wmax": 0})
        return "hbm", cfg.B * EXPAND_W.get(cfg.name, 0) * 8 + cfg.B * 4 + sz.get("requests", 0) * sz["wmax"] * 12, "GB/s"
    return "hbm", 0, "GB/s"


def kernel_roofline(cfg, name, stages, peaks, peak_src, workload, unique_rows=None):
    bound, algo, unit = kernel_algo(cfg, name, peaks, unique_rows)
    dur_s = stages[name]["us_avg"] * 1e-6
    if bound == "tensor":
        achieved, peak = algo / dur_s / 1e12, peaks["bf16_tflops"]
        src = f"{peak_src} (MEASURED_PEAKS.json bf16_tflops, burst)"
    else:
        achieved, peak = algo / dur_s / 1e9, peaks["hbm_gbs"]
        src = f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
    traffic = traffic_from_profiles(name, workload, KERNEL_FILES.get(name, []))
    out = {"kernel": name, "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
           "frac": round(achieved / peak, 4), "traffic": traffic,
           ("algorithmic_flops_per_launch" if bound == "tensor" else "algorithmic_bytes_per_launch"): algo,
           "us_per_launch": round(stages[name]["us_avg"], 3), "peak_source": src}
    if traffic and bound == "hbm" and algo:
        out["traffic_over_algorithmic"] = round(traffic / algo, 3)
    if unique_rows is not None and name in ("rescore", "rescore_ring", "rescore_cluster"):
        e = 2 if cfg.dtype == "bf16" else 4
        out["algorithmic_bytes_bk_rows"] = cfg.B * cfg.K * cfg.d * e + cfg.B * cfg.d * e  # every gathered row
        out["unique_w_rows"] = unique_rows
    return out


def auto_steps(per_step_us: float, chunk: int, floor: int) -> int:
    """Steps for a timed region of at least MIN_TIMED_S, a multiple of chunk."""
    n = max(floor, math.ceil(MIN_TIMED_S / (per_step_us * 1e-6)))
    return int(math.ceil(n / chunk) * chunk)


def run_head_bench(a, cfg, rank, world, local, peaks, peak_src, steps=None, warmup=None, cpu_seconds=None):
    """Times one head workload.  steps None: enough steps for MIN_TIMED_S."""
    from speculative_decoding_draft_dh_gb300 import binding as dh
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    warmup = a.warmup if warmup is None else warmup
    hb = head_bytes(cfg)
    per_step = sum(hb.values())
    copies = max(2, min(8, math.ceil(2 * L2_BYTES / per_step)))
    sets = []
    for i in range(copies):
        x = inputs.make_head(cfg, seed=a.seed + 1000 * rank + i, device=dev)
        x["idx"] = torch.empty(cfg.B, cfg.K, dtype=torch.int32, device=dev)
        x["score"] = torch.empty(cfg.B, cfg.K, dtype=torch.float32, device=dev)
        x["logits"] = torch.empty(cfg.B, cfg.K, dtype=torch.float32, device=dev)
        x["probs"] = torch.empty(cfg.B, cfg.K, dtype=torch.float32, device=dev)
        sets.append(x)
    ws = dh.Workspace()
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # the inputs were made on the current stream

    expand_w = EXPAND_W.get(cfg.name, 0)
    sizing = SIZE_LEVEL.get(cfg.name)
    if sizing:
        cost, bins = inputs.latency_table(sizing["wmax"])
        cost_d, bins_d = torch.from_numpy(cost).to(dev), torch.from_numpy(bins).to(dev)
        R = sizing["requests"]
    for x in sets:
        if expand_w:
            x["par"] = torch.linspace(1.0, 0.25, cfg.B, device=dev, dtype=torch.float32)
            x["ctok"] = torch.empty(cfg.B, expand_w, dtype=torch.int32, device=dev)
            x["cprob"] = torch.empty(cfg.B, expand_w, dtype=torch.float32, device=dev)
            x["keep"] = torch.empty(cfg.B, dtype=torch.int32, device=dev)
        if sizing:
            w = sizing["wmax"]
            x["next"] = {"width": torch.empty(R, dtype=torch.int32, device=dev),
                         "parent": torch.empty(R, w, dtype=torch.int32, device=dev),
                         "token": torch.empty(R, w, dtype=torch.int32, device=dev),
                         "prob": torch.empty(R, w, dtype=torch.float32, device=dev)}

    def step(x, idx=None, logits=None, probs=None):
        idx = x["idx"] if idx is None else idx
        logits = x["logits"] if logits is None else logits
        probs = x["probs"] if probs is None else probs
        if a.api == "head":
            dh.draft_head(x["h"], x["U"], x["V"], x["W"], cfg.K, idx_out=idx, score_out=x["score"],
                          logits_out=logits, probs_out=probs, workspace=ws)
        else:
            dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K, idx_out=idx, score_out=x["score"], workspace=ws)
            dh.exact_rescore(x["h"], x["W"], idx, logits_out=logits, probs_out=probs, workspace=ws)
        if expand_w:  # one draft level: the frontier nodes' children by exact probability
            dh.expand_children(probs, idx, expand_w, parent_prob=x["par"], min_benefit=1e-3,
                               child_token=x["ctok"], child_prob=x["cprob"], n_keep=x["keep"])
        if sizing:  # and the next level's width at the current load
            F = cfg.B // R
            dh.size_level(x["cprob"].view(R, F, expand_w), x["ctok"].view(R, F, expand_w), cost_d, bins_d, R,
                          sizing["theta"], n_valid=x["keep"].view(R, F), out=x["next"])

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(sets[i % copies])
    torch.cuda.synchronize()
    # One graph holds S consecutive steps over the rotating copies (S a multiple of the copy count),
    # so that host-side replay overhead is spread over many steps and the GPU never waits for the
    # host; a second graph holds the remainder of the steps.
    per_graph = max(copies, (64 // copies) * copies)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(n):
                step(sets[j % copies])
        return g

    g_full = capture(per_graph)
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(max(3, warmup) / per_graph))):
            g_full.replay()
    torch.cuda.synchronize()
    if steps is None:  # calibrate on a few replays
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            c0.record(stream)
            for _ in range(3):
                g_full.replay()
            c1.record(stream)
        torch.cuda.synchronize()
        steps = auto_steps(c0.elapsed_time(c1) * 1e3 / (3 * per_graph), per_graph, per_graph)
        steps = int(max_over_ranks(steps, world))
    S = min(steps, per_graph)
    if S != per_graph:
        g_full = capture(S)
    rem = steps % S
    g_rem = capture(rem) if rem else None

    def run_steps(n):
        for _ in range(n // S):
            g_full.replay()
        if n % S:
            assert n % S == rem
            g_rem.replay()

    sampler = ClockSampler(local)
    time.sleep(0.15)
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(min(warmup, 50) / S))):
            g_full.replay()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        run_steps(steps)
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    time.sleep(0.12)
    sampler.stop()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    us_per_call = ms * 1e3 / steps
    value = weak_scaling_value(cfg.B, steps, world, ms)

    # spread: each replay of the S-step graph timed on its own (after the headline measurement)
    n_rep = max(5, min(50, steps // S))
    rep_us = []
    with torch.cuda.stream(stream):
        for _ in range(n_rep):
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            r0.record(stream)
            g_full.replay()
            r1.record(stream)
            rep_us.append((r0, r1))
    torch.cuda.synchronize()
    rep_us = sorted(r0.elapsed_time(r1) * 1e3 / S for r0, r1 in rep_us)
    spread = {"us_per_call_p10": round(rep_us[len(rep_us) // 10], 3),
              "us_per_call_median": round(rep_us[len(rep_us) // 2], 3),
              "us_per_call_p90": round(rep_us[(9 * len(rep_us)) // 10], 3), "replays": n_rep,
              "steps_per_replay": S}
    # stream-queued: the same calls launched eagerly back to back (no graph)
    n_eager = min(steps, 1000 if cfg.B <= 64 else 50)
    with torch.cuda.stream(stream):
        for i in range(3):
            step(sets[i % copies])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_eager):
            step(sets[i % copies])
        e1.record(stream)
    torch.cuda.synchronize()
    spread["us_per_call_stream_queued"] = round(e0.elapsed_time(e1) * 1e3 / n_eager, 3)
    # distinct W rows among the candidates of one step (the rescoring's algorithmic bytes)
    e_sz = 2 if cfg.dtype == "bf16" else 4
    uniq = int(torch.unique(sets[0]["idx"]).numel())

    # per-kernel events on the launch stream (separate pass, eager launches)
    n_prof = min(steps, 2000 if cfg.B <= 64 else 200)
    dh.prof_enable(True)
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            step(sets[i % copies])
    torch.cuda.synchronize()
    dh.prof_enable(False)
    prof = dh.prof_read()
    stages = {k: {"us_avg": v[0] * 1e3 / v[1], "launches": v[1]} for k, v in prof.items()}
    launches_per_step = sum(v[1] for v in prof.values()) / n_prof
    name = ROOFLINE_KERNEL.get(cfg.name)
    if name not in stages:
        name = max(stages, key=lambda k: stages[k]["us_avg"])
    roofline = kernel_roofline(cfg, name, stages, peaks, peak_src, cfg.name, uniq)
    dom = max(stages, key=lambda k: stages[k]["us_avg"])
    roofline_time_dominant = None
    if dom != name:
        roofline_time_dominant = kernel_roofline(cfg, dom, stages, peaks, peak_src, cfg.name, uniq)

    ideal = path_ideal(cfg, uniq, peaks)
    hbm = peaks["hbm_gbs"]
    path_roofline = {"rule": "sum over stages of max(bytes / copy bandwidth, FLOPs / unit peak); stage 2 at "
                             "distinct W rows",
                     "ideal_us": round(ideal["ideal_us"], 3), "measured_us": round(us_per_call, 3),
                     "frac": round(ideal["ideal_us"] / us_per_call, 4),
                     "stage1_us": round(ideal["stage1_us"], 3), "stage1_bound": ideal["stage1_bound"],
                     "stage2_us": round(ideal["stage2_us"], 3), "stage2_bound": ideal["stage2_bound"],
                     "unique_w_rows": uniq, "gathered_w_rows": cfg.B * cfg.K,
                     "peaks": {"hbm_gbs": hbm, "bf16_tflops": peaks["bf16_tflops"],
                               "fp32_core_tflops": round(FP32_CORE_TFLOPS, 1)}}
    # secondary: every byte over the copy bandwidth, with the B*K gathered rows
    path_roofline["frac_hbm_bytes_bk_rows"] = round(per_step / (us_per_call * 1e-6) / 1e9 / hbm, 4)

    e2e = None
    if not a.no_e2e:
        e2e = head_e2e(a, cfg, sets, copies, step, stream, world, e_sz, S)

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_head_baseline(cfg, sets[0], a.cpu_seconds if cpu_seconds is None else cpu_seconds)
    clocks = sampler.summary(t0, t1)
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "rows/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms / steps, 6), "timed_ms": round(ms, 3),
        "us_per_call": round(us_per_call, 3), "timing_spread": spread, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded generators, random weights)",
        "config": {"workload": cfg.name, "B": cfg.B, "d": cfg.d, "vocab": cfg.vocab, "r": cfg.r,
                   "K": cfg.K, "seed": a.seed, "api": "dh_draft_head" if a.api == "head" else
                   "dh_lowrank_topk + dh_exact_rescore", "graph": f"CUDA graphs of {S} steps",
                   "l2": f"inputs rotate over {copies} independent copies "
                         f"({copies * per_step / 2**20:.0f} MiB per cycle > 2x L2)",
                   "parallelism": f"replicas x{world} (rows independent; no collective in the data path)"},
        "roofline": roofline, "roofline_time_dominant": roofline_time_dominant,
        "path_roofline": path_roofline, "stages": stages,
        "draft_level": None if not expand_w else {
            "frontier_nodes_per_s": round(value, 1), "levels_per_s": round(value / cfg.B, 1),
            "children_per_node": expand_w,
            "sizing": None if not sizing else dict(sizing, table="synthetic latency table (inputs.latency_table)",
                                                    next_width=sets[0]["next"]["width"].tolist())},
        "gpu_launches": int(round(launches_per_step * steps)), "e2e": e2e,
        "cpu_baseline": cpu, "clocks": clocks,
    }


def head_e2e(a, cfg, sets, copies, step, stream, world, e_sz, S):
    """End to end through the public API: each step copies its h from pinned host memory, runs
    the head and copies its results (idx, logits, probs) back, in stream order."""
    dev = sets[0]["h"].device
    hosts = [x["h"].cpu().pin_memory() for x in sets]
    BK = cfg.B * cfg.K
    # the three outputs live in one device buffer (idx, logits, probs as int32 / fp32 views), so
    # one device-to-host copy returns a step's results
    packed = [torch.empty(3 * BK, dtype=torch.int32, device=dev) for _ in sets]
    outs = [torch.empty(3 * BK, dtype=torch.int32).pin_memory() for _ in sets]
    views = [(p[:BK].view(cfg.B, cfg.K), p[BK:2 * BK].view(torch.float32).view(cfg.B, cfg.K),
              p[2 * BK:].view(torch.float32).view(cfg.B, cfg.K)) for p in packed]

    def one(j):
        x = sets[j]
        idx, logits, probs = views[j]
        x["h"].copy_(hosts[j], non_blocking=True)
        step(x, idx, logits, probs)
        outs[j].copy_(packed[j], non_blocking=True)

    # (1) graphs of S steps: step j copies its h in on a copy stream (as soon as step j - copies,
    # the last user of that buffer, is done), runs on the compute stream, and copies its results
    # out on a third stream, so the copies of one step overlap the kernels of the others: a
    # pipelined caller that keeps the GPU fed
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    g_steps = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_steps, stream=stream):
        done = [None] * copies   # event after the kernels of the last step that used each buffer set
        out_free = [None] * copies
        for j in range(S):
            c = j % copies
            x = sets[c]
            idx, logits, probs = views[c]
            h2d_s.wait_stream(stream) if done[c] is None else h2d_s.wait_event(done[c])
            with torch.cuda.stream(h2d_s):
                x["h"].copy_(hosts[c], non_blocking=True)
                h_in = torch.cuda.Event()
                h_in.record(h2d_s)
            stream.wait_event(h_in)
            if out_free[c] is not None:
                stream.wait_event(out_free[c])
            step(x, idx, logits, probs)
            ev = torch.cuda.Event()
            ev.record(stream)
            done[c] = ev
            d2h_s.wait_event(ev)
            with torch.cuda.stream(d2h_s):
                outs[c].copy_(packed[c], non_blocking=True)
                of = torch.cuda.Event()
                of.record(d2h_s)
            out_free[c] = of
        stream.wait_stream(h2d_s)
        stream.wait_stream(d2h_s)
    n = S * max(1, min(2000 if cfg.B <= 64 else 200, 20 * S) // S)
    with torch.cuda.stream(stream):
        g_steps.replay()
    stream.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(n // S):
            g_steps.replay()
    stream.synchronize()
    te = max_over_ranks(time.perf_counter() - t0, world)
    # (2) one graph replay per step, synchronising after every step (a caller that waits for each
    # result before the next step)
    graphs = []
    for j in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            one(j)
        graphs.append(g)
    n_sync = max(copies, n // 4)
    with torch.cuda.stream(stream):
        for j in range(copies):
            graphs[j].replay()
    stream.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_sync):
            graphs[i % copies].replay()
            stream.synchronize()
    ts = max_over_ranks(time.perf_counter() - t0, world)
    # (3) eager launches through the Python binding, synchronising every step
    n_py = max(copies, n // 4)
    with torch.cuda.stream(stream):
        for i in range(3):
            one(i % copies)
    stream.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_py):
            one(i % copies)
            stream.synchronize()
    tp = max_over_ranks(time.perf_counter() - t0, world)
    return {"value": round(cfg.B * n * world / te, 2), "unit": "rows/s",
            "us_per_call": round(te * 1e6 / n, 3), "steps": n,
            "how": f"wall clock; every step copies its h from pinned host memory, runs dh_draft_head and "
                   f"copies its results to pinned host memory; copies on their own streams overlap other steps' "
                   f"kernels; CUDA graphs of {S} such steps",
            "h2d_bytes_per_step": int(cfg.B * cfg.d * e_sz), "d2h_bytes_per_step": int(BK * 12),
            "synchronized_each_step": {"us_per_call": round(ts * 1e6 / n_sync, 3), "steps": n_sync},
            "python_eager_each_step": {"us_per_call": round(tp * 1e6 / n_py, 3), "steps": n_py}}


def cpu_head_baseline(cfg, x, seconds):
    import oracle
    oracle.build()
    hc, Uc, Vc, Wc = x["h"].cpu(), x["U"].cpu(), x["V"].cpu(), x["W"].cpu()
    cores = len(os.sched_getaffinity(0))
    rows_done = 0
    t0 = time.perf_counter()
    b = 0
    while time.perf_counter() - t0 < seconds or rows_done == 0:
        chunk = [(b + i) % cfg.B for i in range(min(cfg.B, cores))]
        idx, _ = oracle.lowrank_topk(hc, Uc, Vc, cfg.K, rows=chunk)
        full_idx = np.zeros((cfg.B, cfg.K), dtype=np.int32)
        full_idx[chunk] = idx
        _, p = oracle.exact_rescore(hc, Wc, full_idx, rows=chunk)
        if EXPAND_W.get(cfg.name, 0):
            oracle.expand_children(p.astype(np.float32), idx, EXPAND_W[cfg.name], min_benefit=1e-3)
        rows_done += len(chunk)
        b += len(chunk)
    dt = time.perf_counter() - t0
    used = min(cfg.B, cores)
    what = "stage 1 + stage 2" + (" + expansion" if EXPAND_W.get(cfg.name, 0) else "")
    return {"value": round(rows_done / dt, 4), "unit": "rows/s", "cores": used, "cpu_model": cpu_model(),
            "kind": "oracle",
            "sample": f"{rows_done} rows of the {cfg.name} workload ({what}), {dt:.1f} s, OpenMP over rows"}


# ------------------------------------------------------------------------------------- tree

def run_tree_bench(a, tcfg, rank, world, local, peaks, peak_src, steps=None, warmup=None, cpu_seconds=None):
    from speculative_decoding_draft_dh_gb300 import binding as dh
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    warmup = a.warmup if warmup is None else warmup
    t = inputs.make_tree(tcfg, seed=a.seed + 1000 * rank, device=dev)
    ws = dh.Workspace()
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # the inputs were made on the current stream
    B, N, vocab = tcfg.B, tcfg.N, tcfg.vocab
    elem = 2 if tcfg.dtype == "bf16" else 4
    logit_bytes = B * N * vocab * elem

    def step():
        return dh.tree_accept(t["logits"], t["parent"], t["token"], workspace=ws)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    if steps is None:
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            c0.record(stream)
            for _ in range(5):
                g.replay()
            c1.record(stream)
        torch.cuda.synchronize()
        steps = int(max_over_ranks(auto_steps(c0.elapsed_time(c1) * 1e3 / 5, 1, 10), world))
    sampler = ClockSampler(local)
    time.sleep(0.15)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    time.sleep(0.12)
    sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    us = ms * 1e3 / steps
    value = weak_scaling_value(B, steps, world, ms)
    n_prof = min(steps, 50)
    dh.prof_enable(True)
    with torch.cuda.stream(stream):
        for _ in range(n_prof):
            step()
    torch.cuda.synchronize()
    dh.prof_enable(False)
    prof = dh.prof_read()
    stages = {k: {"us_avg": v[0] * 1e3 / v[1], "launches": v[1]} for k, v in prof.items()}
    dom = "tree_argmax"
    achieved = logit_bytes / (stages[dom]["us_avg"] * 1e-6) / 1e9
    peak = peaks["hbm_gbs"]
    traffic = traffic_from_profiles(dom, tcfg.name, KERNEL_FILES[dom])
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": logit_bytes,
                "us_per_launch": round(stages[dom]["us_avg"], 3),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"}
    if traffic:
        roofline["traffic_over_algorithmic"] = round(traffic / logit_bytes, 3)
    path_bytes = logit_bytes + 2 * B * N * 4
    ideal_us = path_bytes / (peak * 1e9) * 1e6
    path_roofline = {"rule": "logits, parents and tokens read once over the copy bandwidth",
                     "ideal_us": round(ideal_us, 3), "measured_us": round(us, 3), "frac": round(ideal_us / us, 4)}
    e2e = None
    if not a.no_e2e:
        n_e2e = min(steps, 10)
        host = {k: t[k].cpu().pin_memory() for k in ("logits", "parent", "token")}
        out_host = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in step().items()
                    if k in ("path", "len", "bonus")}

        def one():
            for k in host:
                t[k].copy_(host[k], non_blocking=True)
            o = step()
            for k in out_host:
                out_host[k].copy_(o[k], non_blocking=True)
        torch.cuda.synchronize()
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=stream):
            one()
        with torch.cuda.stream(stream):
            ge.replay()
        stream.synchronize()
        te0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(n_e2e):
                ge.replay()
        stream.synchronize()
        te = max_over_ranks(time.perf_counter() - te0, world)
        e2e = {"value": round(B * n_e2e * world / te, 2), "unit": "requests/s",
               "us_per_call": round(te * 1e6 / n_e2e, 1), "steps": n_e2e,
               "how": "wall clock; per step one CUDA-graph replay of: logits, parents and tokens copied from "
                      "pinned host memory, dh_tree_accept, path / len / bonus copied back",
               "h2d_bytes_per_step": int(logit_bytes + 2 * B * N * 4),
               "d2h_bytes_per_step": int(B * N * 4 + 2 * B * 4)}
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_tree_baseline(tcfg, t, a.cpu_seconds if cpu_seconds is None else cpu_seconds)
    return {
        "metric": TREE_METRIC, "value": round(value, 2), "unit": "requests/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms / steps, 6), "timed_ms": round(ms, 3),
        "us_per_call": round(us, 3), "node_rows_per_s": round(value * N, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": tcfg.dtype,
        "data": "synthetic (seeded generators)",
        "config": {"workload": tcfg.name, "B": B, "N": N, "vocab": vocab, "seed": a.seed,
                   "graph": "one CUDA graph per step",
                   "l2": f"logits {logit_bytes / 2**30:.2f} GiB per step > L2",
                   "parallelism": f"replicas x{world} (requests independent; no collective in the data path)"},
        "roofline": roofline, "path_roofline": path_roofline, "stages": stages,
        "gpu_launches": int(round(sum(v[1] for v in prof.values()) / n_prof * steps)),
        "e2e": e2e, "cpu_baseline": cpu, "clocks": sampler.summary(t0, t1),
    }


def cpu_tree_baseline(tcfg, t, seconds):
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    n = min(tcfg.B, cores)
    sl = t["logits"][:n].cpu()
    pa, to = t["parent"][:n].cpu(), t["token"][:n].cpu()
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or done == 0:
        oracle.tree_accept(sl, pa, to)
        done += n
    dt = time.perf_counter() - t0
    return {"value": round(done / dt, 3), "unit": "requests/s", "cores": n, "cpu_model": cpu_model(),
            "kind": "oracle", "sample": f"{done} requests (first {n} of the tree workload, repeated), {dt:.1f} s"}


VERIFY_METRIC = ("chain-verification requests/sec and µs per call (speculative sampling: target softmax "
                 "statistics, acceptance tests, residual or bonus draw); % of HBM roofline")


def run_verify_bench(a, vcfg, rank, world, local, peaks, peak_src, steps=None, warmup=None, cpu_seconds=None):
    """Times dh_verify_chain on the chain-verification workload (B requests of L drafted tokens)."""
    from speculative_decoding_draft_dh_gb300 import binding as dh
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    warmup = a.warmup if warmup is None else warmup
    B, L, vocab = vcfg.B, vcfg.L, vcfg.vocab
    elem = 2 if vcfg.dtype == "bf16" else 4
    logit_bytes = B * (L + 1) * vocab * elem
    copies = max(2, min(8, math.ceil(2 * L2_BYTES / logit_bytes)))
    sets = [inputs.make_verify(vcfg, seed=a.seed + 1000 * rank + i, device=dev) for i in range(copies)]
    for v in sets:
        v["n"] = torch.empty(B, dtype=torch.int32, device=dev)
        v["tok"] = torch.empty(B, dtype=torch.int32, device=dev)
    ws = dh.Workspace()
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # the inputs were made on the current stream

    def step(v):
        dh.verify_chain(v["logits"], v["cand_idx"], v["cand_prob"], v["draft_token"], v["u_accept"], v["u_sample"],
                        temperature=vcfg.temperature, n_accept_out=v["n"], token_out=v["tok"], workspace=ws)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(sets[i % copies])
    torch.cuda.synchronize()
    S = copies * max(1, 16 // copies)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for j in range(S):
            step(sets[j % copies])
    if steps is None:
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            c0.record(stream)
            for _ in range(3):
                g.replay()
            c1.record(stream)
        torch.cuda.synchronize()
        steps = int(max_over_ranks(auto_steps(c0.elapsed_time(c1) * 1e3 / (3 * S), S, S), world))
    steps = max(S, steps // S * S)
    sampler = ClockSampler(local)
    time.sleep(0.15)
    with torch.cuda.stream(stream):
        g.replay()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps // S):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    time.sleep(0.12)
    sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    us = ms * 1e3 / steps
    value = weak_scaling_value(B, steps, world, ms)
    n_prof = min(steps, 200)
    dh.prof_enable(True)
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            step(sets[i % copies])
    torch.cuda.synchronize()
    dh.prof_enable(False)
    prof = dh.prof_read()
    stages = {k: {"us_avg": v[0] * 1e3 / v[1], "launches": v[1]} for k, v in prof.items()}
    dom = "verify_stats"
    achieved = logit_bytes / (stages[dom]["us_avg"] * 1e-6) / 1e9
    peak = peaks["hbm_gbs"]
    traffic = traffic_from_profiles(dom, vcfg.name, ["verify.cu", "dh_internal.cuh"])
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "algorithmic_bytes_per_launch": logit_bytes,
                "us_per_launch": round(stages[dom]["us_avg"], 3),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"}
    if traffic:
        roofline["traffic_over_algorithmic"] = round(traffic / logit_bytes, 3)
    in_bytes = logit_bytes + B * L * vcfg.K * 8 + B * L * 8 + B * 4
    ideal_us = in_bytes / (peak * 1e9) * 1e6
    path_roofline = {"rule": "target logits and the draft's inputs read once over the copy bandwidth",
                     "ideal_us": round(ideal_us, 3), "measured_us": round(us, 3), "frac": round(ideal_us / us, 4)}
    accept = float(sets[0]["n"].float().mean().item())
    e2e = None
    if not a.no_e2e:
        v = sets[0]
        keys = ("logits", "cand_idx", "cand_prob", "draft_token", "u_accept", "u_sample")
        host = {k: v[k].cpu().pin_memory() for k in keys}
        out_host = {k: torch.empty(B, dtype=torch.int32).pin_memory() for k in ("n", "tok")}

        def one():
            for k in keys:
                v[k].copy_(host[k], non_blocking=True)
            step(v)
            for k in out_host:
                out_host[k].copy_(v[k], non_blocking=True)
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=stream):
            one()
        with torch.cuda.stream(stream):
            ge.replay()
        stream.synchronize()
        n_e2e = 50
        te0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(n_e2e):
                ge.replay()
        stream.synchronize()
        te = max_over_ranks(time.perf_counter() - te0, world)
        e2e = {"value": round(B * n_e2e * world / te, 2), "unit": "requests/s", "us_per_call": round(te * 1e6 / n_e2e, 1),
               "steps": n_e2e, "how": "wall clock; per step one CUDA-graph replay of: every input copied from pinned "
                                      "host memory, dh_verify_chain, n_accept and token copied back",
               "h2d_bytes_per_step": int(in_bytes), "d2h_bytes_per_step": int(B * 8)}
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_verify_baseline(vcfg, sets[0], a.cpu_seconds if cpu_seconds is None else cpu_seconds)
    return {
        "metric": VERIFY_METRIC, "value": round(value, 2), "unit": "requests/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms / steps, 6), "timed_ms": round(ms, 3), "us_per_call": round(us, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": vcfg.dtype,
        "data": "synthetic (seeded generators)",
        "config": {"workload": vcfg.name, "B": B, "L": L, "vocab": vocab, "K": vcfg.K, "T": vcfg.temperature,
                   "seed": a.seed, "graph": f"CUDA graphs of {S} steps",
                   "l2": f"inputs rotate over {copies} copies ({copies * logit_bytes / 2**20:.0f} MiB per cycle > 2x L2)",
                   "accepted_per_request": round(accept, 3),
                   "parallelism": f"replicas x{world} (requests independent; no collective in the data path)"},
        "roofline": roofline, "path_roofline": path_roofline, "stages": stages,
        "gpu_launches": int(round(sum(x[1] for x in prof.values()) / n_prof * steps)),
        "e2e": e2e, "cpu_baseline": cpu, "clocks": sampler.summary(t0, t1),
    }


def cpu_verify_baseline(vcfg, v, seconds):
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    n = min(vcfg.B, cores)
    cpu = {k: t[:n].cpu() for k, t in v.items() if k not in ("n", "tok")}
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or done == 0:
        oracle.verify_chain(cpu["logits"], cpu["cand_idx"], cpu["cand_prob"], cpu["draft_token"], cpu["u_accept"],
                            cpu["u_sample"], temperature=vcfg.temperature)
        done += n
    dt = time.perf_counter() - t0
    return {"value": round(done / dt, 3), "unit": "requests/s", "cores": n, "cpu_model": cpu_model(),
            "kind": "oracle", "sample": f"{done} requests (first {n} of the verify workload, repeated), {dt:.1f} s"}


def summarize(line):
    """The fields of a workload's line kept in the headline's `workloads` object."""
    keep = ("metric", "value", "unit", "us_per_call", "steps", "timed_ms", "node_rows_per_s", "draft_level", "config",
            "path_roofline", "roofline", "roofline_time_dominant", "stages", "gpu_launches", "e2e",
            "cpu_baseline", "clocks", "timing_spread")
    return {k: line[k] for k in keep if k in line and line[k] is not None}


# -------------------------------------------------------------------------------- reference

def warm_up(fn, n, budget=20.0):
    """Up to n untimed calls of fn within budget seconds (at least one); returns the number done."""
    done, t0 = 0, time.perf_counter()
    while done < n and (done == 0 or time.perf_counter() - t0 < budget):
        fn()
        done += 1
    return done


def run_reference(a, rank, world):
    """The CPU oracle as the reference arm: bounded samples of the same workload on host cores."""
    if rank != 0:
        return None
    budget = 60.0
    if a.workload == "verify":
        vcfg = inputs.VERIFY_CONFIGS["verify"]
        import oracle
        oracle.build()
        cores = len(os.sched_getaffinity(0))
        n = min(vcfg.B, cores)
        v = {k: t[:n] for k, t in inputs.make_verify(vcfg, seed=a.seed, device="cpu").items()}

        def one_v():
            oracle.verify_chain(v["logits"], v["cand_idx"], v["cand_prob"], v["draft_token"], v["u_accept"],
                                v["u_sample"], temperature=vcfg.temperature)
        warm = warm_up(one_v, a.warmup)
        steps = 0
        t0 = time.perf_counter()
        while steps < a.steps and (time.perf_counter() - t0 < budget or steps == 0):
            one_v()
            steps += 1
        dt = time.perf_counter() - t0
        value = n * steps / dt
        unit, metric = "requests/s", VERIFY_METRIC
        sample = f"{steps} steps of {n} requests of the verify workload (L={vcfg.L}, vocab={vcfg.vocab})"
        cfgd = {"workload": "verify", "B": vcfg.B, "L": vcfg.L, "vocab": vcfg.vocab, "K": vcfg.K}
        threads = n
    elif a.workload == "tree":
        tcfg = inputs.TREE_CONFIGS["tree"]
        small = inputs.tree_config("tree", B=min(16, tcfg.B))
        t = inputs.make_tree(small, seed=a.seed, device="cpu")
        import oracle
        oracle.build()
        cores = len(os.sched_getaffinity(0))
        warm = warm_up(lambda: oracle.tree_accept(t["logits"], t["parent"], t["token"]), a.warmup)
        steps = 0
        t0 = time.perf_counter()
        while steps < a.steps and (time.perf_counter() - t0 < budget or steps == 0):
            oracle.tree_accept(t["logits"], t["parent"], t["token"])
            steps += 1
        dt = time.perf_counter() - t0
        value = small.B * steps / dt
        unit, metric = "requests/s", TREE_METRIC
        sample = f"{steps} steps of {small.B} requests of the tree workload (N=64, vocab=151936)"
        cfgd = {"workload": "tree", "B": tcfg.B, "N": tcfg.N, "vocab": tcfg.vocab}
        threads = min(small.B, cores)
    else:
        cfg = inputs.HEAD_CONFIGS[a.workload]
        x = inputs.make_head(cfg, seed=a.seed, device="cuda" if torch.cuda.is_available() else "cpu")
        x = {k: v.cpu() for k, v in x.items()}
        import oracle
        oracle.build()
        cores = len(os.sched_getaffinity(0))
        rows = list(range(min(cfg.B, cores)))
        ew = EXPAND_W.get(cfg.name, 0)

        def one_step():
            idx, _ = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K, rows=rows)
            full = np.zeros((cfg.B, cfg.K), dtype=np.int32)
            full[rows] = idx
            _, p = oracle.exact_rescore(x["h"], x["W"], full, rows=rows)
            if ew:
                oracle.expand_children(p.astype(np.float32), idx, ew, min_benefit=1e-3)
        warm = warm_up(one_step, a.warmup)
        steps = 0
        t0 = time.perf_counter()
        while steps < a.steps and (time.perf_counter() - t0 < budget or steps == 0):
            one_step()
            steps += 1
        dt = time.perf_counter() - t0
        value = len(rows) * steps / dt
        unit, metric = "rows/s", METRIC
        what = "stage 1 + stage 2" + (" + expansion" if ew else "")
        sample = f"{steps} steps of {len(rows)} rows of the {cfg.name} workload ({what})"
        cfgd = {"workload": cfg.name, "B": cfg.B, "d": cfg.d, "vocab": cfg.vocab, "r": cfg.r, "K": cfg.K}
        threads = len(rows)
    return {"impl": "reference", "metric": metric, "value": round(value, 4), "unit": unit,
            "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": round(dt * 1e3 / steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generators)", "config": cfgd,
            "cpu_baseline": {"value": round(value, 4), "unit": unit, "kind": "oracle", "cores": threads,
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def profile_run(a):
    """Small, bounded run for ncu: the workload's kernels launched eagerly on one input copy."""
    from speculative_decoding_draft_dh_gb300 import binding as dh
    dev = torch.device("cuda", 0)
    if a.workload == "tree":
        t = inputs.make_tree(inputs.TREE_CONFIGS["tree"], seed=a.seed, device=dev)
        for _ in range(a.warmup + a.steps):
            dh.tree_accept(t["logits"], t["parent"], t["token"])
    elif a.workload == "verify":
        v = inputs.make_verify(inputs.VERIFY_CONFIGS["verify"], seed=a.seed, device=dev)
        for _ in range(a.warmup + a.steps):
            dh.verify_chain(v["logits"], v["cand_idx"], v["cand_prob"], v["draft_token"], v["u_accept"],
                            v["u_sample"])
    else:
        cfg = inputs.HEAD_CONFIGS[a.workload]
        x = inputs.make_head(cfg, seed=a.seed, device=dev)
        ew = EXPAND_W.get(cfg.name, 0)
        sizing = SIZE_LEVEL.get(cfg.name)
        if sizing:
            cost, bins = inputs.latency_table(sizing["wmax"])
            cost_d, bins_d = torch.from_numpy(cost).to(dev), torch.from_numpy(bins).to(dev)
            par = torch.linspace(1.0, 0.25, cfg.B, device=dev, dtype=torch.float32)
        for _ in range(a.warmup + a.steps):
            if a.api == "head":
                idx, _, _, probs = dh.draft_head(x["h"], x["U"], x["V"], x["W"], cfg.K)
            else:
                idx, _ = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
                _, probs = dh.exact_rescore(x["h"], x["W"], idx)
            if ew:
                ctok, cprob, keep = dh.expand_children(probs, idx, ew, parent_prob=par if sizing else None,
                                                       min_benefit=1e-3)
                if sizing:
                    R = sizing["requests"]
                    F = cfg.B // R
                    dh.size_level(cprob.view(R, F, ew), ctok.view(R, F, ew), cost_d, bins_d, R, sizing["theta"],
                                  n_valid=keep.view(R, F))
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": a.workload, "steps": a.warmup + a.steps}), flush=True)


def dry_run(a, rank, world):
    """Multi-rank plumbing without a GPU: gloo rendezvous, a timed host loop per rank, the barrier,
    the max over ranks and the weak-scaling aggregate, as the GPU run does them."""
    import torch.distributed as dist
    dist_init(world, rank, backend="gloo")
    try:
        barrier(world)
        t0 = time.perf_counter()
        acc = 0.0
        for i in range(20000 * (1 + rank)):
            acc += math.sqrt(i)
        ms = (time.perf_counter() - t0) * 1e3
        slowest = max_over_ranks(ms, world)
        ranks = [None] * world
        if world > 1:
            dist.all_gather_object(ranks, {"rank": rank, "ms": ms})
        else:
            ranks = [{"rank": 0, "ms": ms}]
        barrier(world)
        if rank == 0:
            print(json.dumps({"dry_run": True, "n_gpus": world, "gpus_requested": a.gpus, "scaling": "weak",
                              "value": weak_scaling_value(1, 1, world, slowest), "ms_slowest": slowest,
                              "ranks": ranks}), flush=True)
    finally:
        if world > 1:
            dist.destroy_process_group()


def main():
    argv = sys.argv[1:]
    a = parse_args(argv)
    if a.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_ranks(a.gpus, argv))
    rank, world, local = dist_env()
    if a.dry_run:
        dry_run(a, rank, world)
        return
    if a.profile_run:
        from speculative_decoding_draft_dh_gb300 import build
        build.build()
        profile_run(a)
        return
    if a.impl == "reference":
        line = run_reference(a, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    if world != a.gpus:
        raise SystemExit(f"bench.py --gpus {a.gpus} but the launcher started {world} ranks")
    dist_init(world, local)
    from speculative_decoding_draft_dh_gb300 import build
    if rank == 0:
        build.build()
    barrier(world)
    build.build()
    peaks, src = load_peaks()
    if a.workload == "tree":
        line = run_tree_bench(a, inputs.TREE_CONFIGS["tree"], rank, world, local, peaks, src, steps=a.steps)
    elif a.workload == "verify":
        line = run_verify_bench(a, inputs.VERIFY_CONFIGS["verify"], rank, world, local, peaks, src, steps=a.steps)
    else:
        line = run_head_bench(a, inputs.HEAD_CONFIGS[a.workload], rank, world, local, peaks, src, steps=a.steps)
    if not a.only and a.workload == "batch1":
        work = {}
        for w in EXTRA_WORKLOADS:
            cpu_s = min(a.cpu_seconds, 5.0)
            if w == "tree":
                sub = run_tree_bench(a, inputs.TREE_CONFIGS["tree"], rank, world, local, peaks, src,
                                     warmup=DEFAULT_WARMUP[w], cpu_seconds=cpu_s)
            elif w == "verify":
                sub = run_verify_bench(a, inputs.VERIFY_CONFIGS["verify"], rank, world, local, peaks, src,
                                       warmup=DEFAULT_WARMUP[w], cpu_seconds=cpu_s)
            else:
                sub = run_head_bench(a, inputs.HEAD_CONFIGS[w], rank, world, local, peaks, src,
                                     warmup=DEFAULT_WARMUP[w], cpu_seconds=cpu_s)
            work[w] = summarize(sub)
            torch.cuda.empty_cache()
        line["workloads"] = work
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
