#!/usr/bin/env python3
"""Benchmark of the GB300 draft-head path (prints one JSON line on rank 0).

A step is one pass of the draft head over one batch: dh_lowrank_topk (projection, vocabulary-wide
low-rank scores, exact top-K) followed by dh_exact_rescore (gathered full-rank logits + softmax),
on the workload's synthetic inputs already resident in HBM.  ``--workload tree`` times
dh_tree_accept instead.

* value: rows per second over the whole job (sum over ranks / slowest rank's time); each step is
  a CUDA-graph replay of the two calls; input sets rotate over enough independent copies that the
  bytes touched between two uses of one copy exceed twice the L2 size.
* e2e: the same metric through the public Python API with the step's per-call input (h, or the
  tree inputs) copied from pinned host memory and the results copied back, synchronising each step.
* roofline: the dominant kernel's algorithmic bytes (or flops) per launch over its CUDA-event
  duration, from a second pass with per-kernel events on the launch stream.
* cpu_baseline: the CPU oracle timed on host cores on a bounded sample of the same workload.
* ``--impl reference``: the CPU oracle as the reference arm (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
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
DEFAULT_STEPS = {"batch1": 20000, "moderate": 5000, "high": 500, "tree": 200, "level": 10000}
DEFAULT_WARMUP = {"batch1": 200, "moderate": 50, "high": 10, "tree": 5, "level": 100}
EXPAND_W = {"level": 4}  # children per frontier node in the draft-level workload


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="batch1", choices=["batch1", "moderate", "high", "tree", "level"])
    ap.add_argument("--api", default="head", choices=["head", "split"],
                    help="head: dh_draft_head (both stages in one call); split: dh_lowrank_topk + "
                         "dh_exact_rescore")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile-run", action="store_true",
                    help="for profilers: one input copy, eager launches of warmup+steps steps, "
                         "no graphs, e2e, CPU baseline or clock sampling; prints a short line")
    a = ap.parse_args()
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


def dist_init(world, local):
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
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
                "tree_walk": ["tree.cu", "dh_internal.cuh"]}


def head_bytes(cfg):
    """Algorithmic HBM bytes of one call pair: U, V, h once and the B*K gathered rows of W."""
    e = 2 if cfg.dtype == "bf16" else 4
    return {"U": cfg.d * cfg.r * e, "V": cfg.r * cfg.vocab * e, "h": cfg.B * cfg.d * e,
            "W_rows": cfg.B * cfg.K * cfg.d * e}


def kernel_algo(cfg, name):
    """(bound, algorithmic work per launch, unit) of a head kernel: HBM bytes the step must move,
    or tensor FLOPs of the dense contraction (rows beyond B padded by the kernel are not counted)."""
    e = 2 if cfg.dtype == "bf16" else 4
    if name in ("scores_small", "scores_lsu"):
        return "hbm", cfg.r * cfg.vocab * e + cfg.B * cfg.r * e, "GB/s"
    if name == "proj_small":
        return "hbm", cfg.d * cfg.r * e + cfg.B * cfg.d * e, "GB/s"
    if name == "scores_summary":
        return "hbm", cfg.r * cfg.vocab * e + cfg.B * cfg.r * e, "GB/s"
    if name == "lowrank_mma":
        return "tensor", 2.0 * cfg.B * cfg.r * cfg.vocab, "TFLOP/s"
    if name == "proj_mma":
        return "tensor", 2.0 * cfg.B * cfg.d * cfg.r, "TFLOP/s"
    if name == "proj_partial":
        return "hbm", cfg.d * cfg.r * e + cfg.B * cfg.d * e, "GB/s"
    if name == "expand":  # candidates' probabilities and ids in, children out
        return "hbm", cfg.B * cfg.K * 8 + cfg.B * 4 * 8 + cfg.B * 8, "GB/s"
    if name == "head_cluster":  # records read once, the candidates' W rows, h
        return "hbm", cfg.B * ((cfg.vocab + 63) // 64) * 16 + cfg.B * cfg.K * cfg.d * e + cfg.B * cfg.d * e, "GB/s"
    if name in ("rescore", "rescore_ring", "rescore_cluster"):
        return "hbm", cfg.B * cfg.K * cfg.d * e + cfg.B * cfg.d * e, "GB/s"
    if name == "select":
        return "hbm", cfg.B * ((cfg.vocab + 63) // 64) * 16, "GB/s"
    return "hbm", 0, "GB/s"


def run_head_bench(a, cfg, rank, world, local, peaks, peak_src):
    from speculative_decoding_draft_dh_gb300 import binding as dh
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
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

    expand_w = EXPAND_W.get(cfg.name, 0)
    for x in sets:
        if expand_w:
            x["par"] = torch.linspace(1.0, 0.25, cfg.B, device=dev, dtype=torch.float32)
            x["ctok"] = torch.empty(cfg.B, expand_w, dtype=torch.int32, device=dev)
            x["cprob"] = torch.empty(cfg.B, expand_w, dtype=torch.float32, device=dev)
            x["keep"] = torch.empty(cfg.B, dtype=torch.int32, device=dev)

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

    with torch.cuda.stream(stream):
        for i in range(a.warmup):
            step(sets[i % copies])
    torch.cuda.synchronize()
    # One graph holds S consecutive steps over the rotating copies (S a multiple of the copy count),
    # so that host-side replay overhead (tens of µs per replay from Python) is spread over many
    # steps and the GPU never waits for the host; a second graph holds the remainder of the steps.
    per_graph = max(copies, (64 // copies) * copies)
    S = min(a.steps, per_graph)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(n):
                step(sets[j % copies])
        return g

    g_full = capture(S)
    rem = a.steps % S
    g_rem = capture(rem) if rem else None

    def run_steps(n):
        for _ in range(n // S):
            g_full.replay()
        if n % S:
            assert n % S == rem
            g_rem.replay()

    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(max(3, a.warmup) / S))):
            g_full.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    time.sleep(0.15)
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(min(a.warmup, 50) / S))):
            g_full.replay()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        run_steps(a.steps)
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    time.sleep(0.12)
    sampler.stop()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    us_per_call = ms * 1e3 / a.steps
    value = weak_scaling_value(cfg.B, a.steps, world, ms)

    # spread: each replay of the S-step graph timed on its own (after the headline measurement)
    n_rep = max(5, min(50, a.steps // S))
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
    n_eager = min(a.steps, 1000 if cfg.B <= 64 else 50)
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
    # distinct W rows among the candidates of one step (stage 2 reads each once from HBM; repeats
    # may hit L2)
    e_sz = 2 if cfg.dtype == "bf16" else 4
    uniq = int(torch.unique(sets[0]["idx"]).numel())

    # per-kernel events on the launch stream (separate pass, eager launches)
    n_prof = min(a.steps, 2000 if cfg.B <= 64 else 200)
    dh.prof_enable(True)
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            step(sets[i % copies])
    torch.cuda.synchronize()
    dh.prof_enable(False)
    prof = dh.prof_read()
    stages = {k: {"us_avg": v[0] * 1e3 / v[1], "launches": v[1]} for k, v in prof.items()}
    launches_per_step = sum(v[1] for v in prof.values()) / n_prof
    dom = max(stages, key=lambda k: stages[k]["us_avg"])
    bound, algo, unit = kernel_algo(cfg, dom)
    dur_s = stages[dom]["us_avg"] * 1e-6
    if bound == "tensor":
        achieved = algo / dur_s / 1e12
        peak = peaks["bf16_tflops"]
        peak_src_s = f"{peak_src} (MEASURED_PEAKS.json bf16_tflops, burst)"
    else:
        achieved = algo / dur_s / 1e9
        peak = peaks["hbm_gbs"]
        peak_src_s = f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
    traffic = traffic_from_profiles(dom, cfg.name, KERNEL_FILES.get(dom, []))
    roofline = {"kernel": dom, "bound": bound, "achieved": round(achieved, 1), "peak": peak,
                "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
                ("algorithmic_flops_per_launch" if bound == "tensor" else "algorithmic_bytes_per_launch"): algo,
                "us_per_launch": round(stages[dom]["us_avg"], 3), "peak_source": peak_src_s}
    # the kernel that moves the most bytes, against the copy bandwidth (when it is not the one above)
    roofline_stream = None
    hbm_k = [k for k in stages if kernel_algo(cfg, k)[0] == "hbm" and kernel_algo(cfg, k)[1] > 0]
    if hbm_k:
        sk = max(hbm_k, key=lambda k: kernel_algo(cfg, k)[1])
        if sk != dom:
            s_algo = kernel_algo(cfg, sk)[1]
            s_ach = s_algo / (stages[sk]["us_avg"] * 1e-6) / 1e9
            roofline_stream = {"kernel": sk, "bound": "hbm", "achieved": round(s_ach, 1), "peak": peaks["hbm_gbs"],
                               "unit": "GB/s", "frac": round(s_ach / peaks["hbm_gbs"], 4),
                               "traffic": traffic_from_profiles(sk, cfg.name, KERNEL_FILES.get(sk, [])),
                               "algorithmic_bytes_per_launch": s_algo,
                               "us_per_launch": round(stages[sk]["us_avg"], 3)}
    path_ach = per_step / (us_per_call * 1e-6) / 1e9
    hbm = peaks["hbm_gbs"]
    path_roofline = {"bound": "hbm", "bytes_per_call": per_step, "achieved": round(path_ach, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(path_ach / hbm, 4),
                     "ideal_us": round(per_step / (hbm * 1e9) * 1e6, 3)}
    uniq_bytes = per_step - hb["W_rows"] + uniq * cfg.d * e_sz
    path_roofline["unique_w_rows"] = uniq
    path_roofline["bytes_per_call_unique_rows"] = uniq_bytes
    path_roofline["frac_unique_rows"] = round(uniq_bytes / (us_per_call * 1e-6) / 1e9 / hbm, 4)

    # end to end through the public API with host buffers
    e2e = None
    if not a.no_e2e:
        n_e2e = min(a.steps, 2000 if cfg.B <= 64 else 100)
        hosts = [x["h"].cpu().pin_memory() for x in sets]
        # the three outputs live in one device buffer (idx, logits, probs as int32 / fp32 views),
        # so one device-to-host copy returns a step's results
        BK = cfg.B * cfg.K
        packed = [torch.empty(3 * BK, dtype=torch.int32, device=dev) for _ in sets]
        outs = [torch.empty(3 * BK, dtype=torch.int32).pin_memory() for _ in sets]
        views = [(p[:BK].view(cfg.B, cfg.K), p[BK:2 * BK].view(torch.float32).view(cfg.B, cfg.K),
                  p[2 * BK:].view(torch.float32).view(cfg.B, cfg.K)) for p in packed]
        def e2e_step(i):
            j = i % copies
            x = sets[j]
            idx, logits, probs = views[j]
            with torch.cuda.stream(stream):
                x["h"].copy_(hosts[j], non_blocking=True)
                step(x, idx, logits, probs)
                outs[j].copy_(packed[j], non_blocking=True)
            stream.synchronize()
        for i in range(3):
            e2e_step(i)
        barrier(world)
        te0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        te = max_over_ranks(time.perf_counter() - te0, world)
        e2e = {"value": round(cfg.B * n_e2e * world / te, 2), "unit": "rows/s",
               "us_per_call": round(te * 1e6 / n_e2e, 2), "steps": n_e2e,
               "h2d_bytes_per_step": int(cfg.B * cfg.d * (2 if cfg.dtype == "bf16" else 4)),
               "d2h_bytes_per_step": int(cfg.B * cfg.K * 12)}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_head_baseline(cfg, sets[0], a.cpu_seconds)
    clocks = sampler.summary(t0, t1)
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "rows/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms / a.steps, 6),
        "us_per_call": round(us_per_call, 3), "timing_spread": spread, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded generators, random weights)",
        "config": {"workload": cfg.name, "B": cfg.B, "d": cfg.d, "vocab": cfg.vocab, "r": cfg.r,
                   "K": cfg.K, "seed": a.seed, "api": "dh_draft_head" if a.api == "head" else
                   "dh_lowrank_topk + dh_exact_rescore", "graph": f"CUDA graphs of {S} steps",
                   "l2": f"inputs rotate over {copies} independent copies "
                         f"({copies * per_step / 2**20:.0f} MiB per cycle > 2x L2)",
                   "parallelism": f"replicas x{world} (rows independent)"},
        "roofline": roofline, "roofline_stream": roofline_stream, "path_roofline": path_roofline, "stages": stages,
        "gpu_launches": int(round(launches_per_step * a.steps)), "e2e": e2e,
        "cpu_baseline": cpu, "clocks": clocks,
    }


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
    return {"value": round(rows_done / dt, 4), "unit": "rows/s", "cores": used, "kind": "oracle",
            "sample": f"{rows_done} rows of the {cfg.name} workload ({what}), {dt:.1f} s, OpenMP over rows"}


# ------------------------------------------------------------------------------------- tree

def run_tree_bench(a, tcfg, rank, world, local, peaks, peak_src):
    from speculative_decoding_draft_dh_gb300 import binding as dh
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    t = inputs.make_tree(tcfg, seed=a.seed + 1000 * rank, device=dev)
    ws = dh.Workspace()
    stream = torch.cuda.Stream(device=dev)
    B, N, vocab = tcfg.B, tcfg.N, tcfg.vocab
    elem = 2 if tcfg.dtype == "bf16" else 4
    logit_bytes = B * N * vocab * elem

    def step():
        return dh.tree_accept(t["logits"], t["parent"], t["token"], workspace=ws)

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
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
        for _ in range(a.steps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    time.sleep(0.12)
    sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    us = ms * 1e3 / a.steps
    value = weak_scaling_value(B, a.steps, world, ms)
    n_prof = min(a.steps, 50)
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
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": traffic_from_profiles(dom, tcfg.name, KERNEL_FILES[dom]),
                "algorithmic_bytes_per_launch": logit_bytes,
                "us_per_launch": round(stages[dom]["us_avg"], 3),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"}
    e2e = None
    if not a.no_e2e:
        n_e2e = min(a.steps, 10)
        host = {k: t[k].cpu().pin_memory() for k in ("logits", "parent", "token")}
        outs = {k: None for k in ("path", "len", "bonus")}
        def e2e_step():
            with torch.cuda.stream(stream):
                for k in host:
                    t[k].copy_(host[k], non_blocking=True)
                o = step()
                res = [o[k].to("cpu", non_blocking=True) for k in ("path", "len", "bonus")]
            stream.synchronize()
            return res
        e2e_step()
        te0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        te = max_over_ranks(time.perf_counter() - te0, world)
        e2e = {"value": round(B * n_e2e * world / te, 2), "unit": "requests/s",
               "us_per_call": round(te * 1e6 / n_e2e, 1), "steps": n_e2e,
               "h2d_bytes_per_step": int(logit_bytes + 2 * B * N * 4),
               "d2h_bytes_per_step": int(B * N * 4 + 2 * B * 4)}
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_tree_baseline(tcfg, t, a.cpu_seconds)
    return {
        "metric": TREE_METRIC, "value": round(value, 2), "unit": "requests/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms / a.steps, 6),
        "us_per_call": round(us, 3), "node_rows_per_s": round(value * N, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": tcfg.dtype,
        "data": "synthetic (seeded generators)",
        "config": {"workload": tcfg.name, "B": B, "N": N, "vocab": vocab, "seed": a.seed,
                   "graph": "one CUDA graph per step",
                   "l2": f"logits {logit_bytes / 2**30:.2f} GiB per step > L2",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline, "stages": stages,
        "gpu_launches": int(round(sum(v[1] for v in prof.values()) / n_prof * a.steps)),
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
    return {"value": round(done / dt, 3), "unit": "requests/s", "cores": n, "kind": "oracle",
            "sample": f"{done} requests (first {n} of the tree workload, repeated), {dt:.1f} s"}


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
    if a.workload == "tree":
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
                             "sample": sample},
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
    else:
        cfg = inputs.HEAD_CONFIGS[a.workload]
        x = inputs.make_head(cfg, seed=a.seed, device=dev)
        for _ in range(a.warmup + a.steps):
            if a.api == "head":
                dh.draft_head(x["h"], x["U"], x["V"], x["W"], cfg.K)
            else:
                idx, _ = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
                dh.exact_rescore(x["h"], x["W"], idx)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": a.workload, "steps": a.warmup + a.steps}), flush=True)


def main():
    a = parse_args()
    if a.profile_run:
        from speculative_decoding_draft_dh_gb300 import build
        build.build()
        profile_run(a)
        return
    rank, world, local = dist_env()
    if a.impl == "reference":
        line = run_reference(a, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dist_init(world, local)
    from speculative_decoding_draft_dh_gb300 import build
    if rank == 0:
        build.build()
    barrier(world)
    build.build()
    peaks, src = load_peaks()
    if a.workload == "tree":
        line = run_tree_bench(a, inputs.TREE_CONFIGS["tree"], rank, world, local, peaks, src)
    else:
        line = run_head_bench(a, inputs.HEAD_CONFIGS[a.workload], rank, world, local, peaks, src)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
