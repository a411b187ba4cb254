#!/usr/bin/env python
"""Benchmark of the batched multi-adapter LoRA branch on GB300.

Workload (default): the Llama-3-8B packed QKV projection at decode, T=256 tokens
(one per request), k=4096, output slices 4096/1024/1024, 32 resident adapters
with ranks drawn from {8, 16, 32, 64}, Zipf(1.1) slot popularity, alpha = 2r.
All inputs are seeded and synthetic (workloads.config(2)).

A step is one pass of the whole hot path over one batch: re-upload one slot
table (what a slot change costs), build the token index, then run the branch on
the QKV projection of each of ``--layers`` (32) layers, each with its own
adapter weights, x and y buffers, so the working set (about 1.3 GB) is far
larger than the 129 MB L2 and every call streams from HBM.  The step is
captured once in a CUDA graph and replayed; CUDA events on the launching stream
time exactly K replays after W warm-up replays.

Metric: LoRA-branch tokens/s (tokens through one projection call per second:
T * layers / step time) and achieved HBM GB/s of the algorithmic bytes of each
call against the measured copy bandwidth.  One JSON line on rank 0.

``--impl reference`` times the CPU oracle (plain C, fp64) on the host cores
instead, on the same workload; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
CONFIG_INDEX = {name: i for i, name in enumerate(W.CONFIG_NAMES)}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="decode_qkv", choices=list(CONFIG_INDEX) + ["decode_moe"])
    p.add_argument("--layers", type=int, default=32)
    p.add_argument("--requests", type=int, default=16, help="prefill_mlp only: requests in the batch")
    p.add_argument("--path", default="best", choices=["best", "auto", "decode_fused", "decode_split", "prefill",
                                                        "decode_direct", "decode_direct_fp8", "decode_tma",
                                                        "decode_cluster"],
                   help="best: the library's fastest measured path for the workload (default_path); auto: "
                        "LORA_PATH_AUTO (decode_direct_fp8 for a workload with FP8 adapters); decode_moe takes "
                        "decode_direct or decode_tma (best: decode_direct)")
    p.add_argument("--configs", default="all",
                   help="after the headline, one record per other workload: 'all', 'none' or a comma list of "
                        + ", ".join(SUB_CONFIGS))
    p.add_argument("--config-seconds", type=float, default=0.3, help="timed region of each per-workload record")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-chunks", type=int, default=8,
                   help="e2e: chunks of layers whose copies overlap the compute of the previous chunk")
    p.add_argument("--no-plan", action="store_true",
                   help="warp-streaming paths: rebuild the tables in every call instead of per-step plans")
    p.add_argument("--with-base", default="none", choices=["none", "serial", "overlap"],
                   help="time the base projection y = x W0^T (bf16 library GEMM) with the branch: one after the "
                        "other on one stream, or the branch on an aux stream overlapping the GEMM")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the CPU-baseline sample")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# Accounting (measurement, not the method): bytes and flops a call must move
# ---------------------------------------------------------------------------
def algorithmic_bytes(slot_ids, ranks, k, widths, wbytes: int = 2) -> int:
    """Each active slot's A and B once (wbytes per weight: 2 for bf16, 1 for
    e4m3), x rows of LoRA tokens once, their y rows read and written (bf16).
    Workspace, index and no-adapter rows excluded."""
    S, n, d = len(ranks), len(widths), int(sum(widths))
    ids = np.asarray(slot_ids)
    valid = (ids >= 0) & (ids < S)
    lora = np.zeros(len(ids), dtype=bool)
    lora[valid] = np.asarray(ranks)[ids[valid]] > 0
    n_l = int(lora.sum())
    weights = sum(wbytes * int(ranks[s]) * (n * k + d) for s in np.unique(ids[lora]))
    return int(weights + 2 * k * n_l + 4 * d * n_l)


def algorithmic_flops(slot_ids, ranks, k, widths) -> int:
    S, n, d = len(ranks), len(widths), int(sum(widths))
    return int(sum(2 * int(ranks[s]) * (n * k + d) for s in slot_ids if 0 <= s < S and ranks[s] > 0))


def captured_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None when
    the kernel's sources changed since the capture (the counters no longer apply)."""
    import hashlib
    here = os.path.dirname(os.path.abspath(__file__))
    try:
        with open(os.path.join(here, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    m = hashlib.sha256()
    for name in rec["sources"]:
        with open(os.path.join(here, "rank_adapter_gemm_gb300", "csrc", name), "rb") as f:
            m.update(f.read())
    if m.hexdigest()[:16] != rec["source_sha256_16"]:
        return None
    return rec["dram_read_bytes"] + rec["dram_write_bytes"]


# Kernels of one lora_apply call whose DRAM traffic was captured with ncu on the
# bench workload (per call: the sum over the call's launches).
TRAFFIC_KERNELS = {
    ("decode_qkv", "decode_fused"): ("fused_decode_kernel",),
    ("decode_qkv", "decode_direct"): ("direct_shrink_kernel", "direct_expand_kernel"),
    ("decode_qkv", "decode_tma"): ("tma_decode_kernel",),
}


def call_traffic(config: str, path: str):
    names = TRAFFIC_KERNELS.get((config, path))
    if not names:
        return None
    parts = [captured_traffic(k) for k in names]
    return None if any(p is None for p in parts) else sum(parts)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas: each rank runs the same workload on its GPU)
# ---------------------------------------------------------------------------
def dist_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_info()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29511")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over ranks (the slowest replica sets the job's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, elapsed_per_rank: float, world: int, device=None) -> float:
    """Whole-job rate: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / max_over_ranks(elapsed_per_rank, device)


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        def flag(v):
            return v.lower() in ("active", "1", "yes", "true") or v.startswith("0x") and int(v, 16) != 0

        window = [s for (t, s) in self.samples if t0 <= t <= t1 and len(s) >= 9]
        if not window:  # the timed region was shorter than the sampling period: nearest samples
            window = sorted((abs(t - (t0 + t1) / 2), s) for (t, s) in self.samples if len(s) >= 9)[:3]
            window = [s for _, s in window]
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(s[1]) for s in window if s[1].replace(".", "").isdigit()]
        smax = [float(s[2]) for s in window if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for s in window for j in range(4) if flag(s[5 + j])})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(window)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def _workload(name, n_requests=16):
    if name == "decode_moe":
        return W.moe_config()
    idx = CONFIG_INDEX[name]
    return W.config(idx, y_init="normal", n_requests=n_requests)


HEADLINE = "LoRA-branch tokens/sec and achieved HBM GB/s (% of peak), Llama-3-8B QKV decode"


def workload_name(config, wl):
    """The `config.workload` string both arms print."""
    if config == "decode_qkv":
        return ("decode packed QKV, Llama-3-8B shapes: T=256, k=4096, slices 4096/1024/1024, S=32, "
                "r in {8,16,32,64} (r_max 64), Zipf(1.1) slot popularity, alpha=2r")
    return wl.description


def metric_name(config):
    return HEADLINE if config == "decode_qkv" else \
        f"LoRA-branch tokens/sec and achieved HBM GB/s (% of peak), {config}"


def _index_ids(wl):
    """Slot ids the step uploads: one per token, or one per sequence of
    tokens_per_seq tokens (speculative decode, sequence-major)."""
    return np.ascontiguousarray(wl.slot_ids[::wl.tokens_per_seq])


def _build_index(index, slot_dev, table, tokens_per_seq):
    if tokens_per_seq > 1:
        index.build_seq(slot_dev, tokens_per_seq, table)
    else:
        index.build(slot_dev, table)


def time_steps(args, dev, local, index_part, apply_part):
    """Capture a step's two parts (the per-step index, then the calls) in CUDA
    graphs, warm up, and time ``args.steps`` replays with CUDA events on the
    launching stream, sampling the SM clocks meanwhile.  Returns (elapsed s,
    mean ms of the calls part, mean ms of the rest, clocks, peaks)."""
    import torch
    stream = torch.cuda.Stream(device=dev)
    # eager warm-up (sets kernel attributes), then capture the two parts of a step
    with torch.cuda.stream(stream):
        index_part()
        apply_part()
    torch.cuda.synchronize()
    g_index, g_apply = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_index, stream=stream):
        index_part()
    with torch.cuda.graph(g_apply, stream=stream):
        apply_part()
    torch.cuda.synchronize()

    def replay(events=None):
        g_index.replay()
        if events is not None:
            events[0].record()
        g_apply.replay()
        if events is not None:
            events[1].record()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            replay()
    torch.cuda.synchronize()

    peaks = measured_peaks()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    with torch.cuda.stream(stream):
        t_start.record()
        for k in range(args.steps):
            replay(marks[k])
        t_end.record()
    torch.cuda.synchronize()
    w1 = time.time()
    barrier()
    time.sleep(0.1)
    sampler.stop()
    elapsed_s = t_start.elapsed_time(t_end) / 1e3
    apply_ms = [a.elapsed_time(b) for a, b in marks]          # the calls of every step
    apply_ms_mean = float(np.mean(apply_ms))
    index_ms_mean = (elapsed_s * 1e3 - float(np.sum(apply_ms))) / args.steps
    return elapsed_s, apply_ms_mean, index_ms_mean, sampler.summary(w0, w1), peaks


class ProjectionBench:
    """One workload of packed projections on the device for timing: layer l runs
    projection l % len(modules) in its own buffers (weights, x, y, slot table),
    one token index per step, per-step plans where the path has them."""

    def __init__(self, wl, n_layers, path, dev, no_plan=False, with_base="none"):
        import torch
        import rank_adapter_gemm_gb300 as L
        from rank_adapter_gemm_gb300.resident import ResidentProjection
        self.L, self.wl, self.dev, self.with_base = L, wl, dev, with_base
        self.wbytes = 1 if wl.weights == "e4m3" else 2
        self.mods = list(range(len(wl.modules)))
        n_layers = max(len(self.mods), n_layers // len(self.mods) * len(self.mods))
        base = [ResidentProjection.from_workload(wl, m, device=dev) for m in self.mods]
        self.layers = [base[l % len(base)] if l < len(base) else base[l % len(base)].clone(device=dev)
                       for l in range(n_layers)]
        self.T, self.S = wl.T, wl.S
        counts = np.bincount(wl.slot_ids[wl.slot_ids >= 0], minlength=self.S)
        self.max_seg = int(counts.max()) if counts.size else 0
        self.slot_dev = torch.from_numpy(_index_ids(wl)).to(dev)
        self.index = L.TokenIndex(self.T, self.S, device=dev)
        self.ws = [L.Workspace(self.T, lay.shape, device=dev) for lay in self.layers[:len(base)]]
        self.ws_of = [self.ws[l % len(self.ws)].buf for l in range(len(self.layers))]
        self.w0 = []
        if with_base != "none":
            g = torch.Generator(device=dev).manual_seed(1234)
            for lay in self.layers:
                d = int(lay.y.shape[1])
                self.w0.append((torch.randn(d, lay.x.shape[1], device=dev, generator=g) * 0.02).to(torch.bfloat16))
        self.aux = torch.cuda.Stream(device=dev)
        self.path = path
        self.resolved, self.launches_per_apply = L.lora_resolve_path(path, self.T, self.max_seg)
        self.use_plan = (not no_plan and with_base == "none" and
                         self.resolved in ("decode_direct", "decode_direct_fp8", "decode_tma"))
        if self.use_plan and self.resolved == "decode_tma":
            self.launches_per_apply = 1  # the plan replaces the per-call plan launch
        self.plans = ([L.Plan(self.T, lay.shape, self.resolved, device=dev) for lay in self.layers]
                      if self.use_plan else [])
        m = wl.modules
        self.bytes_per_call = [algorithmic_bytes(wl.slot_ids, wl.ranks, m[j].k, m[j].slice_widths, self.wbytes)
                               for j in self.mods]
        self.flops_per_call = [algorithmic_flops(wl.slot_ids, wl.ranks, m[j].k, m[j].slice_widths) for j in self.mods]
        if with_base != "none":  # the base GEMM's W0, x and y bytes too
            self.bytes_per_call = [b + 2 * m[j].k * sum(m[j].slice_widths) + 2 * self.T * (m[j].k + sum(m[j].slice_widths))
                                   for b, j in zip(self.bytes_per_call, self.mods)]

    def apply_layer(self, l):
        L, lay, torch = self.L, self.layers[l], __import__("torch")
        if self.use_plan:
            self.plans[l].apply(lay.x, lay.y, self.ws[l % len(self.ws)], self.index.err)
            return
        if self.with_base == "overlap":
            L.apply_with_base(lay.x, self.w0[l], lay.y, lay.shape, lay.table.dev, self.index, self.ws_of[l], self.aux,
                              max_seg_hint=self.max_seg, path=self.path)
            return
        if self.with_base == "serial":
            torch.matmul(lay.x, self.w0[l].t(), out=lay.y)
        L.lora_apply(lay.x, lay.y, lay.shape, lay.table.dev, self.index.sorted_ids, self.index.seg_offsets,
                     self.index.active, self.ws_of[l], self.index.err, max_seg_hint=self.max_seg, path=self.path)

    def index_part(self):
        L = self.L
        self.layers[0].refresh_table()
        _build_index(self.index, self.slot_dev, self.layers[0].table, self.wl.tokens_per_seq)
        if self.use_plan:  # one launch per shape: a plan per layer, each with its layer's weight pointers
            n = len(self.mods)
            for m in self.mods:
                L.lora_build_plans(self.plans[m::n], [lay.table for lay in self.layers[m::n]], self.index)

    def apply_part(self):
        for l in range(len(self.layers)):
            self.apply_layer(l)

    def per_layer(self, values):
        return [values[l % len(self.mods)] for l in range(len(self.layers))]


def default_path(wl):
    """The library's fastest measured path for a workload: the one-kernel TMA
    decode path on per-step plans for bf16 decode batches, AUTO's one cluster per
    slot for batches of 64 tokens and fewer, the FP8 variant of the warp-streaming
    kernels for FP8 adapters, the tensor-core prefill kernels for long segments."""
    if wl.weights == "e4m3":
        return "decode_direct_fp8"
    counts = np.bincount(wl.slot_ids[wl.slot_ids >= 0], minlength=wl.S)
    if counts.size and int(counts.max()) > 256:
        return "auto"  # prefill
    if wl.T <= 64:
        return "auto"  # the one-cluster-per-slot kernel (LORA_PATH_DECODE_CLUSTER)
    ok = all(wl.r_max <= 64 and len(m.slice_widths) * wl.r_max <= 192 and m.k % 64 == 0 for m in wl.modules)
    return "decode_tma" if ok else "auto"


def run_ours(args):
    import torch
    import rank_adapter_gemm_gb300 as L

    rank, world = dist_init("nccl")
    _, _, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    wl = _workload(args.config, args.requests)
    if args.path == "best":
        args.path = default_path(wl)
    if wl.weights == "e4m3":
        if args.path == "auto":
            args.path = "decode_direct_fp8"
        if args.path != "decode_direct_fp8":
            raise SystemExit(f"{args.config} holds FP8 adapters: only --path decode_direct_fp8 serves it")
    pb = ProjectionBench(wl, args.layers, args.path, dev, no_plan=args.no_plan, with_base=args.with_base)
    T, mods, layers = pb.T, pb.mods, pb.layers

    elapsed_s, apply_ms_mean, index_ms_mean, clocks, (peak_gbs, peak_tf, peak_src) = \
        time_steps(args, dev, local, pb.index_part, pb.apply_part)
    err = int(pb.index.err.item())

    units = T * len(layers) * args.steps
    value = job_throughput(units, elapsed_s, world, dev)
    ms_per_step = max_over_ranks(elapsed_s, dev) / args.steps * 1e3
    per_layer_bytes = pb.per_layer(pb.bytes_per_call)
    per_layer_flops = pb.per_layer(pb.flops_per_call)
    call_s = apply_ms_mean / 1e3 / len(layers)
    achieved_gbs = sum(per_layer_bytes) / len(layers) / call_s / 1e9
    resolved = pb.resolved
    gpu_launches = args.steps * (1 + len(layers) * pb.launches_per_apply + (len(mods) if pb.use_plan else 0))

    e2e = None
    if not args.no_e2e and args.with_base == "none":
        e2e = run_e2e(args, wl, layers, pb.index, pb.slot_dev, pb.ws_of, pb.max_seg, dev, world, pb.plans, mods,
                      pb.ws)

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    configs = None
    if args.configs != "none" and rank == 0 and world == 1:
        del pb  # free the headline's buffers before the other workloads
        torch.cuda.empty_cache()
        configs = config_records(args, dev, local, peak_gbs)

    out = {
        "metric": metric_name(args.config),
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 (adapters; x rounded to e4m3, y bf16)" if wl.weights == "e4m3" else "bf16",
        "data": "synthetic (seeded: workloads.config)",
        "config": {
            "workload": workload_name(args.config, wl),
            "config": args.config,
            "value_definition": "tokens through one projection call per second: T x calls per step / step time "
                                "(one call = the branch of one packed projection of one layer)",
            "layers_per_step": len(layers),
            "calls_per_step": len(layers),
            "path": resolved + (" with per-step plans" if pb_use_plan(resolved, args) else ""),
            "l2": f"inputs larger than L2: {len(layers)} distinct layer buffer sets, "
                  f"{sum(per_layer_bytes) / 1e9:.2f} GB of algorithmic bytes per step",
            "parallelism": f"replicas x{world}",
            **({"base": "bf16 library GEMM y = x W0^T, then the branch on the same stream"
                if args.with_base == "serial" else
                "bf16 library GEMM y = x W0^T, the branch on an aux stream: its shrink overlaps the GEMM"}
               if args.with_base != "none" else {}),
        },
        "gbs": achieved_gbs,
        "roofline": {
            "bound": "hbm",
            "achieved": achieved_gbs,
            "peak": peak_gbs,
            "unit": "GB/s",
            "frac": achieved_gbs / peak_gbs,
            "traffic": call_traffic(args.config, resolved),
            "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
            "kernel": ("lora_apply (shrink + expand) per projection call" if args.with_base == "none" else
                       "base GEMM + lora_apply per projection call"),
            "bytes_per_call": sum(per_layer_bytes) / len(layers),
            "flops_per_call": sum(per_layer_flops) / len(layers),
            "us_per_call": call_s * 1e6,
            "index_and_table_us": index_ms_mean * 1e3,
            "frac_of_8000": achieved_gbs / 8000.0,
        },
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "device_error": err,
    }
    if e2e is not None:
        out["e2e"] = e2e
    if cpu is not None:
        out["cpu_baseline"] = cpu
    if configs is not None:
        out["configs"] = configs
    return out, rank


def pb_use_plan(resolved, args):
    return not args.no_plan and args.with_base == "none" and resolved in ("decode_direct", "decode_direct_fp8",
                                                                          "decode_tma")


def run_e2e(args, wl, layers, index, slot_dev, ws_of, max_seg, dev, world, plans=(), mods=(0,), ws=()):
    """Same metric with host buffers: every step copies the slot ids and every
    layer's x and y from pinned host memory, runs the step, and reads every y
    back.  The layers of one shape keep their rows in one device buffer (a view
    per layer); a step moves them in chunks of layers (--e2e-chunks) per shape and
    direction, the inputs of a chunk on one copy stream and its results on
    another while the next chunk computes (events order them inside the graph)."""
    import torch
    import rank_adapter_gemm_gb300 as L
    T = wl.T
    h_slots = torch.from_numpy(_index_ids(wl)).pin_memory()
    groups = [list(range(m, len(layers), len(mods))) for m in mods]
    d_x = [torch.stack([layers[l].x for l in g]) for g in groups]      # [layers of the shape, T, k]
    d_y = [torch.stack([layers[l].y for l in g]) for g in groups]
    h_x = [t.cpu().pin_memory() for t in d_x]
    h_y = [t.cpu().pin_memory() for t in d_y]
    h_out = [torch.empty_like(t).pin_memory() for t in h_y]
    xv, yv = {}, {}
    for gi, g in enumerate(groups):
        for j, l in enumerate(g):
            xv[l], yv[l] = d_x[gi][j], d_y[gi][j]
    stream = torch.cuda.Stream(device=dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    n_chunks = max(1, min(args.e2e_chunks, min(len(g) for g in groups)))  # copies of c+1 / c-1 overlap chunk c
    parts = [[np.array_split(np.arange(len(g)), n_chunks)[c] for g in groups] for c in range(n_chunks)]

    def rows(t, j):
        return t[int(j[0]):int(j[-1]) + 1]

    def step():
        cur = torch.cuda.current_stream()
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        ev_in = []
        with torch.cuda.stream(s_in):
            slot_dev.copy_(h_slots, non_blocking=True)
            ev_slots = torch.cuda.Event()
            ev_slots.record(s_in)
            for c in range(n_chunks):
                for gi in range(len(groups)):
                    j = parts[c][gi]
                    if len(j):
                        rows(d_x[gi], j).copy_(rows(h_x[gi], j), non_blocking=True)
                        rows(d_y[gi], j).copy_(rows(h_y[gi], j), non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                ev_in.append(ev)
        cur.wait_event(ev_slots)
        _build_index(index, slot_dev, layers[0].table, wl.tokens_per_seq)
        if plans:
            for m in mods:
                L.lora_build_plans(plans[m::len(mods)], [lay.table for lay in layers[m::len(mods)]], index)
        for c in range(n_chunks):
            cur.wait_event(ev_in[c])
            for gi, g in enumerate(groups):
                for jj in parts[c][gi]:
                    l = g[int(jj)]
                    lay = layers[l]
                    if plans:
                        plans[l].apply(xv[l], yv[l], ws[l % len(ws)], index.err)
                    else:
                        L.lora_apply(xv[l], yv[l], lay.shape, lay.table.dev, index.sorted_ids, index.seg_offsets,
                                     index.active, ws_of[l], index.err, max_seg_hint=max_seg, path=args.path)
            ev = torch.cuda.Event()
            ev.record(cur)
            s_out.wait_event(ev)
            with torch.cuda.stream(s_out):
                for gi in range(len(groups)):
                    j = parts[c][gi]
                    if len(j):
                        rows(h_out[gi], j).copy_(rows(d_y[gi], j), non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(steps):
            graph.replay()
        e1.record()
    torch.cuda.synchronize()
    elapsed = e0.elapsed_time(e1) / 1e3
    value = job_throughput(T * len(layers) * steps, elapsed, world, dev)
    h2d = h_slots.numel() * 4 + sum(h.numel() * 2 for h in h_x) + sum(h.numel() * 2 for h in h_y)
    d2h = sum(h.numel() * 2 for h in h_out)
    return {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def moe_algorithmic_bytes(wl, m) -> int:
    """Routed-expert call: each (adapter, expert) pair in use reads its A and B
    once (bf16), the x rows in use once (per token or per pair), and the y rows
    of the pairs with an adapter are read and written (bf16)."""
    mod = wl.modules[m]
    n, k, d = len(mod.slice_widths), mod.k, mod.d
    s = np.repeat(wl.slot_ids, wl.K)
    e = wl.expert_ids.reshape(-1)
    lora = s >= 0
    lora[lora] = wl.ranks[s[lora]] > 0
    used = np.unique(s[lora] * wl.E + e[lora])
    weights = sum(2 * int(wl.ranks[v // wl.E]) * (n * k + d) for v in used)
    x_rows = int(lora.reshape(wl.T, wl.K).any(axis=1).sum()) if mod.x_per_token else int(lora.sum())
    return int(weights + 2 * k * x_rows + 4 * d * int(lora.sum()))


class MoeBench:
    """The routed-expert workload on the device: layer l runs module l % 2 (w1
    with x per token, w2 with x per pair) in its own buffers; one pair index per
    step, per-step plans unless no_plan."""

    def __init__(self, wl, n_layers, dev, no_plan=False, path=None):
        import torch
        import rank_adapter_gemm_gb300 as L
        from rank_adapter_gemm_gb300.resident import ResidentMoeProjection, clone_moe
        self.L, self.wl = L, wl
        self.mods = list(range(len(wl.modules)))
        base = [ResidentMoeProjection(wl, m, device=dev) for m in self.mods]
        self.layers = [base[l % len(base)] if l < len(base) else clone_moe(base[l % len(base)], device=dev)
                       for l in range(max(n_layers, len(base)))]
        P, V = wl.T * wl.K, wl.n_adapters * wl.E
        self.index = L.TokenIndex(P, V, device=dev)
        self.slot_dev = torch.from_numpy(wl.slot_ids).to(dev)
        self.expert_dev = torch.from_numpy(wl.expert_ids.reshape(-1).copy()).to(dev)
        self.ws = [L.Workspace(P, b.shape, device=dev) for b in base]
        if path is None:
            # measured on GB300 (Mixtral expert shapes, 32 interleaved w1/w2 calls): both paths take
            # about 24.3 us per call, and the TMA plans cost 17 us more per step
            path = "decode_direct"
        self.path = path
        self.plans = ([] if no_plan or path == "decode_cluster"  # the cluster kernel has no plan
                      else [L.Plan(P, lay.shape, path=path, device=dev) for lay in self.layers])
        self.bytes_per_call = [moe_algorithmic_bytes(wl, m) for m in self.mods]

    def index_part(self):
        L, n, wl = self.L, len(self.mods), self.wl
        self.index.build_moe(self.slot_dev, self.expert_dev, wl.K, wl.E, self.layers[0].table)
        if self.plans:  # one launch per module shape
            for m in self.mods:
                L.lora_build_plans(self.plans[m::n], [lay.table for lay in self.layers[m::n]], self.index)

    def apply_part(self):
        L, wl = self.L, self.wl
        for l, lay in enumerate(self.layers):
            L.lora_apply_moe(lay.x, lay.y, wl.K, lay.shape, lay.table.dev, self.index.sorted_ids,
                             self.index.seg_offsets, self.index.active, self.ws[l % len(self.ws)].buf, self.index.err,
                             x_per_token=lay.x_per_token, plan=self.plans[l] if self.plans else None, path=self.path)


def run_moe(args):
    """The routed-expert workload as the headline line."""
    import torch

    rank, world = dist_init("nccl")
    _, _, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.moe_config()
    mb = MoeBench(wl, args.layers, dev, no_plan=args.no_plan,
                  path=args.path if args.path in ("decode_direct", "decode_tma", "decode_cluster") else None)
    elapsed_s, apply_ms_mean, index_ms_mean, clocks, (peak_gbs, peak_tf, peak_src) = \
        time_steps(args, dev, local, mb.index_part, mb.apply_part)
    err = int(mb.index.err.item())
    layers = mb.layers
    units = wl.T * len(layers) * args.steps
    value = job_throughput(units, elapsed_s, world, dev)
    ms_per_step = max_over_ranks(elapsed_s, dev) / args.steps * 1e3
    per_layer_bytes = [mb.bytes_per_call[l % len(mb.mods)] for l in range(len(layers))]
    call_s = apply_ms_mean / 1e3 / len(layers)
    achieved_gbs = sum(per_layer_bytes) / len(layers) / call_s / 1e9
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(wl, args.cpu_seconds)
    out = {
        "metric": metric_name(args.config),
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded: workloads.moe_config)",
        "config": {
            "workload": workload_name(args.config, wl),
            "config": args.config,
            "layers_per_step": len(layers),
            "calls_per_step": len(layers),
            "path": f"lora_apply_moe on {mb.path} over n_adapters * E virtual slots"
                    + (" with per-step plans" if mb.plans else ""),
            "l2": f"inputs larger than L2: {len(layers)} distinct layer buffer sets, "
                  f"{sum(per_layer_bytes) / 1e9:.2f} GB of algorithmic bytes per step",
            "parallelism": f"replicas x{world}",
        },
        "gbs": achieved_gbs,
        "roofline": {
            "bound": "hbm",
            "achieved": achieved_gbs,
            "peak": peak_gbs,
            "unit": "GB/s",
            "frac": achieved_gbs / peak_gbs,
            "traffic": None,
            "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
            "kernel": "lora_apply_moe (shrink + expand) per expert-projection call",
            "bytes_per_call": sum(per_layer_bytes) / len(layers),
            "us_per_call": call_s * 1e6,
            "index_and_table_us": index_ms_mean * 1e3,
        },
        "gpu_launches": args.steps * (1 + 2 * len(layers) + (len(mb.mods) if mb.plans else 0)),
        "clocks": clocks,
        "device_error": err,
    }
    if cpu is not None:
        out["cpu_baseline"] = cpu
    return out, rank


# ---------------------------------------------------------------------------
# One record per other workload, in the same run
# ---------------------------------------------------------------------------
SUB_CONFIGS = {
    "decode_q_proj": {"index": 1},
    "large_decode": {"index": 4},
    "layer_sweep": {"index": 4, "sweep": True},
    "prefill_mlp": {"index": 3},
    "decode_qkv_spec": {"index": 5},
    "decode_qkv_fp8": {"index": 6},
    "decode_moe": {"moe": True},
}
L2_BYTES = 129e6


def _timed(dev, local, index_part, apply_part, seconds):
    """time_steps with about `seconds` of timed calls (a 3-step probe sizes it)."""
    import types
    probe = time_steps(types.SimpleNamespace(steps=3, warmup=3), dev, local, index_part, apply_part)
    per_step = max(probe[1], 1e-3) / 1e3
    steps = int(min(2000, max(5, seconds / per_step)))
    return time_steps(types.SimpleNamespace(steps=steps, warmup=3), dev, local, index_part, apply_part), steps


def config_records(args, dev, local, peak_gbs):
    """Per-call time, algorithmic bytes and roofline fraction of every other
    workload of the method (the driver's run sees all of them), each with the
    oracle's one-core and all-core rates on a bounded sample."""
    import torch
    names = list(SUB_CONFIGS) if args.configs == "all" else [c for c in args.configs.split(",") if c]
    out = {}
    for name in names:
        spec = SUB_CONFIGS[name]
        t0 = time.time()
        if spec.get("moe"):
            wl = W.moe_config()
            per_call = [moe_algorithmic_bytes(wl, m) for m in range(len(wl.modules))]
            n_layers = len(per_call) * max(1, int(np.ceil(4 * L2_BYTES / sum(per_call))))
            bench = MoeBench(wl, n_layers, dev)
            path = f"lora_apply_moe on {bench.path} with per-step plans"
            calls_per_step = len(bench.layers)
        else:
            wl = W.config(spec["index"], y_init="normal", sweep=spec.get("sweep", False))
            path = default_path(wl)
            wb = 1 if wl.weights == "e4m3" else 2
            per_call = [algorithmic_bytes(wl.slot_ids, wl.ranks, m.k, m.slice_widths, wb) for m in wl.modules]
            n_layers = len(per_call) * max(1, int(np.ceil(4 * L2_BYTES / sum(per_call))))
            bench = ProjectionBench(wl, n_layers, path, dev)
            path = bench.resolved + (" with per-step plans" if bench.use_plan else "")
            calls_per_step = len(bench.layers)
        (elapsed_s, apply_ms, index_ms, clocks, _), steps = _timed(dev, local, bench.index_part, bench.apply_part,
                                                                   args.config_seconds)
        err = int(bench.index.err.item())
        per_layer = [per_call[l % len(per_call)] for l in range(calls_per_step)]
        call_s = apply_ms / 1e3 / calls_per_step
        gbs = sum(per_layer) / calls_per_step / call_s / 1e9
        rec = {
            "workload": wl.description,
            "path": path,
            "calls_per_step": calls_per_step,
            "steps": steps,
            "us_per_call": call_s * 1e6,
            "bytes_per_call": sum(per_layer) / calls_per_step,
            "tokens_per_call": int(wl.T),
            "tokens_per_s": wl.T / call_s,
            "gbs": gbs,
            "frac": gbs / peak_gbs,
            "index_and_plans_us": index_ms * 1e3,
            "clocks": clocks,
            "device_error": err,
        }
        del bench
        torch.cuda.empty_cache()
        rec["oracle"] = oracle_rates(wl, seconds=2.0)
        rec["wall_s"] = round(time.time() - t0, 1)
        out[name] = rec
    return out


def _oracle_call(wl, rows):
    import oracle
    if isinstance(wl, W.MoeWorkload):  # rows are (token, choice) pairs of the first module
        m = wl.modules[0]
        scales = oracle.slot_scales(wl.ranks, wl.alphas, wl.scale_rule, False)
        t0 = time.perf_counter()
        oracle.apply_moe(m.x, m.x_per_token, m.y_in, m.slice_widths, wl.slot_ids, wl.expert_ids, wl.E, wl.ranks,
                         scales, m.A, m.B, rows=rows)
        return time.perf_counter() - t0
    m = wl.modules[0]
    fp8 = wl.weights == "e4m3"
    rule = oracle.slot_scales(wl.ranks, wl.alphas, wl.scale_rule, False)
    premul = oracle.premultiply_e4m3 if fp8 else oracle.premultiply
    if wl.premultiplied:
        B = [[(premul(b, rule[s]) if b is not None else None) for b in row] for s, row in enumerate(m.B)]
        scales = np.ones(wl.S)
    else:
        B, scales = m.B, rule
    t0 = time.perf_counter()
    if fp8:
        oracle.apply_e4m3(m.x, m.y_in, m.slice_widths, wl.slot_ids, wl.ranks, scales, m.A, B, rows=rows)
    else:
        oracle.apply(m.x, m.y_in, m.slice_widths, wl.slot_ids, wl.ranks, scales, m.A, B, rows=rows)
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_rows(wl):
    moe = isinstance(wl, W.MoeWorkload)  # rows are the T*K pairs, T tokens
    return np.arange(wl.T * wl.K if moe else wl.T, dtype=np.int32), (wl.K if moe else 1)


def oracle_rates(wl, seconds: float):
    """The oracle as it stands on the host: one thread, then every core (the
    sample's rows split into one chunk per core, run on a thread pool: the C
    oracle releases the GIL and keeps no state between calls), each the median
    of three timed passes over a bounded sample of the batch's rows."""
    import concurrent.futures as cf
    rows, per_tok = _oracle_rows(wl)
    cores = host_cores()
    probe = max(1, min(len(rows), 8))
    per_row = _oracle_call(wl, rows[:probe]) / probe
    n = int(max(min(len(rows), cores), min(len(rows), seconds / 6 / max(per_row, 1e-9))))
    sample = rows[:n]

    def one():
        return _oracle_call(wl, sample)

    chunks = [c for c in np.array_split(sample, cores) if len(c)]
    with cf.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        def many():
            t0 = time.perf_counter()
            list(ex.map(lambda c: _oracle_call(wl, c), chunks))
            return time.perf_counter() - t0
        t1 = statistics.median(one() for _ in range(3))
        tn = statistics.median(many() for _ in range(3))
    return {"one_core": n / per_tok / t1, "all_cores": n / per_tok / tn, "cores": len(chunks), "unit": "tokens/s",
            "sample": f"{n} of {len(rows)} rows of the first projection, median of 3 passes per leg"}


def cpu_baseline(wl, seconds: float):
    """The oracle as it stands on the host cores (oracle_rates): the all-core
    rate is the value, the one-core rate beside it."""
    r = oracle_rates(wl, seconds)
    return {"value": r["all_cores"], "unit": "tokens/s", "cores": r["cores"], "kind": "oracle",
            "one_core": r["one_core"],
            "sample": r["sample"] + f"; fp64 C oracle on {r['cores']} threads (one core: {r['one_core']:.0f} tokens/s)"}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return None, rank
    import concurrent.futures as cf
    wl = _workload(args.config, args.requests)
    rows, per_tok = _oracle_rows(wl)  # MoE rows are (token, choice) pairs
    cores = host_cores()
    for _ in range(max(args.warmup, 0)):
        _oracle_call(wl, rows[:max(1, len(rows) // 8)])
    # each step: the branch for one projection call over a bounded sample of rows,
    # the rows split over every host core (the C oracle releases the GIL)
    budget_s = 150.0
    per_row = _oracle_call(wl, rows[:8]) / 8
    n_rows = int(max(1, min(len(rows), cores * budget_s / max(args.steps, 1) / max(per_row, 1e-9))))
    sample = rows[:n_rows]
    chunks = [c for c in np.array_split(sample, cores) if len(c)]
    t = 0.0
    with cf.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        for _ in range(args.steps):
            t0 = time.perf_counter()
            list(ex.map(lambda c: _oracle_call(wl, c), chunks))
            t += time.perf_counter() - t0
    value = n_rows * args.steps / t / per_tok
    out = {
        "metric": metric_name(args.config),
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded: workloads.config)",
        "config": {"workload": workload_name(args.config, wl), "config": args.config},
        "impl": "reference",
        "cpu_baseline": {"kind": "oracle", "cores": len(chunks), "value": value,
                         "sample": f"{n_rows} of {len(rows)} rows ({'token-expert pairs' if per_tok > 1 else 'tokens'}) "
                                   f"of the first projection per step, split over {len(chunks)} threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return out, rank


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        out, rank = run_reference(args)
    else:
        out, rank = run_moe(args) if args.config == "decode_moe" else run_ours(args)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
