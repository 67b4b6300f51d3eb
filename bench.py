#!/usr/bin/env python3
"""Benchmark of the fused GQA decode-attention step on GB300.

One "step" is one pass of the whole hot path -- prologue (QK-norm + RoPE + cache append),
split-KV attention, log-sum-exp combine -- over one decode batch of synthetic, seeded
inputs already resident in HBM (for the 40-layer sweep: the 40 layers' calls).

Prints ONE JSON line.  `value` is microseconds per step (lower is better), K steps timed
as one CUDA graph replay with CUDA events; `roofline` reports the attention kernel's
KV-read bandwidth (algorithmic bytes sum_b L_b * H_kv * d * 2 * 2 per launch, times the
launches, over the timed region) against the measured HBM copy peak; `e2e` is the same
step through the host-buffer entry point with the per-step inputs copied in and the
output copied out inside the timed region; `cpu_baseline` is the fp64 oracle timed on
the host cores on a bounded sample.  The headline workload is the 40-layer sweep.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the step
has no cross-GPU exchange): weak scaling, max time over ranks.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "qwen3-14b-40layer"
# Steps of each by_config row's graph (whatever --steps is): enough that a short step's
# first launches, which have no preceding step to overlap, weigh little in the mean.
BY_CONFIG_STEPS = 200
METRIC = "GQA decode-attn µs/step and KV-read GB/s as fraction of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_traffic.json")


# ----------------------------------------------------------------------------- helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, device):
    """Element-wise maximum over all ranks of the initialised process group (the slowest
    replica sets a time-like metric)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if k in d:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s (burst: the prefill call is timed alone):
    MEASURED_PEAKS.json when present, else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        v = d.get("bf16_tflops")
        if v:
            return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


KERNEL_SOURCES = {
    "attn_cluster_kernel": ("attention.cu", "gqa_common.cuh", "rowmath.cuh"),
    "attn_splitkv_kernel": ("attention.cu", "gqa_common.cuh", "rowmath.cuh"),
    "q4_cluster_kernel": ("attention_q4.cu", "gqa_common.cuh", "launch.h"),
}


def _code_only(src: str) -> str:
    """C/CUDA source with comments removed and whitespace runs collapsed (string and
    character literals kept verbatim), so that editing a comment does not change the
    hash of a kernel's code."""
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
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str = "attn_cluster_kernel"):
    """Hash of the code (comments and layout excluded) of the files `kernel` is built from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "gqa_decode_attention_fa_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` (read + write) from the committed ncu capture of
    this workload, if it was taken on the kernel's current source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    rec = d.get("workloads", {}).get(workload)
    if rec is None or rec.get("kernel") != kernel or kernel not in KERNEL_SOURCES:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    return int(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.05)
        return self

    def __exit__(self, *a):
        self.result = self._collect()

    def _collect(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads

def build_layers(name: str, device: str, l2_bytes: int, layers: int = 0):
    """Per-step list of workloads: the 40 layers for the sweep, else one workload.  Small
    caches are replicated into enough copies (> 3x L2) that every step reads from HBM;
    caches larger than 2x L2 get a second copy.  The copies rotate across steps (as a
    model's layers do), so that consecutive steps -- which overlap on the device -- never
    read the same cache.  `layers` > 0 cuts the 40-layer sweep to that many layers (for
    profiling one layer under ncu)."""
    import torch

    from gqa_decode_attention_fa_gb300 import workloads as wl

    if name == "qwen3-14b-40layer":
        n = layers if layers > 0 else wl.LAYERS_40
        ws = [wl.named(name, device=device, layer=l) for l in range(n)]
        if n == 1:  # one layer: alternate with a second one
            return [ws, [wl.named(name, device=device, layer=1)]], "inputs > L2 (1 GiB KV per layer, 2 layers alternating)"
        return [ws], f"inputs > L2 (1 GiB KV per layer, {n} layers)"
    if name == "qwen3-14b-4k-decode":
        steps = wl.decode_sweep(device=device)
        kvb = sum(w.kv_bytes() for w in steps[-1])
        return steps, (f"inputs > L2 ({kvb / 2**20:.0f} MiB KV over {len(steps[-1])} layers); the {len(steps)} "
                       f"autoregressive steps repeat (each rewrites the rows it appended)")
    w = wl.named(name, device=device)
    kvb = w.kv_bytes()
    copies = 2 if kvb >= 2 * l2_bytes else int(math.ceil(3 * l2_bytes / kvb))
    sets = [[w]]
    for _ in range(copies - 1):
        c = wl.Workload(**{**w.__dict__})
        c.k_cache = w.k_cache.clone()
        c.v_cache = w.v_cache.clone()
        sets.append([c])
    torch.cuda.synchronize()
    if copies == 2 and kvb >= 2 * l2_bytes:
        return sets, f"inputs > L2 ({kvb / 2**20:.0f} MiB KV per step, 2 cache copies alternating)"
    return sets, f"rotating {copies} cache copies ({copies * kvb / 2**20:.0f} MiB > 3x L2)"


def algorithmic_kv_bytes(layers) -> int:
    return sum(w.kv_bytes() for w in layers)


def workload_config(name: str, layers: int = 0) -> dict:
    """The workload's description (no device work): both arms print it in `config`."""
    from gqa_decode_attention_fa_gb300 import workloads as wl

    if name == "qwen3-14b-4k-decode":
        return {"workload": name, "batch": 1, "q_heads": 40, "kv_heads": 8, "head_dim": 128,
                "layers": wl.LAYERS_40, "seq_lens": f"{4096 - wl.DECODE_STEPS + 1}..4096 (one token per step)",
                "cache": "contiguous", "parallelism": "replicas"}
    geo = {"qwen3-14b-tiny": (1, 40, 8, 256, "contiguous"), "qwen3-14b-4k": (1, 40, 8, 4096, "contiguous"),
           "qwen3-14b-ragged": (32, 40, 8, "ragged U[512,8192]", "paged-64"),
           "llama3-70b-128k": (1, 64, 8, 131072, "contiguous"),
           "qwen3-14b-40layer": (8, 40, 8, 32768, "paged-64")}[name]
    n = (layers if layers > 0 else wl.LAYERS_40) if name == "qwen3-14b-40layer" else 1
    return {"workload": name, "batch": geo[0], "q_heads": geo[1], "kv_heads": geo[2], "head_dim": 128,
            "layers": n, "seq_lens": geo[3], "cache": geo[4], "parallelism": "replicas"}


def percentiles(xs):
    xs = sorted(xs)

    def q(f):
        if len(xs) == 1:
            return xs[0]
        i = f * (len(xs) - 1)
        lo = int(math.floor(i))
        return xs[lo] + (xs[min(lo + 1, len(xs) - 1)] - xs[lo]) * (i - lo)
    return {"median": round(q(0.5), 3), "p10": round(q(0.1), 3), "p90": round(q(0.9), 3), "n": len(xs)}


# ----------------------------------------------------------------------------- our arm

INVOCATIONS = 20


def run_ours(args, rank, world, local):
    import torch

    from gqa_decode_attention_fa_gb300 import binding

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    free, _ = torch.cuda.mem_get_info(local)
    need = 48 * 2**30 if args.workload == "qwen3-14b-40layer" and args.layers == 0 else 4 * 2**30
    if free < need:
        raise SystemExit(f"bench: {free / 2**30:.1f} GiB free on {dev}, workload needs ~{need / 2**30:.0f} GiB")
    sets, l2_note = build_layers(args.workload, dev, l2, args.layers)
    first = sets[0][0]
    plan = binding.Plan(first.B, first.Hq, first.Hkv, first.max_seq, block_size=first.block_size,
                        num_cache_blocks=max(w.num_blocks for s in sets for w in s), device=local,
                        seq_lens_host=first.seq_lens.cpu().numpy())
    outs = [torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device=dev) for w in sets[0]]
    stream = torch.cuda.Stream(device=dev)
    kv_per_step = sum(algorithmic_kv_bytes(s) for s in sets) // len(sets)  # mean over the step list
    single = plan.cluster_size > 0
    launches_per_layer = 1 if single else 2
    launches_per_step = launches_per_layer * len(sets[0])
    form = (f"single launch, clusters of {plan.cluster_size} CTAs per (sequence, KV head)" if single
            else f"split-KV ({plan.num_workers} workers) + combine")

    def step(k):
        """One decode step through the fused entry point (prologue, attention, combine)."""
        for li, w in enumerate(sets[k % len(sets)]):
            plan.run(w, outs[li], stream)

    barrier = (lambda: torch.distributed.barrier()) if world > 1 else (lambda: None)
    K, W = args.steps, args.warmup
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    with torch.cuda.stream(stream), ClockSampler(local) as clk:
        # warm-up: at least W steps and at least --warmup-seconds of GPU work so the clock
        # record covers the loaded state
        t0 = time.perf_counter()
        done = 0
        while done < W or time.perf_counter() - t0 < args.warmup_seconds:
            step(done)
            done += 1
            if done % 64 == 0:
                stream.synchronize()
        stream.synchronize()
        graph = None
        if args.launch == "graph":
            # the K steps captured once (their launches keep their programmatic dependencies)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for k in range(K):
                    step(k)
            graph.replay()
            stream.synchronize()

        def region():
            a, b = ev(), ev()
            a.record(stream)
            if graph is not None:
                graph.replay()
            else:
                for k in range(K):
                    step(k)
            b.record(stream)
            return a, b

        region()  # one untimed pass of the exact timed sequence
        stream.synchronize()
        barrier()
        torch.cuda.synchronize()
        e_start, e_end = region()
        torch.cuda.synchronize()
        barrier()
        # the same K steps again as separate invocations: their spread
        inv = []
        for _ in range(INVOCATIONS):
            a, b = region()
            inv.append((a, b))
        # and launched eagerly (host launch rate included)
        a_eager, b_eager = ev(), ev()
        a_eager.record(stream)
        for k in range(K):
            step(k)
        b_eager.record(stream)
        torch.cuda.synchronize()
        # each step's kernel launched in plain stream order (no overlap between steps, as after
        # a caller kernel that writes the step's inputs); the plan re-selects its cluster size
        plan.set_ordered_start(True)
        ordered_form = plan.cluster_size
        for k in range(max(3, W)):
            step(k)
        o_graph = None
        if args.launch == "graph":
            o_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(o_graph, stream=stream):
                for k in range(K):
                    step(k)
            o_graph.replay()
        stream.synchronize()
        a_ord, b_ord = ev(), ev()
        a_ord.record(stream)
        if o_graph is not None:
            o_graph.replay()
        else:
            for k in range(K):
                step(k)
        b_ord.record(stream)
        torch.cuda.synchronize()
        plan.set_ordered_start(False)
        del o_graph
    clocks = clk.result
    region_ms = e_start.elapsed_time(e_end)
    inv_us = [a.elapsed_time(b) * 1e3 / K for a, b in inv]
    eager_us = a_eager.elapsed_time(b_eager) * 1e3 / K
    ordered_us = a_ord.elapsed_time(b_ord) * 1e3 / K
    del graph
    if plan.device_errors() != 0:
        raise SystemExit("bench: device error flags set during the timed region")

    # e2e: host buffers through gqa_decode_attn_host, inputs in / output out every step
    host = []
    for w in sets[0]:
        host.append({k: getattr(w, k).cpu().pin_memory() for k in ("q_new", "k_new", "v_new", "seq_lens", "positions")})
    out_h = [torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16).pin_memory() for w in sets[0]]
    h2d = sum(sum(t.numel() * t.element_size() for t in h.values()) for h in host)
    d2h = sum(t.numel() * t.element_size() for t in out_h)

    def e2e_step(k):
        for li, w in enumerate(sets[k % len(sets)]):
            h = host[li]
            plan.decode_attn_host(h["q_new"], h["k_new"], h["v_new"], w.k_cache, w.v_cache, w.page_table,
                                  h["seq_lens"], h["positions"], w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps,
                                  out_h[li], stream)
        stream.synchronize()   # the step's result is on the host before the next step

    for k in range(max(3, W)):
        e2e_step(k)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(K):
        e2e_step(k)
    e2e_s = time.perf_counter() - t0
    barrier()

    us_step = region_ms * 1e3 / K
    e2e_us = e2e_s * 1e6 / K
    if world > 1:
        us_step, e2e_us = max_over_ranks([us_step, e2e_us], dev)

    peak, peak_src = hbm_peak()
    kv_per_launch = kv_per_step / len(sets[0])
    per_launch_us = us_step / len(sets[0]) if single else None
    kernel = "attn_cluster_kernel" if single else "attn_splitkv_kernel"
    achieved = kv_per_step / (us_step * 1e-6) / 1e9
    traffic = recorded_traffic(args.workload, kernel)
    config = workload_config(args.workload, args.layers)
    config.update({"parallelism": f"replicas x{world}", "l2": l2_note, "form": form,
                   "launch": (f"CUDA graph of the {K} timed steps (programmatic dependent launches kept)"
                              if args.launch == "graph" else "eager launches")})
    result = {
        "metric": METRIC,
        "value": round(us_step, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(us_step / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the named workload)",
        "config": config,
        "kv_bytes_per_step": kv_per_step,
        "kv_gbs": round(kv_per_step / (us_step * 1e-6) / 1e9, 1),
        "invocations": {**percentiles(inv_us), "unit": "us/step",
                        "how": f"{INVOCATIONS} further timed regions of the same {K} steps"},
        "eager_us_per_step": round(eager_us, 3),
        "ordered_start": {"us_per_step": round(ordered_us, 3), "cluster_size": ordered_form,
                          "how": ("the same steps with each step's kernel launched in plain stream order "
                                  "(gqa_plan_set_ordered_start): no overlap between steps, as in a model whose "
                                  "projection kernel before each attention call writes its inputs")},
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_of_8TBs": round(achieved / 8000.0, 4),
                     "per_launch_us": None if per_launch_us is None else round(per_launch_us, 3),
                     "algorithmic_bytes_per_launch": int(kv_per_launch),
                     "note": ("one kernel per layer; consecutive launches overlap (programmatic dependent "
                              "launch), so a launch's share of the timed region is the region over the launches"
                              if single else
                              "two kernels per layer (attention, combine); achieved is over the whole step"),
                     "traffic": traffic},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/step", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches_per_step * K,
        "gpu_launches_note": (f"{launches_per_layer} kernel(s) per layer (" +
                              ("the single-launch step" if single else "split-KV attention + combine") +
                              "); the RoPE table kernel runs once per theta, before the timed region"),
        "clocks": clocks,
    }
    return result, sets


# ----------------------------------------------------------------------------- prefill

PREFILL = "qwen3-14b-prefill-4k"


def run_prefill(name: str, steps: int, warmup: int, local: int):
    """One chunk of causal prefill (gqa_prefill_attn: the prologue kernel and the tcgen05
    attention kernel) timed call by call with CUDA events; L2 is flushed between calls by
    writing a buffer twice its size outside the events.  The roofline is the tensor pipe:
    algorithmic flops (4 d per query head and visible key) over the call's duration."""
    import torch

    from gqa_decode_attention_fa_gb300 import binding, workloads as wl

    dev = f"cuda:{local}"
    w = wl.named_prefill(name, device=dev)
    out = torch.empty((w.B, w.T, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        binding.prefill_attn_workload(w, out, device_errors=err, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(local) as clk:
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            binding.prefill_attn_workload(w, out, device_errors=err, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit("bench: device error flags set during the prefill calls")
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    flops = w.flops()
    peak, src = bf16_peak()
    achieved = flops / (us * 1e-6) / 1e12
    return {"us_per_call": round(us, 3), "tokens": w.B * w.T, "q_start": int(w.q_start[0]),
            "tflops": round(achieved, 1),
            "roofline": {"bound": "tensor", "kernel": "prefill_rope_kernel + prefill_attn_kernel (whole call)",
                         "achieved": round(achieved, 1), "peak": peak, "peak_source": src, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "algorithmic_flops_per_call": int(flops)},
            "l2": "flushed between calls (2x L2 write outside the events)", "steps": steps,
            "clocks_sm_mhz": clk.result["sm_mhz"]}


# ----------------------------------------------------------------------------- 4-bit KV cache

Q4 = ("qwen3-14b-4k-q4", "qwen3-14b-ragged-q4")


def run_q4(name: str, steps: int, warmup: int, local: int):
    """The decode step over a 4-bit cache (gqa_decode_attn_q4), K steps as one CUDA graph
    replayed between CUDA events after warm-up, the median of seven replays.  Caches
    smaller than twice L2 are replicated (> 3x L2 of copies, rotated across steps) so that
    every step reads from HBM.  Roofline: the cache bytes a step reads (64 index bytes + a
    4-byte scale per token, KV head and tensor) over the step's time."""
    import torch

    from gqa_decode_attention_fa_gb300 import binding, workloads as wl

    dev = f"cuda:{local}"
    w = wl.named_q4(name, device=dev)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    kvb = w.kv_bytes()
    sets = [w]
    if kvb < 2 * l2:
        for _ in range(int(math.ceil(3 * l2 / kvb)) - 1):
            c = wl.Q4Workload(**{**w.__dict__})
            c.k_idx, c.v_idx = w.k_idx.clone(), w.v_idx.clone()
            c.k_scale, c.v_scale = w.k_scale.clone(), w.v_scale.clone()
            sets.append(c)
    l2_note = (f"rotating {len(sets)} cache copies ({len(sets) * kvb / 2**20:.0f} MiB > 3x L2)" if len(sets) > 1
               else f"inputs > L2 ({kvb / 2**20:.0f} MiB per step)")
    plan = binding.Plan(w.B, w.Hq, w.Hkv, w.max_seq, block_size=w.block_size, num_cache_blocks=w.num_blocks,
                        device=local, seq_lens_host=w.seq_lens.cpu().numpy())
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream), ClockSampler(local) as clk:
        for k in range(max(3, warmup)):
            plan.run_q4(sets[k % len(sets)], out, stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()  # the timed steps captured once, as for the bf16 cache
        with torch.cuda.graph(graph, stream=stream):
            for k in range(steps):
                plan.run_q4(sets[k % len(sets)], out, stream)
        graph.replay()
        stream.synchronize()
        reps = []
        for _ in range(7):  # the median of seven timed replays
            a.record(stream)
            graph.replay()
            b.record(stream)
            stream.synchronize()
            reps.append(a.elapsed_time(b) * 1e3 / steps)
        del graph
    if plan.device_errors() != 0:
        raise SystemExit("bench: device error flags set during the 4-bit-cache steps")
    us = statistics.median(reps)
    peak, src = hbm_peak()
    gbs = kvb / (us * 1e-6) / 1e9
    single = plan.cluster_size > 0
    kernel = "q4_cluster_kernel" if single else "q4 prologue + attention + combine (whole step)"
    return {"us_per_step": round(us, 3), "kv_bytes_per_step": kvb, "kv_gbs": round(gbs, 1),
            "bf16_cache_bytes_per_step": int(w.seq_lens.long().sum().item()) * w.Hkv * w.d * 2 * 2,
            "roofline": {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 1), "peak": peak,
                         "peak_source": src, "unit": "GB/s", "frac": round(gbs / peak, 4),
                         "traffic": recorded_traffic(name, kernel) if single else None},
            "form": (f"single launch, clusters of {plan.cluster_size} CTAs per (sequence, KV head)" if single
                     else f"split-KV ({plan.num_workers} workers): prologue, attention, combine"),
            "l2": l2_note, "steps": steps, "clocks_sm_mhz": clk.result["sm_mhz"]}


_ORACLE_CORES = []  # the oracle's thread count before anything changed it


def cpu_baseline(name: str, budget_s: float = 12.0, layers: int = 0, threads: int = 0):
    """The fp64 oracle, as it stands, on the host cores (all of them, or `threads`): whole
    decode steps of the workload (for the 40-layer sweep: whole layers, scaled by the step's
    layer count) until ~budget_s of CPU time."""
    import oracle
    from gqa_decode_attention_fa_gb300 import workloads as wl
    from gqa_decode_attention_fa_gb300.workloads import bits, ints

    w = wl.named(name, device="cpu")
    args = [bits(w.q_new), bits(w.k_new), bits(w.v_new), bits(w.k_cache), bits(w.v_cache), ints(w.page_table),
            ints(w.seq_lens), ints(w.positions), bits(w.q_norm_w), bits(w.k_norm_w), w.rope_theta, w.eps]
    g = oracle.geom(w.B, w.Hq, w.Hkv, w.d, w.block_size, w.max_seq, w.num_rows)
    if not _ORACLE_CORES:
        _ORACLE_CORES.append(oracle.max_threads())
    oracle.set_threads(threads or _ORACLE_CORES[0])
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        r = oracle.decode_step(g, *args)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > budget_s or len(times) >= 200:
            break
    oracle.set_threads(_ORACLE_CORES[0])  # leave the oracle on all cores
    per_unit = statistics.median(times)
    layers = (layers or wl.LAYERS_40) if name == "qwen3-14b-40layer" else 1
    unit = "layer" if name == "qwen3-14b-40layer" else "step"
    return {"value": round(per_unit * layers * 1e6, 1), "unit": "us/step", "cores": int(r["threads"]),
            "kind": "oracle",
            "sample": f"{len(times)} full {unit}(s) of {name} in fp64 (median), x{layers} per step"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: whole steps of the same workload on the host."""
    if rank != 0:
        return None
    import oracle
    from gqa_decode_attention_fa_gb300 import workloads as wl
    from gqa_decode_attention_fa_gb300.workloads import bits, ints

    layers = (getattr(args, "layers", 0) or wl.LAYERS_40) if args.workload == "qwen3-14b-40layer" else 1
    w = wl.named(args.workload, device="cpu")
    g = oracle.geom(w.B, w.Hq, w.Hkv, w.d, w.block_size, w.max_seq, w.num_rows)
    a = [bits(w.q_new), bits(w.k_new), bits(w.v_new), bits(w.k_cache), bits(w.v_cache), ints(w.page_table),
         ints(w.seq_lens), ints(w.positions), bits(w.q_norm_w), bits(w.k_norm_w), w.rope_theta, w.eps]
    # bounded sample: one layer stands for each of the 40 identical-shape layers
    K, W = args.steps, args.warmup
    budget = 150.0
    r = None
    for _ in range(W):
        r = oracle.decode_step(g, *a)
    t0 = time.perf_counter()
    done = 0
    for _ in range(K):
        r = oracle.decode_step(g, *a)
        done += 1
        if time.perf_counter() - t0 > budget:
            break
    per = (time.perf_counter() - t0) / done
    us = per * layers * 1e6
    threads = int(r["threads"]) if r else oracle.max_threads()
    sample = (f"{done} timed oracle step(s) of {args.workload}" if layers == 1 else
              f"{done} timed oracle layer(s) of {args.workload}, x{layers} layers per step")
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/step", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, getattr(args, "layers", 0)),
        "cpu_baseline": {"value": round(us, 1), "unit": "us/step", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(us, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--warmup-seconds", type=float, default=0.3,
                    help="keep warming up for at least this long (so the clock record sees the loaded GPU)")
    ap.add_argument("--by-config", default="qwen3-14b-tiny,qwen3-14b-4k,qwen3-14b-ragged,llama3-70b-128k,"
                                           "qwen3-14b-4k-decode," + PREFILL + "," + ",".join(Q4),
                    help="other workloads to time (GPU only) into the line's by_config; '' for none")
    ap.add_argument("--layers", type=int, default=0,
                    help="cut the 40-layer sweep to this many layers (for profiling one layer); 0 = all 40")
    ap.add_argument("--launch", default="graph", choices=["graph", "eager"],
                    help="time the K steps as one CUDA graph replay (default) or as eager launches")
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        r = run_reference(args, rank, world)
        if r is not None:
            print(json.dumps(r), flush=True)
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    from gqa_decode_attention_fa_gb300 import binding
    binding.load()
    result, sets = run_ours(args, rank, world, local)
    del sets
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.workload, layers=result["config"]["layers"])
    by = {}
    for name in [n for n in args.by_config.split(",") if n and n != args.workload]:
        if name == PREFILL:
            by[name] = run_prefill(name, min(args.steps, 20), args.warmup, local)
            torch.cuda.empty_cache()
            continue
        if name in Q4:
            by[name] = run_q4(name, BY_CONFIG_STEPS, args.warmup, local)
            torch.cuda.empty_cache()
            continue
        sub = argparse.Namespace(**{**vars(args), "workload": name, "steps": BY_CONFIG_STEPS, "layers": 0})
        r, s = run_ours(sub, rank, world, local)
        del s
        torch.cuda.empty_cache()
        by[name] = {"us_per_step": r["value"], "eager_us_per_step": r["eager_us_per_step"],
                    "ordered_start": r["ordered_start"],
                    "invocations": r["invocations"], "kv_gbs": r["kv_gbs"], "roofline": r["roofline"],
                    "e2e_us": r["e2e"]["value"], "steps": r["steps"], "form": r["config"]["form"],
                    "l2": r["config"]["l2"], "clocks_sm_mhz": r["clocks"]["sm_mhz"]}
        from gqa_decode_attention_fa_gb300 import workloads as wl
        if rank == 0 and not args.no_cpu_baseline and name in wl.WORKLOADS:
            # the oracle on all host cores, and on one core for the two short steps
            by[name]["cpu_baseline"] = cpu_baseline(name, budget_s=3.0)
            if name in ("qwen3-14b-tiny", "qwen3-14b-4k"):
                by[name]["cpu_baseline_1_core"] = cpu_baseline(name, budget_s=3.0, threads=1)
    if by:
        result["by_config"] = by
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
