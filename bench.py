#!/usr/bin/env python
"""Benchmark of batched tree attention on GB300.

One step = one ``tree_attn`` call = the plan kernel (work enumeration, tile
classification), with RoPE the key rotation with its cos/sin table (folded
into the plan kernel for small problems), and the persistent attention
kernel, over one batch of the named synthetic workload (default: the
ragged-large workload, the largest of the benchmark set).  Prints one JSON
line (rank 0) whose ``per_config`` object holds the same measurement for the
spec-decode, prefix+tree, ragged-large and degenerate workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--repeats R]
                  [--workload NAME] [--impl gb300|reference]

Under torchrun each rank runs its own copy of the workload on its own GPU
(weak scaling, no data-path collective); the step time is the max over ranks.
``--impl reference`` times the CPU oracle on bounded samples of the same
workload (rank 0 only).
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "tree-attn TFLOP/s (unmasked pairs) + % of roofline, 1 GB300"
UNIT = "TFLOP/s"
WORKLOADS = {name: i + 1 for i, name in enumerate(wl.CONFIG_NAMES)}
# beyond the five workloads: few sequences with a 32768-token prefix (the case
# split-KV is for)
EXTRA_WORKLOADS = {"long-prefix": lambda: wl.long_prefix()}


def make_workload(name: str):
    if name in WORKLOADS:
        return wl.config(WORKLOADS[name])
    return EXTRA_WORKLOADS[name]()
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------
# multi-rank helpers (host logic; covered by gloo tests on CPU)
# --------------------------------------------------------------------------

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank processed ``units_per_rank``."""
    return units_per_rank * world / max_seconds


# --------------------------------------------------------------------------
# measurement helpers
# --------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("ta_attn.cu", "ta_device.cuh", "ta_layout.h"):
        with open(os.path.join(ROOT, "tree_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[workload]
        if e.get("kernel_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(", ") for r in self.file.read().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def set_bytes(w) -> int:
    es = 2
    return (2 * w.total_q * w.h_q * w.head_dim * es + 2 * w.total_kv * w.h_kv * w.head_dim * es
            + 4 * w.total_q * w.h_q)


# --------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# --------------------------------------------------------------------------

def oracle_sample(w, budget_s: float):
    """Pick a prefix of the sequences whose oracle time fits ``budget_s``
    (estimated from visible pairs after timing one sequence)."""
    import oracle
    t0 = time.perf_counter()
    oracle.tree_attention_workload(w, seqs=[0])
    t1 = max(time.perf_counter() - t0, 1e-4)
    per_pair = t1 / max(1, _pairs(w, [0]))
    seqs, acc = [], 0.0
    for b in range(w.batch_size):
        est = per_pair * _pairs(w, [b])
        if seqs and acc + est > budget_s:
            break
        seqs.append(b)
        acc += est
    return seqs


def _pairs(w, seqs) -> int:
    tot = 0
    for b in seqs:
        n = len(w.parents[b])
        dep = wl.tree_depths(w.parents[b])
        rows = np.arange(n - w.qo_lens[b], n)
        tot += int(np.sum(dep[rows] + 1)) + w.prefix_lens[b] * len(rows)
    return tot


def time_oracle(w, seqs):
    import oracle
    t0 = time.perf_counter()
    oracle.tree_attention_workload(w, seqs=seqs)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.head_dim * w.h_q * _pairs(w, seqs)
    return flops, dt


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, budget_s=15.0):
    seqs = oracle_sample(w, budget_s)
    flops, dt = time_oracle(w, seqs)
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{len(seqs)} of {w.batch_size} sequences of the {w.name} workload, "
                      f"one pass, {dt:.1f} s (numpy float64, BLAS threads = host cores)"}


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def run_reference(args):
    rank, _, world = dist_info()
    if rank != 0:
        return 0
    w = make_workload(args.workload)
    per_step_budget = max(0.5, 150.0 / (args.steps + args.warmup))
    seqs = oracle_sample(w, per_step_budget)
    for _ in range(args.warmup):
        time_oracle(w, seqs)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        f, _dt = time_oracle(w, seqs)
        flops += f
    total = time.perf_counter() - t0
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config_dict(w, None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{len(seqs)} of {w.batch_size} sequences per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config_dict(w, l2_note):
    d = {"workload": w.name, "batch": w.batch_size, "total_q": w.total_q,
         "total_kv": w.total_kv, "h_q": w.h_q, "h_kv": w.h_kv, "head_dim": w.head_dim,
         "rotary": bool(w.rotary_mode), "visible_pairs_per_head": wl.visible_pairs(w)}
    if l2_note:
        d["l2"] = l2_note
    return d


PER_CONFIG = ("spec-decode", "prefix+tree", "ragged-large", "degenerate", "long-prefix")


def _roofline(nbytes, flops, seconds, peaks):
    """The bound that applies to ``nbytes`` / ``flops`` (the slower of HBM
    copy bandwidth and the bf16 tensor peak) and the fraction reached in
    ``seconds``."""
    if nbytes / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops"] * 1e12):
        r = {"bound": "hbm", "achieved": nbytes / seconds / 1e9, "peak": peaks["hbm_gbs"],
             "unit": "GB/s"}
    else:
        r = {"bound": "tensor", "achieved": flops / seconds / 1e12,
             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    return r


def measure_workload(ta, w, args, dev, stream, world, local, headline=False):
    """Times the one-call ``tree_attn`` step on workload ``w``: ``repeats``
    runs of exactly ``steps`` back-to-back steps (each run bracketed by a
    barrier and a device synchronisation, CUDA events on the launching
    stream), the median run giving ms per step; then a second pass through
    the plan / run entry points with events between the launches for the
    per-kernel split.  With ``headline`` it also samples clocks during the
    timed runs (stretching the repeats so that the sampler sees them) and
    measures the end-to-end call with host buffers."""
    flops = wl.algorithmic_flops(w)
    nbytes = wl.algorithmic_bytes(w)
    sb = set_bytes(w)
    n_sets = args.sets or max(1, min(16, math.ceil(2.2 * L2_BYTES / sb)))
    l2_note = (f"rotating {n_sets} input/output sets ({n_sets * sb / 1e6:.0f} MB > 2x L2)"
               if n_sets > 1 else f"inputs larger than L2 ({sb / 1e6:.0f} MB)")
    base = wl.device_inputs(w, dev)
    sets = []
    for i in range(n_sets):
        d = {k: (v.clone() if v is not None else None) for k, v in base.items()}
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=dev)
        dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode)
        d["ws"] = torch.zeros(ta.workspace_size(dims), dtype=torch.uint8, device=dev)
        d["dims"] = dims
        sets.append(d)

    def step(d):
        # one call: plan kernel, key rotation under RoPE, attention kernel
        ta.tree_attn(d["q"], d["q_indptr"], d["k"], d["v"], d["kv_indptr"],
                     d["q_rope_position"], d["mn_indptr"], d["tree_order"], d["out"], d["lse"],
                     w.rotary_mode, w.rope_scale, w.rope_theta, w.sm_scale, d["ws"], stream)

    def step_two_launch(d, ev):
        # the plan / run entry points, events between them (run = key rotation
        # under RoPE + attention kernel)
        ev[0].record(stream)
        ta.plan(d["q"], d["q_indptr"], d["k"], d["kv_indptr"], d["q_rope_position"],
                d["mn_indptr"], d["tree_order"], w.rotary_mode, w.rope_scale, w.rope_theta,
                d["ws"], stream)
        ev[1].record(stream)
        ta.run(d["q"], d["k"], d["v"], d["q_indptr"], d["kv_indptr"], d["q_rope_position"],
               d["mn_indptr"], d["tree_order"], d["out"], d["lse"], w.rotary_mode, w.rope_scale,
               w.rope_theta, w.sm_scale, d["ws"], stream)
        ev[2].record(stream)

    def check_status(when):
        for d in sets:
            st = ta.device_status(d["ws"], stream)
            if st != ta.TA_OK:
                raise RuntimeError(f"{w.name}: device status {when}: {ta.status_string(st)}")

    K = args.steps
    for i in range(args.warmup):
        step(sets[i % n_sets])
    torch.cuda.synchronize(dev)
    check_status("after warm-up")

    def timed_run():
        # events only around the whole run: an event between two launches is
        # a stream operation of its own and would break the overlap of
        # programmatic dependent launch
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for i in range(K):
            step(sets[i % n_sets])
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return max_over_ranks(a.elapsed_time(b), world, dev)

    repeats = max(1, args.repeats)
    clk = None
    sample_clocks = headline and not args.no_clocks
    if sample_clocks:
        # enough repeats that the timed runs span about a second of clock samples
        probe = timed_run()
        repeats = max(repeats, min(400, math.ceil(1000.0 / max(probe, 1e-3))))
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.3)
    runs = [timed_run() for _ in range(repeats)]
    if sample_clocks:
        clk = clocks.stop()
    run_ms = statistics.median(runs)
    ms_step = run_ms / K
    # per-kernel split for the roofline (the plan / run entry points never
    # split: when the one-call step splits the kv range by itself, the step
    # time stands for the kernels)
    split_cap = ta.auto_split_chunks(sets[0]["dims"])
    attn_ms = plan_ms = None
    if split_cap == 1:
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for i in range(K):
            step_two_launch(sets[i % n_sets], evs[i])
        torch.cuda.synchronize(dev)
        attn_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
        plan_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    check_status("after timing")

    peaks, peak_src = measured_peaks()
    roof = _roofline(nbytes, flops, (attn_ms if attn_ms is not None else ms_step) / 1e3, peaks)
    roof["traffic"] = recorded_traffic(w.name)
    roof["peak_source"] = peak_src
    step_roof = _roofline(nbytes, flops, ms_step / 1e3, peaks)
    res = {
        "workload": w.name, "ms_per_step": ms_step, "runs": repeats, "steps_per_run": K,
        "run_ms_min": min(runs) / K, "run_ms_max": max(runs) / K,
        "tflops": flops / (ms_step / 1e3) / 1e12,
        "tokens_per_s": w.total_q / (ms_step / 1e3),
        "bound": roof["bound"], "frac": roof["frac"], "step_frac": step_roof["frac"],
        "attn_kernel_ms": attn_ms, "plan_kernel_ms": plan_ms, "traffic": roof["traffic"],
        "auto_split_chunks": split_cap,
        "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
        "gpu_launches_per_step": (2 + (w.rotary_mode == 1 and not ta.folds_rotation(w.total_kv))
                                  + (split_cap > 1)),
        "l2": l2_note,
    }
    if not headline:
        return res, None

    # end to end through the public call with host buffers: every step's
    # inputs in from pinned host memory and its out and lse back
    keys_in = ["q", "k", "v", "q_indptr", "kv_indptr", "mn_indptr", "tree_order",
               "q_rope_position"]
    host = {k: (base[k].cpu().pin_memory() if base[k] is not None else None) for k in keys_in}
    host_out = torch.empty(base["q"].shape, dtype=base["q"].dtype).pin_memory()
    host_lse = torch.empty(base["q"].shape[:2], dtype=torch.float32).pin_memory()
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys_in if host[k] is not None)
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * 4

    # two device sets in flight: while step i computes on one, step i+1's
    # inputs are copied into the other and step i-1's results copied out
    # (copy-in and copy-out streams of their own, ordered by events)
    e2e_sets = sets[:2] if len(sets) >= 2 else sets + [
        {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in sets[0].items()}]
    cin = torch.cuda.Stream(dev)
    cout = torch.cuda.Stream(dev)
    ev = [{n: torch.cuda.Event() for n in ("in", "done", "read")} for _ in e2e_sets]
    started = [False] * len(e2e_sets)

    def e2e_step(i):
        j = i % len(e2e_sets)
        d, e = e2e_sets[j], ev[j]
        if started[j]:
            cin.wait_event(e["done"])      # the set's previous step has read its inputs
        with torch.cuda.stream(cin):
            for k in keys_in:
                if host[k] is not None:
                    d[k].copy_(host[k], non_blocking=True)
            e["in"].record(cin)
        stream.wait_event(e["in"])
        if started[j]:
            stream.wait_event(e["read"])   # its previous results are out
        step(d)
        e["done"].record(stream)
        cout.wait_event(e["done"])
        with torch.cuda.stream(cout):
            host_out.copy_(d["out"], non_blocking=True)
            host_lse.copy_(d["lse"], non_blocking=True)
            e["read"].record(cout)
        started[j] = True

    for i in range(min(args.warmup, 3)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cin)
    for i in range(K):
        e2e_step(i)
    e1.record(cout)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    sets.extend(x for x in e2e_sets if all(x is not y for y in sets))
    check_status("after the end-to-end pass")
    extra = {"roofline": roof, "clocks": clk, "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h,
             "l2_note": l2_note, "flops": flops}
    return res, extra


def run_gb300(args):
    import tree_attention_gb300 as ta
    from tree_attention_gb300 import build as ta_build

    rank, local, world = dist_info()
    init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ta_build.build()
    ta.lib()
    ta.set_scheduler(1 if args.sched == "clc" else 0)
    stream = torch.cuda.current_stream(dev)
    w = make_workload(args.workload)
    head, extra = measure_workload(ta, w, args, dev, stream, world, local, headline=True)
    per_config = {}
    if not args.no_per_config:
        for name in PER_CONFIG:
            if name == w.name:
                per_config[name] = head
                continue
            res, _ = measure_workload(ta, make_workload(name), args, dev, stream, world, local)
            per_config[name] = res
            torch.cuda.empty_cache()

    K = args.steps
    ms = head["ms_per_step"]
    flops = extra["flops"]
    roof = dict(extra["roofline"])
    roof["kernel"] = ("run: attn_kernel (persistent tcgen05 tree attention), after the key "
                      "rotation under RoPE (timed through the plan / run entry points)")
    roof["kernel_ms"] = head["attn_kernel_ms"]
    roof["plan_kernel_ms"] = head["plan_kernel_ms"]
    roof["note"] = ("kernel_ms: median over the steps of the run half (key rotation under RoPE "
                    "+ attention kernel) timed with events between the launches, so without "
                    "launch overlap; the timed one-call step overlaps its launches, so "
                    "ms_per_step can be below plan + kernel")
    peaks, _ = measured_peaks()
    roof["t_roof_8tbs_us"] = max(head["algorithmic_bytes"] / 8e12,
                                 flops / (peaks["bf16_tflops"] * 1e12)) * 1e6
    roof["step_frac_of_t_roof"] = roof["t_roof_8tbs_us"] / (ms * 1e3)
    clk = extra["clocks"]
    if clk:
        clk["ms_per_step_x_sm_mhz"] = ms * clk["sm_mhz"]
    line = {
        "metric": METRIC,
        "value": weak_scaling_value(flops, world, ms / 1e3) / 1e12,
        "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(_config_dict(w, extra["l2_note"]), scheduler=args.sched),
        "timing": (f"median of {head['runs']} runs of {K} steps (min {head['run_ms_min']:.4f}, "
                   f"max {head['run_ms_max']:.4f} ms per step), CUDA events on the launching "
                   f"stream, max over ranks"),
        "tokens_per_s": weak_scaling_value(w.total_q, world, ms / 1e3),
        "roofline": roof,
        "e2e": {"value": weak_scaling_value(flops * K, world, extra["e2e_ms"] / 1e3) / 1e12,
                "unit": UNIT, "h2d_bytes_per_step": int(extra["h2d"]),
                "d2h_bytes_per_step": int(extra["d2h"])},
        # per timed run: plan kernel, key-rotation kernel (RoPE, unless the
        # plan kernel folds it in: small problems), attention kernel
        "gpu_launches": head["gpu_launches_per_step"] * K,
        "clocks": clk,
        "per_config": per_config,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_gb300_paged(args):
    """The paged-KV path (``tree_attn_paged``) on the named workload's shapes,
    its K/V moved into 16-slot pages in a scattered order.  The pages' paged
    kernel has no RoPE, so the workload runs with RoPE off.  ``tree_attn_paged``
    is one call (plan + attention kernel); the roofline covers that call."""
    import dataclasses
    import tree_attention_gb300 as ta
    from tree_attention_gb300 import build as ta_build

    rank, local, world = dist_info()
    init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ta_build.build()
    ta.lib()
    ta.set_scheduler(1 if args.sched == "clc" else 0)
    w = dataclasses.replace(make_workload(args.workload), rotary_mode=0)
    flops = wl.algorithmic_flops(w)
    nbytes = wl.algorithmic_bytes(w)
    pk = wl.paged_from(w, seed=17, fill=0.0)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))

    host = {"q": w.q.contiguous(), "pages": pk.pages.contiguous(), "q_indptr": i32(w.q_indptr),
            "page_indptr": i32(pk.page_indptr), "page_values": i32(pk.page_values),
            "length_info": i32(pk.last_page_len), "mn_indptr": i32(w.mn_indptr),
            "tree_order": i32(w.tree_order.reshape(-1, 2))}
    sb = sum(t.numel() * t.element_size() for t in host.values()) + w.q.numel() * 2
    n_sets = args.sets or max(1, min(16, math.ceil(2.2 * L2_BYTES / sb)))
    l2_note = (f"rotating {n_sets} input/output sets ({n_sets * sb / 1e6:.0f} MB > 2x L2)"
               if n_sets > 1 else f"inputs larger than L2 ({sb / 1e6:.0f} MB)")
    sets = []
    for _ in range(n_sets):
        d = {k: v.to(dev) for k, v in host.items()}
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=dev)
        dims = ta.make_paged_dims(d["q"], d["pages"], d["q_indptr"], d["page_values"],
                                  d["tree_order"])
        d["ws"] = torch.zeros(ta.paged_workspace_size(dims), dtype=torch.uint8, device=dev)
        sets.append(d)
    stream = torch.cuda.current_stream(dev)

    def step(d):
        ta.tree_attn_paged(d["q"], d["q_indptr"], d["pages"], d["page_indptr"], d["page_values"],
                           d["length_info"], d["mn_indptr"], d["tree_order"], d["out"], d["lse"],
                           0, w.sm_scale, d["ws"], stream)

    for i in range(args.warmup):
        step(sets[i % n_sets])
    torch.cuda.synchronize(dev)
    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for i in range(K):
        step(sets[i % n_sets])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    max_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    for d in sets:
        st = ta.device_status(d["ws"], stream)
        if st != ta.TA_OK:
            raise RuntimeError(f"device status after timing: {ta.status_string(st)}")

    # end to end with host buffers: inputs in, out and lse back, every step
    hp = {k: v.pin_memory() for k, v in host.items()}
    host_out = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    host_lse = torch.empty(w.q.shape[:2], dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hp.values())
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * 4

    def e2e_step(d):
        for k in hp:
            d[k].copy_(hp[k], non_blocking=True)
        step(d)
        host_out.copy_(d["out"], non_blocking=True)
        host_lse.copy_(d["lse"], non_blocking=True)

    for i in range(min(args.warmup, 3)):
        e2e_step(sets[i % n_sets])
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        e2e_step(sets[i % n_sets])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    peaks, peak_src = measured_peaks()
    call_s = max_ms / K / 1e3
    if nbytes / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops"] * 1e12):
        roof = {"bound": "hbm", "achieved": nbytes / call_s / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / call_s / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = None
    roof["peak_source"] = peak_src
    roof["kernel"] = "tree_attn_paged call (plan kernel + paged attention kernel)"
    roof["kernel_ms"] = max_ms / K
    cfg = _config_dict(w, l2_note)
    cfg.update({"paged": True, "page_size": wl.PAGE_SIZE, "num_pages": int(pk.pages.shape[0]),
                "note": "the pages' paged kernel has no RoPE: run with rotary off"})
    line = {
        "metric": METRIC,
        "value": weak_scaling_value(flops * K, world, max_ms / 1e3) / 1e12,
        "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": max_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": cfg,
        "tokens_per_s": weak_scaling_value(w.total_q * K, world, max_ms / 1e3),
        "roofline": roof,
        "e2e": {"value": weak_scaling_value(flops * K, world, e2e_ms / 1e3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": 2 * K,   # per step: plan kernel, paged attention kernel
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_gb300_split(args):
    """The split-KV path (``tree_attn_split``: plan, key rotation, attention
    over kv chunks, merge) on the named workload, with the unsplit
    ``tree_attn`` timed on the same buffers in the same run for comparison.
    The roofline covers the whole split call."""
    import tree_attention_gb300 as ta
    from tree_attention_gb300 import build as ta_build

    rank, local, world = dist_info()
    init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ta_build.build()
    ta.lib()
    ta.set_scheduler(1 if args.sched == "clc" else 0)
    w = make_workload(args.workload)
    flops = wl.algorithmic_flops(w)
    nbytes = wl.algorithmic_bytes(w)
    sb = set_bytes(w)
    n_sets = args.sets or max(1, min(16, math.ceil(2.2 * L2_BYTES / sb)))
    l2_note = (f"rotating {n_sets} input/output sets ({n_sets * sb / 1e6:.0f} MB > 2x L2)"
               if n_sets > 1 else f"inputs larger than L2 ({sb / 1e6:.0f} MB)")
    base = wl.device_inputs(w, dev)
    mc, ct = args.max_chunks, args.chunk_tiles
    sets = []
    for i in range(n_sets):
        d = {k: (v.clone() if v is not None else None) for k, v in base.items()}
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=dev)
        dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode)
        d["ws"] = torch.zeros(ta.split_workspace_size(dims, mc), dtype=torch.uint8, device=dev)
        d["ws1"] = torch.zeros(ta.workspace_size(dims), dtype=torch.uint8, device=dev)
        sets.append(d)
    stream = torch.cuda.current_stream(dev)
    keys_in = ["q", "k", "v", "q_indptr", "kv_indptr", "mn_indptr", "tree_order",
               "q_rope_position"]

    def step(d):
        ta.tree_attn_split(d["q"], d["q_indptr"], d["k"], d["v"], d["kv_indptr"],
                           d["q_rope_position"], d["mn_indptr"], d["tree_order"], d["out"],
                           d["lse"], w.rotary_mode, w.rope_scale, w.rope_theta, w.sm_scale, mc,
                           ct, d["ws"], stream)

    def step_unsplit(d):
        ta.tree_attn(d["q"], d["q_indptr"], d["k"], d["v"], d["kv_indptr"], d["q_rope_position"],
                     d["mn_indptr"], d["tree_order"], d["out"], d["lse"], w.rotary_mode,
                     w.rope_scale, w.rope_theta, w.sm_scale, d["ws1"], stream)

    K = args.steps

    def timed(fn):
        for i in range(args.warmup):
            fn(sets[i % n_sets])
        torch.cuda.synchronize(dev)
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(K):
            fn(sets[i % n_sets])
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return max_over_ranks(a.elapsed_time(b), world, dev)

    unsplit_ms = timed(step_unsplit)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    max_ms = timed(step)
    clk = clocks.stop()
    for d in sets:
        for key in ("ws", "ws1"):
            st = ta.device_status(d[key], stream)
            if st != ta.TA_OK:
                raise RuntimeError(f"device status after timing: {ta.status_string(st)}")

    # end to end through the public call with host buffers
    host = {k: (base[k].cpu().pin_memory() if base[k] is not None else None) for k in keys_in}
    host_out = torch.empty(base["q"].shape, dtype=base["q"].dtype).pin_memory()
    host_lse = torch.empty(base["q"].shape[:2], dtype=torch.float32).pin_memory()
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys_in if host[k] is not None)
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * 4

    def e2e_step(d):
        for k in keys_in:
            if host[k] is not None:
                d[k].copy_(host[k], non_blocking=True)
        step(d)
        host_out.copy_(d["out"], non_blocking=True)
        host_lse.copy_(d["lse"], non_blocking=True)

    e2e_ms = timed(e2e_step)

    peaks, peak_src = measured_peaks()
    call_s = max_ms / K / 1e3
    if nbytes / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops"] * 1e12):
        roof = {"bound": "hbm", "achieved": nbytes / call_s / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / call_s / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = None
    roof["peak_source"] = peak_src
    roof["kernel"] = ("tree_attn_split call (plan, key rotation, attention over kv chunks, "
                      "merge)")
    roof["kernel_ms"] = max_ms / K
    roof["t_roof_8tbs_us"] = max(nbytes / 8e12, flops / (peaks["bf16_tflops"] * 1e12)) * 1e6
    cfg = _config_dict(w, l2_note)
    cfg.update({"split_kv": True, "max_chunks": mc, "chunk_tiles": ct or "auto"})
    line = {
        "metric": METRIC,
        "value": weak_scaling_value(flops * K, world, max_ms / 1e3) / 1e12,
        "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": max_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": cfg,
        "tokens_per_s": weak_scaling_value(w.total_q * K, world, max_ms / 1e3),
        "unsplit_ms_per_step": unsplit_ms / K,
        "roofline": roof,
        "e2e": {"value": weak_scaling_value(flops * K, world, e2e_ms / 1e3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        # per step: plan kernel, key-rotation kernel (RoPE, unless folded into
        # the plan kernel), attention kernel, merge kernel
        "gpu_launches": (3 + (w.rotary_mode == 1 and not ta.folds_rotation(w.total_kv))) * K,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="ragged-large",
                    choices=list(WORKLOADS) + list(EXTRA_WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--sets", type=int, default=0, help="input/output buffer sets to rotate")
    ap.add_argument("--sched", choices=("queue", "clc"), default="clc",
                    help="attention work scheduling: cluster launch control over one CTA per "
                         "work unit (default) or the atomic work queue over one CTA per SM")
    ap.add_argument("--no-clocks", action="store_true",
                    help="no clock sampling (and no stretching of the timed runs to the "
                         "sampler's second): for runs under a profiler, whose line is not a "
                         "bench value")
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed runs of --steps steps each; the median run is reported")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --workload, not the four benchmark workloads beside it")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--paged", action="store_true",
                    help="time the paged-KV path (tree_attn_paged) on the workload's shapes")
    ap.add_argument("--split", action="store_true",
                    help="time the split-KV path (tree_attn_split), the unsplit call beside it")
    ap.add_argument("--max-chunks", type=int, default=16, help="split-KV: chunks per pair, max")
    ap.add_argument("--chunk-tiles", type=int, default=0,
                    help="split-KV: kv tiles per chunk (0: chosen by the plan)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.paged:
        return run_gb300_paged(args)
    if args.split:
        return run_gb300_split(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
