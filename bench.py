"""Benchmark of the paged-KV decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload peak] [--impl ours|reference]

One step = the whole decode hot path for one batch: the KV append (RoPE on the
new keys, K/V written into their page slots) followed by paged decode
attention (plus the split merge when the plan splits), for every layer of the
workload.  The default workload is 256 sequences x 2048 tokens of context,
one layer, 32 query / 8 kv heads, head dim 64, 32768 live pages randomly
scattered in a 40000-page pool.

Prints one JSON line.  `value` is achieved algorithmic HBM GB/s of the whole
step with all inputs resident in device memory; `e2e` repeats the measurement
with the per-step inputs copied from pinned host memory and the output copied
back inside the timed region.  `--impl reference` times the FP64 CPU oracle on
the host cores instead (a deliberately slow baseline, not a target).
Multi-GPU runs (torchrun) are independent replicas, one per rank (weak
scaling): the path has no exchange step.
"""
from __future__ import annotations

import argparse
import copy
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attn achieved HBM GB/s (% of peak); decode steps/s at bs=256"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "paged_decode_attention_peak_traffic.json")
CSRC = os.path.join(ROOT, "paged_kv_decode_04_gb300", "csrc")
# The source file of each decode kernel; every one of them also includes these headers.
KERNEL_FILES = {
    "paged_decode_kernel": "decode_attention.cu",
    "merge_plan_kernel": "decode_attention.cu",
    "merge_splits_kernel": "decode_attention.cu",
    "paged_decode_pagebox_kernel": "decode_pagebox.cu",
    "paged_decode_shared_kernel": "decode_shared.cu",
}
COMMON_SOURCES = ("decode_page.cuh", "pkv_device.cuh", "pkv_internal.h")
KERNEL_SOURCES = [os.path.join(CSRC, f)
                  for f in sorted(set(KERNEL_FILES.values())) + list(COMMON_SOURCES)]
# The traffic file holds a list of records {workload, kernel, kernel_sha, dram_bytes_per_launch};
# kernel_sha covers the sources of the kernels the record names.

WORKLOAD_TEXT = {
    "peak": "peak: 256 seqs x 2048 ctx, 1 layer, 32q/8kv/64 bf16, 32768 live pages (1 GiB K/V) "
            "randomly scattered in a 40000-page pool",
    "mix": "mix: 128 seqs (115 of 16-128, 13 of 1536-2048 tokens), 16 layers with per-layer "
           "tables, 32q/8kv/64 bf16, 8 GiB pool",
    "long": "long: 1 seq x 2048 ctx x 16 layers, 32q/8kv/64 bf16, shuffled pages, 4096-page pool",
    "small": "small: 8 seqs, lengths U[1,2048], 1 layer, 4096-page pool",
    "tiny": "tiny: 1 seq x 37 ctx, 1 layer, 64-page pool",
    "prefix": "prefix: 256 seqs x 2048 ctx, groups of 16 share a 1536-token prefix (96 aliased "
              "pages) + 32 private pages each, 9728 live pages in a 40000-page pool; K/V bytes "
              "are counted per sequence (effective bandwidth: shared pages may hit in L2)",
}


# ------------------------------------------------------------------ bytes --

def algorithmic_bytes(w, part: str = "step") -> int:
    """Bytes the step must move at minimum, per step (all layers).

    attention: K/V rows read once per kv head (sum L x Hkv x D x 2 x 2 B), q read
               and out written (B x Hq x D x 2 B each), the live block-table
               entries (4 B per page) and seq_lens (4 B per sequence);
    append:    new K/V read and written once (B x Hkv x D x 2 x 2 B, twice) and
               positions (4 B per sequence) -- the table entry it reads is
               counted with the attention's tables.
    """
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    lens = w.seq_lens.astype(np.int64)
    pages = (lens + w.page_size - 1) // w.page_size
    attn = int(lens.sum()) * Hkv * D * 2 * 2 + B * Hq * D * 2 * 2 + int(pages.sum()) * 4 + B * 4
    app = B * Hkv * D * 2 * 2 * 2 + B * 4
    per_layer = {"attention": attn, "append": app, "step": attn + app}[part]
    return per_layer * w.layers


# ------------------------------------------------------------- utilities --

def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["hbm_gbs"])
            return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources(kernel: str = None):
    """Source files of the kernels named in `kernel` ("a+b (fused step)"), or of all of them."""
    if kernel is None:
        return KERNEL_SOURCES
    names = kernel.split(" (")[0].split("+")
    files = sorted({KERNEL_FILES[n] for n in names if n in KERNEL_FILES})
    return [os.path.join(CSRC, f) for f in files + list(COMMON_SOURCES)]


def kernel_sha(kernel: str = None) -> str:
    """Hash of the code of the sources `kernel` is built from (all kernel
    sources if None): comments and whitespace do not count, so a comment edit
    does not orphan the recorded counters, and a change to one kernel's file
    does not orphan another kernel's."""
    h = hashlib.sha256()
    for p in kernel_sources(kernel):
        with open(p, encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def recorded_traffic(workload: str, kernel: str):
    """ncu DRAM bytes per launch of `kernel`, if recorded for the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            recs = json.load(f)
    except Exception:
        return None
    for rec in recs if isinstance(recs, list) else [recs]:
        if (rec.get("kernel_sha") == kernel_sha(kernel) and rec.get("workload") == workload
                and rec.get("kernel") == kernel):
            return rec.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_selector: str):
        self.rows = []
        self.proc = None
        self.thread = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_selector],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 - 0.15 <= t <= t1 + 0.15] or [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


def gpu_selector(dev_index: int) -> str:
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(dev_index).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v for v in vis.split(",") if v.strip()]
    if dev_index < len(ids) and ids[dev_index].strip().isdigit():
        return ids[dev_index].strip()
    return str(dev_index)


# ---------------------------------------------------------- distributed --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle --

def oracle_sample_run(w, n_seqs: int, rng_seed: int = 0, threads: int = 0):
    """Time the FP64 oracle on n_seqs sequences of every layer (append + attention).

    The sample's inputs are relabelled into compact host copies first (not
    timed).  Returns (seconds, algorithmic bytes of the sample, threads, number
    of sequences, the sampled sequence ids, the oracle's outputs per layer)."""
    import oracle
    from paged_kv_decode_04_gb300 import synth
    rng = np.random.default_rng(rng_seed)
    seqs = np.sort(rng.choice(w.batch, size=min(n_seqs, w.batch), replace=False))
    threads = threads or oracle.default_threads()
    comps = [synth.compact(w, layer, seqs) for layer in range(w.layers)]
    refs = []
    t0 = time.perf_counter()
    for c in comps:
        oracle.kv_append(c.k_new, c.v_new, c.pool, c.block_table, c.positions,
                         page_size=w.page_size, theta=w.rope_theta)
        refs.append(oracle.decode_attention(c.q, c.pool, c.block_table, c.seq_lens,
                                            num_kv_heads=w.num_kv_heads, page_size=w.page_size,
                                            scale=w.scale, threads=threads))
    dt = time.perf_counter() - t0
    sub = synth.Workload(
        name=w.name, seed=w.seed, layers=w.layers, batch=len(seqs), num_pages=w.num_pages,
        seq_lens=w.seq_lens[seqs], block_tables=w.block_tables[:, seqs], live_pages=w.live_pages,
        page_data=w.page_data[:0], q=w.q[:, seqs], k_new=w.k_new[:, seqs],
        v_new=w.v_new[:, seqs])
    return dt, algorithmic_bytes(sub, "step"), threads, len(seqs), seqs, refs


# ------------------------------------------------------------------ main --

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from paged_kv_decode_04_gb300 import synth
    w = synth.make_workload(args.workload, args.seed)
    n_seqs = args.ref_seqs
    for _ in range(args.warmup):
        oracle_sample_run(w, n_seqs, 1)
    total_t = 0.0
    total_b = 0
    threads = 1
    for k in range(args.steps):
        dt, nb, threads, used, _, _ = oracle_sample_run(w, n_seqs, 100 + k)
        total_t += dt
        total_b += nb
    value = total_b / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "seed": args.seed,
                   "sample": f"{used} of {w.batch} sequences x {w.layers} layer(s) per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{used} of {w.batch} sequences per step, FP64 C oracle, "
                                   f"{threads} threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import torch
    from paged_kv_decode_04_gb300 import binding, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    w = synth.make_workload(args.workload, args.seed, num_pages=args.pool_pages)
    d = synth.device_inputs(w, dev)
    B, layers = w.batch, w.layers
    stream = torch.cuda.current_stream(dev)
    planned = args.plan in ("host", "lengths")
    # the host plan is built from the lengths and layer 0's tables (shared
    # prefixes become shared-prefix items); the workloads share the same runs
    # of pages in every layer, so it serves every layer
    plan_kw = {"block_tables": w.block_tables[0]} if args.plan == "host" else {}
    plan = binding.Plan(w.seq_lens, w.max_blocks, device=dev, **plan_kw) if planned else None
    plan_build_us = None
    if planned:
        # host cost of planning one step (a serving loop builds one plan per step)
        t = time.perf_counter()
        for _ in range(200):
            binding.Plan(w.seq_lens, w.max_blocks, **plan_kw)
        plan_build_us = round((time.perf_counter() - t) / 200 * 1e6, 2)
    if planned:
        d["plan"] = plan.dev
        splits = max(1, max((int(m[2]) for m in plan.merges()), default=1))
        ws_bytes = plan.workspace_bytes
        split_text = (f"host work plan: {plan.num_items} items of at most {plan.range_pages} "
                      f"pages or 4 packed sequences, {plan.num_merges} merged sequences")
        if plan.num_shared:
            split_text += (f", {plan.num_shared} shared-prefix items of at most "
                           f"{plan.shared_pages} pages")
    else:
        splits = binding.plan_splits(B, w.max_blocks, args.splits)
        ws_bytes = binding.workspace_bytes(B, w.max_blocks, args.splits)
        split_text = f"fixed: {splits} ranges per sequence"
    workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    outs = torch.empty((layers, B, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    fused = args.path == "fused"
    merges = (plan.num_merges > 0) if planned else (splits > 1)
    launched = binding.attention_kernels(B, w.max_blocks, args.splits, plan)
    kernels_per_layer = ((1 if fused else 2) + (1 if merges else 0)
                         + (1 if planned and plan.num_shared else 0))

    def plan_for(dset):
        """The plan whose device copy is dset["plan"] (one per input set)."""
        if not planned:
            return None
        if dset["plan"] is plan.dev:
            return plan
        p2 = copy.copy(plan)
        p2.dev = dset["plan"]
        return p2

    def attend_on(dset, layer, out):
        if planned:
            binding.paged_decode_attention_planned(
                dset["q"][layer], d["pool"], dset["block_tables"][layer], dset["seq_lens"],
                plan_for(dset), out, scale=w.scale, workspace=workspace, dev_err=err)
        else:
            binding.paged_decode_attention(
                dset["q"][layer], d["pool"], dset["block_tables"][layer], dset["seq_lens"], out,
                scale=w.scale, workspace=workspace, num_splits=args.splits, dev_err=err)

    def fused_on(dset, layer, out):
        if planned:
            binding.decode_step_planned(
                dset["q"][layer], dset["k_new"][layer], dset["v_new"][layer], d["pool"],
                dset["block_tables"][layer], dset["seq_lens"], plan_for(dset), out,
                rope_theta=w.rope_theta, scale=w.scale, workspace=workspace, dev_err=err)
        else:
            binding.decode_step(
                dset["q"][layer], dset["k_new"][layer], dset["v_new"][layer], d["pool"],
                dset["block_tables"][layer], dset["seq_lens"], out, rope_theta=w.rope_theta,
                scale=w.scale, workspace=workspace, num_splits=args.splits, dev_err=err)

    def append_on(dset, layer):
        binding.kv_append(dset["k_new"][layer], dset["v_new"][layer], d["pool"],
                          dset["block_tables"][layer], dset["positions"], rope_theta=w.rope_theta,
                          dev_err=err)

    def attend(layer):
        attend_on(d, layer, outs[layer])

    def append(layer):
        append_on(d, layer)

    def fused_layer(layer):
        fused_on(d, layer, outs[layer])

    def launch_step():
        """Enqueue one whole step (every layer) on the current stream."""
        for layer in range(layers):
            if fused:
                fused_layer(layer)
            else:
                append(layer)
                attend(layer)

    # ---- warm-up (eager), then optionally capture one step as a CUDA graph
    for _ in range(args.warmup):
        launch_step()
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} during warm-up")
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            launch_step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)
        run_step = graph.replay
    else:
        run_step = launch_step

    # ---- timed region: K whole steps, device-resident inputs
    sampler = ClockSampler(gpu_selector(local)) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        run_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    if sampler:
        sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    step_bytes = algorithmic_bytes(w, "step")
    total_bytes = sum_over_ranks(step_bytes * args.steps, world, dev)
    value = total_bytes / (ms / 1e3) / 1e9
    ms_per_step = ms / args.steps

    # ---- per-kernel durations: CUDA events around each launch on the same stream.
    # The launches are queued in chunks behind a short fixed-length busy kernel
    # (torch.cuda._sleep) so that the host is ahead of the GPU and the events
    # see back-to-back kernels, not the host's launch pace.
    n_prof = min(args.steps, max(50, args.steps // 4))
    kern = {}
    chunk = 64

    def prequeue(i):
        if i % chunk == 0:
            torch.cuda._sleep(int(2e9 * 100e-6 * min(chunk, n_prof - i) * layers))

    if fused:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_prof)]
        for i in range(n_prof):
            prequeue(i)
            ev[i][0].record(stream)
            for layer in range(layers):
                fused_layer(layer)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        per = [e[0].elapsed_time(e[1]) / layers for e in ev]
        dom_ms = statistics.mean(per)
        kern["decode_step_median"] = round(statistics.median(per) * 1e3, 2)
        dom_bytes = algorithmic_bytes(w, "step") / layers
        kern["decode_step"] = round(dom_ms * 1e3, 2)
        dom_name = launched + " (fused step)"
    else:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_prof)]
        for i in range(n_prof):
            prequeue(i)
            ev[i][0].record(stream)
            for layer in range(layers):
                append(layer)
            ev[i][1].record(stream)
            for layer in range(layers):
                attend(layer)
            ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
        app_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / layers
        dom_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) / layers
        dom_bytes = algorithmic_bytes(w, "attention") / layers
        kern["kv_append"] = round(app_ms * 1e3, 2)
        kern["paged_decode_attention"] = round(dom_ms * 1e3, 2)
        dom_name = launched + " (attention)"
    peak, peak_kind = measured_hbm_peak()
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    duration_source = "CUDA events around each launch, in a separate pass of the same loop"
    if fused and kernels_per_layer == 1:
        # the timed steps are this one kernel, `layers` launches per step back to back: its
        # average launch duration is the timed region's own CUDA-event time per launch (the
        # separate pass above puts an event record between launches, which keeps each launch
        # from starting before the previous one has finished)
        dom_ms = ms_per_step / layers
        kern["decode_step_timed_region"] = round(dom_ms * 1e3, 2)
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        duration_source = "timed region: CUDA events around the K steps, which are this kernel alone"

    # ---- end to end: per-step inputs from pinned host memory, output back to host.
    # Two device copies of the per-step inputs and outputs alternate, so the
    # copies of step k+1 (and the read-back of step k) run on a copy stream
    # while step k computes; every step still moves its own inputs in and its
    # output out inside the timed region.  (Three sets on separate upload and
    # read-back streams measured no better: short steps are bound by the
    # host's per-step stream calls.)
    names = ["q", "k_new", "v_new", "positions", "seq_lens", "block_tables"]
    if planned:
        names.append("plan")                  # the step's work plan travels with its inputs
    # One pinned host buffer holds all of a step's inputs, each at a 256-byte
    # aligned offset; a step moves it with one copy into one of two device
    # buffers, and the step's graph reads views of that buffer.
    layout, total = [], 0
    for k in names:
        nb = d[k].numel() * d[k].element_size()
        layout.append((k, total, nb, d[k].dtype, tuple(d[k].shape)))
        total += (nb + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k, off, nb, _, _ in layout:
        host_buf[off:off + nb].copy_(d[k].reshape(-1).view(torch.uint8).cpu())
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    sets = [{k: buf[off:off + nb].view(dt).view(shape) for k, off, nb, dt, shape in layout}
            for buf in dev_bufs]
    for dset in sets:
        for k in names:
            dset[k].copy_(d[k])
    out_host = [torch.empty(outs.shape, dtype=outs.dtype).pin_memory() for _ in range(2)]
    h2d = total
    d2h = out_host[0].numel() * out_host[0].element_size()
    set_outs = [outs, torch.empty_like(outs)]

    def make_step(dset, out):
        def launch():
            for layer in range(layers):
                if fused:
                    fused_on(dset, layer, out[layer])
                else:
                    append_on(dset, layer)
                    attend_on(dset, layer, out[layer])
        if not args.graph:
            return launch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            launch()
        return g.replay

    steps_e2e = [make_step(sets[i], set_outs[i]) for i in range(2)]
    copy_stream = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, computed, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e_ in computed + out_done:
        e_.record(stream)

    def h2d_into(i):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(computed[i])     # the last step that read set i is done
            dev_bufs[i].copy_(host_buf, non_blocking=True)
            in_ready[i].record(copy_stream)

    def run_e2e(n):
        h2d_into(0)
        for k in range(n):
            i = k % 2
            stream.wait_event(in_ready[i])
            stream.wait_event(out_done[i])           # read-back of step k-2 left set_outs[i]
            steps_e2e[i]()
            computed[i].record(stream)
            if k + 1 < n:
                h2d_into(1 - i)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(computed[i])
                out_host[i].copy_(set_outs[i], non_blocking=True)
                out_done[i].record(copy_stream)
        stream.wait_stream(copy_stream)

    run_e2e(max(3, min(args.warmup, 20)))
    torch.cuda.synchronize(dev)
    barrier(world)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    run_e2e(args.steps)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev)
    e2e_value = sum_over_ranks(step_bytes * args.steps, world, dev) / (e2e_ms / 1e3) / 1e9
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} during the timed runs")

    # ---- CPU baseline: the oracle on a bounded sample of the same workload
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # repeat the bounded sample until it has used about 10 s of CPU time
        dt, nb, threads, used, seqs, refs = oracle_sample_run(w, args.cpu_seqs)
        reps = 1
        while dt * threads < 10.0 and reps < 30:
            dt2, nb2, _, _, _, _ = oracle_sample_run(w, args.cpu_seqs)
            dt, nb, reps = dt + dt2, nb + nb2, reps + 1
        cpu = {"value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": f"{used} of {w.batch} sequences x {w.layers} layer(s), {reps} time(s): "
                         f"FP64 append + two-pass attention, {dt:.2f} s wall on {threads} "
                         f"threads ({dt * threads:.1f} CPU-s)"}
        # the same sample, set against the GPU's outputs of the timed steps
        # (every step recomputes the same outputs from the same inputs)
        got = outs.view(torch.int16).cpu().numpy().view(np.uint16)[:, seqs]
        got = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ref = np.stack(refs)
        err = np.abs(got - ref)
        cpu["parity_vs_gpu"] = {
            "max_abs_err": float(err.max()),
            "worst_err_over_tolerance": float((err / (1e-3 + 8e-3 * np.abs(ref))).max()),
            "tolerance": "|err| <= 1e-3 + 8e-3 |ref|"}

    if rank != 0:
        return 0
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    traffic = recorded_traffic(args.workload, dom_name)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "storage_dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": WORKLOAD_TEXT[args.workload], "seed": args.seed,
            "path": ("fused append+attention (pkv_decode_step)" if fused
                     else "pkv_kv_append then pkv_paged_decode_attention"),
            "launch": "one CUDA graph per step" if args.graph else "eager launches",
            "num_splits": splits, "split_plan": split_text,
            "plan_build_us_host": plan_build_us,
            "layers_per_step": layers, "pool_pages": w.num_pages,
            "l2": ("inputs larger than L2: %.2f GiB of K/V streamed per step vs 129 MB L2; no flush"
                   % (w.kv_bytes() / 2 ** 30)) if w.kv_bytes() > 512 * 2 ** 20 else
                  "working set fits in L2 (no flush): L2-resident figure",
            "parallelism": f"replicas x{world}",
        },
        "steps_per_s": round(1e3 / ms_per_step * world, 1),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_copy": round(100 * value / world / peak, 2),
        "algorithmic_bytes_per_step": step_bytes,
        "kernels_us": kern,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": dom_name, "peak_kind": f"{peak_kind} copy bandwidth",
                     "bytes_per_launch": dom_bytes, "duration_source": duration_source},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 5),
                "pipelining": "copies of step k+1 and read-back of step k overlap step k; "
                              "a step's inputs travel as one packed copy"},
        "gpu_launches": kernels_per_layer * layers * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_prefill(args, world, rank, local):
    """Throughput of the paged prefill write: 256 prompts x 2047 tokens per call."""
    import torch
    from paged_kv_decode_04_gb300 import binding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    B, L, num_pages = 256, 2047, 40000
    g = torch.Generator(device=dev).manual_seed(args.seed)
    perm = torch.randperm(num_pages, generator=g, device=dev)[:B * 128].view(B, 128).int()
    k = torch.randn((B * L, 8, 64), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((B * L, 8, 64), generator=g, device=dev).to(torch.bfloat16)
    off = torch.arange(0, B * L + 1, L, dtype=torch.int32, device=dev)
    st = torch.zeros(B, dtype=torch.int32, device=dev)
    pool = torch.full((num_pages, 2, 16, 8, 64), -1, dtype=torch.int16, device=dev).view(
        torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        binding.kv_write_prefill(k, v, off, st, pool, perm, dev_err=err)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    T = B * L
    step_bytes = T * 8 * 64 * 2 * 2 * 2 + (B + 1) * 4 + B * 4 + B * 128 * 4
    value = sum_over_ranks(step_bytes * args.steps, world, dev) / (ms / 1e3) / 1e9
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())}")
    if rank == 0:
        peak, kind = measured_hbm_peak()
        print(json.dumps({
            "metric": "paged prefill write achieved HBM GB/s", "value": round(value, 2),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "storage_dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"prefill write: {B} prompts x {L} tokens, 32q/8kv/64 bf16, "
                                   f"{num_pages}-page pool", "seed": args.seed},
            "algorithmic_bytes_per_step": step_bytes,
            "roofline": {"bound": "hbm", "achieved": round(value / world, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(value / world / peak, 4),
                         "traffic": None, "kernel": "kv_write_prefill_kernel",
                         "peak_kind": f"{kind} copy bandwidth"},
            "gpu_launches": args.steps}), flush=True)
    return 0


def run_serve(args, world, rank, local):
    """Continuous-batching serving simulation driven by the host scheduler."""
    import torch
    from paged_kv_decode_04_gb300.engine import Engine

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    rng = np.random.default_rng(args.seed)
    layers, num_pages = 16, 65536
    reqs = [(int(rng.integers(16, 1025)), int(rng.integers(16, 513)))
            for _ in range(args.serve_requests)]
    use_plan = args.plan != "auto"
    warm = Engine(num_pages, layers, dev, static_batching=args.static, seed=args.seed + 1,
                  use_plan=use_plan)
    warm_iters = warm.run(reqs[:8])["iterations"]   # a warm-up run of 8 requests
    eng = Engine(num_pages, layers, dev, static_batching=args.static, seed=args.seed,
                 use_plan=use_plan)
    barrier(world)
    res = eng.run(reqs)
    barrier(world)
    secs = max_over_ranks(res["seconds"], world, dev)
    toks = sum_over_ranks(res["decode_tokens"], world, dev)
    if rank == 0:
        st = res["stats"]
        print(json.dumps({
            "metric": "serving simulation decode tokens/s (scheduler-driven, 16 layers)",
            "value": round(toks / secs, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": res["iterations"], "warmup": warm_iters, "ms_per_step": round(secs / res["iterations"] * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "storage_dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{len(reqs)} requests, prompt U[16,1024], max_new U[16,512], "
                                   f"{layers} layers, {num_pages}-page pool (2 GiB), "
                                   f"{'static' if args.static else 'continuous'} batching",
                       "split_plan": "host work plan per step" if use_plan else "fixed (automatic)",
                       "seed": args.seed},
            "stats": {k: st[k] for k in ("pool_pages", "peak_active", "largest_decode_batch",
                                         "peak_allocated_pages", "admission_wait_total",
                                         "admission_wait_max", "free_pages", "rejected",
                                         "finished")},
            "wall_s": round(secs, 3)}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOAD_TEXT), default="peak")
    ap.add_argument("--splits", type=int, default=0, help="0 = automatic split plan")
    ap.add_argument("--plan", choices=["auto", "host", "lengths"], default="host",
                    help="host (default): a work plan built on the host from the lengths and "
                         "the block tables, shared prefixes as shared-prefix items "
                         "(pkv_plan_build_shared), passed to the planned entry points; "
                         "lengths: the plan from the lengths alone (pkv_plan_build), as the "
                         "serving engine builds it; auto: the fixed automatic split plan")
    ap.add_argument("--path", choices=["fused", "separate"], default="fused",
                    help="fused: one pkv_decode_step launch per layer; separate: pkv_kv_append "
                         "then pkv_paged_decode_attention")
    ap.add_argument("--graph", action=argparse.BooleanOptionalAction, default=True,
                    help="replay each step as one captured CUDA graph")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seqs", type=int, default=256,
                    help="sequences of the CPU-oracle baseline sample")
    ap.add_argument("--ref-seqs", type=int, default=1,
                    help="sequences per step of the --impl reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=["decode", "prefill", "serve"], default="decode",
                    help="decode: the decode step (headline); prefill: the paged prefill write; "
                         "serve: scheduler-driven serving simulation")
    ap.add_argument("--serve-requests", type=int, default=512)
    ap.add_argument("--pool-pages", type=int, default=None,
                    help="override the workload's pool size in pages (same live pages, denser pool)")
    ap.add_argument("--static", action="store_true", help="serve: static instead of continuous")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.op == "prefill":
        return run_prefill(args, world, rank, local)
    if args.op == "serve":
        return run_serve(args, world, rank, local)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
