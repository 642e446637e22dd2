"""Benchmark of the paged-KV decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload peak] [--impl ours|reference]

One step = the whole decode hot path for one batch: the KV append (RoPE on the
new keys, K/V written into their page slots) followed by paged decode
attention (plus the split merge when the plan splits), for every layer of the
workload.  The default workload is 256 sequences x 2048 tokens of context,
one layer, 32 query / 8 kv heads, head dim 64, 32768 live pages randomly
scattered in a 40000-page pool.

Prints one JSON line.  `value` is achieved algorithmic HBM GB/s of the whole
step with all inputs resident in device memory (the median of repeated timed
regions of K steps); `e2e` repeats the measurement through the same public
calls with the per-step work plan built on the host, the per-step inputs
copied from pinned host memory and the output copied back inside the timed
region.  `per_workload` measures the other workloads (tiny, long, small, mix,
prefix, the prefill write) the same way, each checked element by element
against the FP64 oracle on every output.  `--impl reference` times the FP64
CPU oracle on the host cores instead (a deliberately slow baseline, not a
target).  Multi-GPU runs (torchrun) are independent replicas, one per rank
(weak scaling): the path has no exchange step.
"""
from __future__ import annotations

import argparse
import copy
import hashlib
import json
import math
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
    "paged_decode_kernel": ("decode_attention.cu",),
    "merge_plan_kernel": ("decode_attention.cu",),
    "merge_splits_kernel": ("decode_attention.cu",),
    "paged_decode_pagebox_kernel": ("decode_pagebox.cu",),
    "paged_decode_shared_kernel": ("decode_shared.cu",),
    "paged_decode_segments_kernel": ("decode_segments.cu",),
}
COMMON_SOURCES = ("decode_page.cuh", "pkv_device.cuh", "pkv_internal.h")
KERNEL_SOURCES = [os.path.join(CSRC, f)
                  for f in sorted({f for fs in KERNEL_FILES.values() for f in fs})
                  + list(COMMON_SOURCES)]
# The traffic file holds a list of records {workload, kernel, kernel_sha, dram_bytes_per_launch};
# kernel_sha covers the sources of the kernels the record names.
# Every kernel of the library, for the per-kernel shares of a step.
LIBRARY_KERNELS = ("paged_decode_segments_kernel", "paged_decode_pagebox_kernel",
                   "paged_decode_shared_kernel",
                   "paged_decode_kernel", "merge_plan_kernel", "merge_splits_kernel",
                   "kv_append_kernel", "kv_write_prefill_kernel", "rope_table_kernel",
                   "rope_tag_kernel")

WORKLOAD_TEXT = {
    "peak": "peak: 256 seqs x 2048 ctx, 1 layer, 32q/8kv/64 bf16, 32768 live pages (1 GiB K/V) "
            "randomly scattered in a 40000-page pool",
    "mix": "mix: 128 seqs (115 of 16-128, 13 of 1536-2048 tokens), 16 layers with per-layer "
           "tables, 32q/8kv/64 bf16, 8 GiB pool",
    "long": "long: 1 seq x 2048 ctx x 16 layers, 32q/8kv/64 bf16, shuffled pages, 4096-page pool",
    "small": "small: 8 seqs, lengths U[1,2048], 1 layer, 4096-page pool",
    "tiny": "tiny: 1 seq x 37 ctx, 1 layer, 64-page pool",
    "prefix": "prefix: 256 seqs x 2048 ctx, groups of 16 share a 1536-token prefix (96 aliased "
              "pages) + 32 private pages each, 9728 live pages in a 40000-page pool",
}
# The workloads measured next to the headline (in this order), then the prefill write.
PER_WORKLOADS = ("tiny", "long", "small", "mix", "prefix")
PREFILL_TEXT = "prefill write: 256 prompts x 2047 tokens, 8 kv heads x 64 bf16, 40000-page pool"
# Repeated timed regions: at least this many, and for at least this long (the
# clock sampler then sees the whole span).
MIN_REPEATS = 10
MIN_TIMED_SECONDS = 1.5
MAX_REPEATS = 5000
# Spin (clock cycles, about 50 us) that holds the stream after each L2 flush
# while the host queues the next step.
FLUSH_SPIN_CYCLES = 100000
E2E_MIN_STEPS = 500   # steps per end-to-end region, at least
E2E_REGIONS = 3
TOL_ABS, TOL_REL = 1e-3, 8e-3


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


def unique_bytes(w) -> int:
    """algorithmic_bytes(w) with each physical page's K/V counted once per
    layer (the tokens it holds for the longest sequence naming it): the bytes
    a step must read from DRAM when sequences share prefix pages."""
    Hkv, D, P = w.num_kv_heads, w.head_dim, w.page_size
    total = algorithmic_bytes(w, "step") - int(w.seq_lens.astype(np.int64).sum()) * Hkv * D * 4 \
        * w.layers
    for layer in range(w.layers):
        tokens = {}
        for b in range(w.batch):
            L = int(w.seq_lens[b])
            for k, p in enumerate(w.pages_of(layer, b)):
                tokens[int(p)] = max(tokens.get(int(p), 0), min(P, L - k * P))
        total += sum(tokens.values()) * Hkv * D * 4
    return total


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
    files = sorted({f for n in names if n in KERNEL_FILES for f in KERNEL_FILES[n]})
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


def spread(times_ms, steps):
    """Median / min / max of per-step times (ms) over repeated timed regions."""
    per = sorted(t / steps for t in times_ms)
    med = statistics.median(per)
    return {"repeats": len(per), "steps_per_repeat": steps, "ms_per_step_median": round(med, 6),
            "ms_per_step_min": round(per[0], 6), "ms_per_step_max": round(per[-1], 6),
            "spread_pct": round(100.0 * (per[-1] - per[0]) / med, 2)}


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
                "span_s": round(t1 - t0, 3),
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

def oracle_sample_run(w, n_seqs: int, rng_seed: int = 0, threads: int = 0,
                      want_slots: bool = False):
    """Time the FP64 oracle on n_seqs sequences of every layer (append + attention).

    The sample's inputs are relabelled into compact host copies first (not
    timed).  Returns (seconds, algorithmic bytes of the sample, threads, number
    of sequences, the sampled sequence ids, the oracle's outputs per layer);
    with want_slots, also the appended K and V rows per layer ([n][2][Hkv][D]
    bits, from the oracle's pool after its append)."""
    import oracle
    from paged_kv_decode_04_gb300 import synth
    if n_seqs >= w.batch:
        seqs = np.arange(w.batch)
    else:
        rng = np.random.default_rng(rng_seed)
        seqs = np.sort(rng.choice(w.batch, size=n_seqs, replace=False))
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
    res = (dt, algorithmic_bytes(sub, "step"), threads, len(seqs), seqs, refs)
    if not want_slots:
        return res
    slots = []
    for c in comps:
        rows = np.zeros((len(seqs), 2, w.num_kv_heads, w.head_dim), dtype=np.uint16)
        for r in range(len(seqs)):
            pos = int(c.positions[r])
            if pos >= 0:
                rows[r] = c.pool[c.block_table[r, pos // w.page_size], :, pos % w.page_size]
        slots.append(rows)
    return res + (slots,)


def parity_report(got_bits, refs):
    """Element-wise check of bf16 outputs against the oracle (float64)."""
    got = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = np.stack(refs)
    err = np.abs(got - ref)
    with np.errstate(invalid="ignore"):
        over = err / (TOL_ABS + TOL_REL * np.abs(ref))
    worst = float(np.nanmax(over)) if over.size else 0.0
    if not np.all(np.isfinite(got)):
        worst = float("inf")
    return {"outputs_checked": int(ref.size), "max_abs_err": float(np.nanmax(err)) if err.size
            else 0.0, "worst_err_over_tolerance": round(worst, 5),
            "tolerance": "|err| <= 1e-3 + 8e-3 |ref|", "within_tolerance": bool(worst <= 1.0)}


# ------------------------------------------------------------ the decode --

class DecodeBench:
    """One workload resident on the device with everything a timed step needs:
    the plan, workspace, outputs, the step as a CUDA graph, and the
    measurements (repeated timed regions, per-launch events, e2e)."""

    def __init__(self, w, args, dev, *, world=1, plan_mode=None):
        import torch
        from paged_kv_decode_04_gb300 import binding, synth
        self.torch, self.binding, self.synth = torch, binding, synth
        self.w, self.args, self.dev, self.world = w, args, dev, world
        self.d = synth.device_inputs(w, dev)
        self.stream = torch.cuda.current_stream(dev)
        self.plan_mode = plan_mode or args.plan
        self.planned = self.plan_mode in ("host", "lengths")
        # the host plan is built from the lengths and layer 0's tables (shared
        # prefixes become shared-prefix items); the workloads share the same
        # runs of pages in every layer, so it serves every layer
        self.plan_kw = ({"block_tables": w.block_tables[0]} if self.plan_mode == "host" else {})
        B = w.batch
        if self.planned:
            self.plan = binding.Plan(w.seq_lens, w.max_blocks, device=dev, **self.plan_kw)
            self.d["plan"] = self.plan.dev
            ws_bytes = self.plan.workspace_bytes
            p = self.plan
            self.split_text = (f"host work plan: {p.num_items} items of at most {p.range_pages} "
                               f"pages or 4 packed sequences, {p.num_merges} merged sequences")
            if p.num_shared:
                self.split_text += (f", {p.num_shared} shared-prefix items of at most "
                                    f"{p.shared_pages} pages")
            self.splits = max(1, max((int(m[2]) for m in p.merges()), default=1))
        else:
            self.plan = None
            self.splits = binding.plan_splits(B, w.max_blocks, args.splits)
            ws_bytes = binding.workspace_bytes(B, w.max_blocks, args.splits)
            self.split_text = f"fixed: {self.splits} ranges per sequence"
        self.workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.outs = torch.empty((w.layers, B, w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                                device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.fused = args.path == "fused"
        merges = (self.plan.num_merges > 0) if self.planned else (self.splits > 1)
        self.launched = binding.attention_kernels(B, w.max_blocks, args.splits, self.plan)
        self.kernels_per_layer = ((1 if self.fused else 2) + (1 if merges else 0)
                                  + (1 if self.planned and self.plan.num_shared else 0))
        self.run_step = self.launch_step

    # -- launches
    def plan_for(self, dset):
        """The plan whose device copy is dset["plan"] (one per input set)."""
        if not self.planned:
            return None
        if dset["plan"] is self.plan.dev:
            return self.plan
        p2 = copy.copy(self.plan)
        p2.dev = dset["plan"]
        return p2

    def fused_on(self, dset, layer, out):
        w, b, d = self.w, self.binding, self.d
        if self.planned:
            b.decode_step_planned(
                dset["q"][layer], dset["k_new"][layer], dset["v_new"][layer], d["pool"],
                dset["block_tables"][layer], dset["seq_lens"], self.plan_for(dset), out,
                rope_theta=w.rope_theta, scale=w.scale, workspace=self.workspace,
                dev_err=self.err)
        else:
            b.decode_step(
                dset["q"][layer], dset["k_new"][layer], dset["v_new"][layer], d["pool"],
                dset["block_tables"][layer], dset["seq_lens"], out, rope_theta=w.rope_theta,
                scale=w.scale, workspace=self.workspace, num_splits=self.args.splits,
                dev_err=self.err)

    def append_on(self, dset, layer):
        self.binding.kv_append(dset["k_new"][layer], dset["v_new"][layer], self.d["pool"],
                               dset["block_tables"][layer], dset["positions"],
                               rope_theta=self.w.rope_theta, dev_err=self.err)

    def attend_on(self, dset, layer, out):
        w, b, d = self.w, self.binding, self.d
        if self.planned:
            b.paged_decode_attention_planned(
                dset["q"][layer], d["pool"], dset["block_tables"][layer], dset["seq_lens"],
                self.plan_for(dset), out, scale=w.scale, workspace=self.workspace,
                dev_err=self.err)
        else:
            b.paged_decode_attention(
                dset["q"][layer], d["pool"], dset["block_tables"][layer], dset["seq_lens"], out,
                scale=w.scale, workspace=self.workspace, num_splits=self.args.splits,
                dev_err=self.err)

    def launch_on(self, dset, out):
        """Enqueue one whole step (every layer) on the current stream."""
        for layer in range(self.w.layers):
            if self.fused:
                self.fused_on(dset, layer, out[layer])
            else:
                self.append_on(dset, layer)
                self.attend_on(dset, layer, out[layer])

    def launch_step(self):
        self.launch_on(self.d, self.outs)

    def warm_and_capture(self, warmup, graph):
        torch = self.torch
        for _ in range(warmup):
            self.launch_step()
        torch.cuda.synchronize(self.dev)
        self.check_err("warm-up")
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.launch_step()
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(self.dev)
            self.graph = g
            self.run_step = g.replay

    def check_err(self, when):
        if int(self.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(self.err.item())} during the {when} "
                               f"({self.w.name} workload)")

    # -- timing
    def one_region(self, steps, flush=None):
        """CUDA-event time (ms) of `steps` steps on the launching stream, with a
        barrier and a synchronize on both sides; with `flush` (a device buffer
        larger than L2), L2 is flushed before every step, outside the per-step
        event pairs, and the region's time is the sum of the step events.  After
        each flush a short spin kernel holds the stream while the host queues
        the step and its events, so a step's events time its kernels on the
        device, not the host's launch of them."""
        torch = self.torch
        barrier(self.world)
        torch.cuda.synchronize(self.dev)
        if flush is None:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for _ in range(steps):
                self.run_step()
            e1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            ms = e0.elapsed_time(e1)
        else:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
            for i in range(steps):
                flush.fill_(i & 0xFF)
                torch.cuda._sleep(FLUSH_SPIN_CYCLES)
                ev[i][0].record(self.stream)
                self.run_step()
                ev[i][1].record(self.stream)
            torch.cuda.synchronize(self.dev)
            ms = sum(a.elapsed_time(b) for a, b in ev)
        barrier(self.world)
        return max_over_ranks(ms, self.world, self.dev)

    def timed(self, steps, flush=None, min_seconds=None):
        """Repeated timed regions of `steps` steps: at least --min-repeats of
        them and at least min_seconds (--repeat-seconds) in all (the count is
        fixed from a probe region, the same on every rank).  Returns (region
        times in ms, wall t0, t1)."""
        if min_seconds is None:
            min_seconds = self.args.repeat_seconds
        probe = self.one_region(steps, flush)
        per_region_s = max(probe, 1e-3) / 1e3
        if flush is not None:
            per_region_s += steps * 1.7e-4         # the flushes and spins between steps
        reps = int(min(MAX_REPEATS, max(self.args.min_repeats,
                                        math.ceil(min_seconds / per_region_s))))
        t0 = time.time()
        times = [self.one_region(steps, flush) for _ in range(reps)]
        return times, t0, time.time()

    def per_launch(self, steps):
        """Per-launch CUDA events in a separate pass of the same loop (the
        launches queued behind a short busy kernel so the events time
        back-to-back kernels, not the host's launch pace)."""
        torch = self.torch
        layers = self.w.layers
        n_prof = min(steps, max(50, steps // 4))
        chunk = 64
        kern = {}

        def prequeue(i):
            if i % chunk == 0:
                torch.cuda._sleep(int(2e9 * 100e-6 * min(chunk, n_prof - i) * layers))

        if self.fused:
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_prof)]
            for i in range(n_prof):
                prequeue(i)
                ev[i][0].record(self.stream)
                for layer in range(layers):
                    self.fused_on(self.d, layer, self.outs[layer])
                ev[i][1].record(self.stream)
            torch.cuda.synchronize(self.dev)
            per = [e[0].elapsed_time(e[1]) / layers for e in ev]
            dom_ms = statistics.mean(per)
            kern["decode_step_median"] = round(statistics.median(per) * 1e3, 2)
            kern["decode_step"] = round(dom_ms * 1e3, 2)
            dom_bytes = algorithmic_bytes(self.w, "step") / layers
            dom_name = self.launched + " (fused step)"
        else:
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_prof)]
            for i in range(n_prof):
                prequeue(i)
                ev[i][0].record(self.stream)
                for layer in range(layers):
                    self.append_on(self.d, layer)
                ev[i][1].record(self.stream)
                for layer in range(layers):
                    self.attend_on(self.d, layer, self.outs[layer])
                ev[i][2].record(self.stream)
            torch.cuda.synchronize(self.dev)
            app_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / layers
            dom_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) / layers
            kern["kv_append"] = round(app_ms * 1e3, 2)
            kern["paged_decode_attention"] = round(dom_ms * 1e3, 2)
            dom_bytes = algorithmic_bytes(self.w, "attention") / layers
            dom_name = self.launched + " (attention)"
        return kern, dom_ms, dom_bytes, dom_name

    def kernel_shares(self, n=20):
        """Each library kernel's share of the device time of n eager steps,
        from the CUPTI kernel records torch.profiler collects (a ratio; no
        duration taken under the profiler is reported).  Kernels launched with
        programmatic dependent launch start before the previous kernel ends and
        wait for it on the device, so a kernel is charged only for the time
        after every earlier-started kernel has ended (the serialised
        timeline)."""
        torch = self.torch
        try:
            from torch.autograd import DeviceType
            from torch.profiler import ProfilerActivity, profile
            with profile(activities=[ProfilerActivity.CUDA]):   # initialises CUPTI
                self.launch_step()
                torch.cuda.synchronize(self.dev)
            with profile(activities=[ProfilerActivity.CUDA]) as prof:
                for _ in range(n):
                    self.launch_step()
                torch.cuda.synchronize(self.dev)
            pat = re.compile(r"\b(" + "|".join(LIBRARY_KERNELS) + r")\b")
            spans = []
            for ev in prof.events():
                if getattr(ev, "device_type", DeviceType.CUDA) != DeviceType.CUDA:
                    continue
                m = pat.search(ev.name)
                if m:
                    spans.append((ev.time_range.start, ev.time_range.end, m.group(1)))
            spans.sort()
            excl, last_end = {}, -math.inf
            for t0, t1, name in spans:
                s0 = max(t0, last_end)
                excl[name] = excl.get(name, 0.0) + max(0.0, t1 - s0)
                last_end = max(last_end, t1)
            s = sum(excl.values())
            if s <= 0:
                return None
            return {k: round(v / s, 4) for k, v in sorted(excl.items(), key=lambda x: -x[1])}
        except Exception as exc:  # the profiler is optional on a box
            return {"unavailable": str(exc)[:120]}

    # -- end to end
    def e2e(self, steps, warmup):
        """The same step with every per-step input coming from pinned host
        memory and the output going back to it.  Each step the host builds the
        step's work plan from the host lengths (and tables) through the C ABI,
        straight into the pinned buffer that holds the step's packed inputs
        (q, k_new, v_new, positions, seq_lens, block tables, plan), then
        launches the step.  Two input sets alternate; the step of set s is one
        CUDA graph: the upload of the NEXT step's packed inputs (set 1 - s,
        one copy) runs beside this step's kernels, which are followed by the
        read-back of this step's output.  So every step moves its own inputs
        in and its output out, and the copies overlap the compute."""
        torch, w = self.torch, self.w
        names = ["q", "k_new", "v_new", "positions", "seq_lens", "block_tables"]
        layout, total = [], 0
        for k in names:
            nb = self.d[k].numel() * self.d[k].element_size()
            layout.append((k, total, nb, self.d[k].dtype, tuple(self.d[k].shape)))
            total += (nb + 255) // 256 * 256
        plan_off, plan_cap = total, 0
        lens_host = np.ascontiguousarray(w.seq_lens.astype(np.int32))
        bt_host = (np.ascontiguousarray(w.block_tables[0].astype(np.int32))
                   if self.plan_mode == "host" else None)
        if self.planned:
            plan_cap = self.binding.plan_bytes(w.batch, w.max_blocks)
            total = plan_off + (plan_cap + 255) // 256 * 256
        host_bufs = [torch.empty(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
        for hb in host_bufs:
            for k, off, nb, _, _ in layout:
                hb[off:off + nb].copy_(self.d[k].reshape(-1).view(torch.uint8).cpu())
        plans = [None, None]
        if self.planned:
            for i in range(2):
                view = host_bufs[i][plan_off:plan_off + plan_cap].numpy().view(np.int32)
                plans[i] = self.binding.Plan(lens_host, w.max_blocks, out=view, **self.plan_kw)
        n_copy = total if not self.planned else \
            plan_off + (plans[0].bytes_used + 255) // 256 * 256
        dev_bufs = [torch.empty(total, dtype=torch.uint8, device=self.dev) for _ in range(2)]
        sets = [{k: buf[off:off + nb].view(dt).view(shape) for k, off, nb, dt, shape in layout}
                for buf in dev_bufs]
        for i, dset in enumerate(sets):
            dev_bufs[i][:n_copy].copy_(host_bufs[i][:n_copy])
            if self.planned:
                dset["plan"] = dev_bufs[i][plan_off:plan_off + plans[i].bytes_used].view(
                    torch.int32)
        out_host = [torch.empty(self.outs.shape, dtype=self.outs.dtype).pin_memory()
                    for _ in range(2)]
        d2h = out_host[0].numel() * out_host[0].element_size()
        set_outs = [self.outs, torch.empty_like(self.outs)]
        side = torch.cuda.Stream(self.dev)

        def step_body(s):
            """The kernels of set s, and beside them the upload of set 1 - s
            (the next step's inputs) and the read-back of set 1 - s's output
            (the previous step's)."""
            cur = torch.cuda.current_stream(self.dev)   # the capture stream when capturing
            fork = torch.cuda.Event()
            fork.record(cur)
            side.wait_event(fork)
            with torch.cuda.stream(side):
                out_host[1 - s].copy_(set_outs[1 - s], non_blocking=True)
                dev_bufs[1 - s][:n_copy].copy_(host_bufs[1 - s][:n_copy], non_blocking=True)
            dset, out = sets[s], set_outs[s]
            for layer in range(w.layers):
                if self.fused:
                    self.fused_on(dset, layer, out[layer])
                else:
                    self.append_on(dset, layer)
                    self.attend_on(dset, layer, out[layer])
            cur.wait_stream(side)

        graphs = []
        for s in range(2):
            if self.args.graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    step_body(s)
                graphs.append(g.replay)
            else:
                graphs.append(lambda s=s: step_body(s))
        done = [torch.cuda.Event(), torch.cuda.Event()]
        plan_us = []

        def run_e2e(n):
            # the first step's inputs (set 0), then each step uploads the next one's
            dev_bufs[0][:n_copy].copy_(host_bufs[0][:n_copy], non_blocking=True)
            done[1].record(self.stream)
            for k in range(n):
                s = k % 2
                if self.planned:
                    # host buffer 1 - s is about to be uploaded again: its last
                    # upload (step k - 2's graph; for step 1 the first copy
                    # above) must be over before the plan of step k + 1 is
                    # built into it
                    if k >= 1:
                        done[s].synchronize()
                    t = time.perf_counter()
                    plans[1 - s].rebuild(lens_host, bt_host)
                    plan_us.append((time.perf_counter() - t) * 1e6)
                graphs[s]()
                done[s].record(self.stream)
            # the last step's output (the earlier ones were read back beside
            # the following step's kernels)
            out_host[(n - 1) % 2].copy_(set_outs[(n - 1) % 2], non_blocking=True)

        run_e2e(max(3, min(warmup, 20)))
        torch.cuda.synchronize(self.dev)
        plan_us.clear()
        # E2E_REGIONS regions of at least E2E_MIN_STEPS steps each (more when
        # --steps asks for more), so that the pipeline's fill and drain -- the
        # first step's upload and the last step's read-back, both inside each
        # region -- are a serving loop's share of it, not a 20-step job's
        n = max(steps, E2E_MIN_STEPS)
        region_ms = []
        for _ in range(E2E_REGIONS):
            barrier(self.world)
            torch.cuda.synchronize(self.dev)
            f0 = torch.cuda.Event(enable_timing=True)
            f1 = torch.cuda.Event(enable_timing=True)
            f0.record(self.stream)
            run_e2e(n)
            f1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            barrier(self.world)
            region_ms.append(max_over_ranks(f0.elapsed_time(f1), self.world, self.dev))
        e2e_ms = statistics.median(region_ms)
        self.check_err("end-to-end runs")
        if self.planned:
            for p in plans:       # the rebuilt plans are the plan the graphs were made with
                assert np.array_equal(p.host, self.plan.host)
        # (shared prefix pages once per step, as the device-resident value)
        step_bytes = unique_bytes(w) if w.name == "prefix" else algorithmic_bytes(w, "step")
        value = sum_over_ranks(step_bytes * n, self.world, self.dev) / (e2e_ms / 1e3) / 1e9
        rec = {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": n_copy,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / n, 5),
               "timing": {"regions": E2E_REGIONS, "steps_per_region": n,
                          "ms_per_step_median": round(e2e_ms / n, 6),
                          "ms_per_step_min": round(min(region_ms) / n, 6),
                          "ms_per_step_max": round(max(region_ms) / n, 6)},
               "pipelining": "each step is one CUDA graph per input set: the upload of the next "
                             "step's packed inputs and the read-back of the previous step's "
                             "output run beside this step's kernels; each region starts with "
                             "its first step's upload and ends with its last step's read-back, "
                             "both inside the timed region"}
        if self.planned:
            rec["plan_built_per_step"] = True
            rec["plan_build_us_host_median"] = round(statistics.median(plan_us), 2) \
                if plan_us else None
        return rec

    # -- results
    def output_bits(self):
        return self.synth.bits(self.outs)

    def appended_rows(self):
        """The pool's K and V rows at every sequence's appended slot, per layer:
        uint16 [layers][B][2][Hkv][D]."""
        torch, w = self.torch, self.w
        pos = torch.from_numpy(w.positions.astype(np.int64)).to(self.dev)
        bt = self.d["block_tables"].long()
        blk = (pos // w.page_size).clamp(min=0)
        pages = bt.gather(2, blk.view(1, -1, 1).expand(w.layers, -1, 1)).squeeze(2)
        slot = (pos % w.page_size).view(1, -1).expand(w.layers, -1)
        pool = self.d["pool"]
        rows = pool[pages.clamp(min=0), :, slot]          # [layers][B][2][Hkv][D]
        return self.synth.bits(rows)

    def close(self):
        for k in list(vars(self)):
            if k not in ("torch", "binding", "synth", "w", "args", "dev", "world"):
                delattr(self, k)
        self.torch.cuda.synchronize(self.dev)
        self.torch.cuda.empty_cache()


def l2_flush_buffer(dev):
    """A device buffer twice the L2 size, written between steps of the
    L2-resident workloads."""
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (132 << 20)
    return torch.empty(2 * l2, dtype=torch.uint8, device=dev), l2


def measure_workload(name, args, dev, peak):
    """One per-workload record: the step timed like the headline (repeated
    regions of K steps; L2 flushed between steps when the workload fits in
    L2), its roofline on the step's algorithmic bytes, the kernels' shares,
    the oracle's time, and every output against the oracle."""
    import torch
    from paged_kv_decode_04_gb300 import synth
    t_start = time.time()
    w = synth.make_workload(name, args.seed)
    db = DecodeBench(w, args, dev)
    db.warm_and_capture(args.warmup, args.graph)
    fits_l2 = w.kv_bytes() <= 96 * 2 ** 20
    flush, l2 = l2_flush_buffer(dev) if fits_l2 else (None, 0)
    times, _, _ = db.timed(args.steps, flush, min_seconds=min(0.5, args.repeat_seconds))
    db.check_err("timed runs")
    sp = spread(times, args.steps)
    ms = sp["ms_per_step_median"]
    step_bytes = algorithmic_bytes(w, "step")
    gbs = step_bytes / (ms / 1e3) / 1e9
    shares = db.kernel_shares()
    got = db.output_bits()
    rows = db.appended_rows()
    rec = {
        "workload": WORKLOAD_TEXT[name], "layers_per_step": w.layers,
        "split_plan": db.split_text, "kernels": db.launched,
        "algorithmic_bytes_per_step": step_bytes,
        "ms_per_step": ms, "timing": sp,
        "value": round(gbs, 2), "unit": "GB/s", "steps_per_s": round(1e3 / ms, 1),
        "l2": (f"flushed: {2 * l2 >> 20} MiB written between steps, outside the per-step "
               f"CUDA-event pairs (K/V {w.kv_bytes() / 2 ** 20:.1f} MiB per step fits in L2); "
               f"each step queued behind a spin, so its events time the device, not the "
               f"host's launch"
               if fits_l2 else f"inputs larger than L2: {w.kv_bytes() / 2 ** 30:.2f} GiB of "
               f"K/V streamed per step; no flush"),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                     "frac": round(gbs / peak, 4), "unit": "GB/s",
                     "basis": "the whole step's algorithmic bytes / its median CUDA-event time"},
        "kernel_shares": shares,
        "gpu_launches": db.kernels_per_layer * w.layers * args.steps * sp["repeats"],
    }
    if shares and "unavailable" not in shares:
        dom = next(iter(shares))
        rec["dominant_kernel"] = {"name": dom, "share": shares[dom]}
        rec["roofline"]["traffic"] = recorded_traffic(name, db.launched + " (fused step)")
    if name == "prefix":
        ub = unique_bytes(w)
        ug = ub / (ms / 1e3) / 1e9
        rec["unique_bytes_per_step"] = ub
        rec["roofline"] = {"bound": "hbm", "achieved": round(ug, 1), "peak": peak,
                           "frac": round(ug / peak, 4), "unit": "GB/s",
                           "basis": "bytes with every shared prefix page counted once per step "
                                    "(what DRAM must deliver) / the median CUDA-event time",
                           "traffic": recorded_traffic(name, db.launched + " (fused step)")}
        rec["value"] = round(ug, 2)
        rec["dedup_work_rate"] = {
            "value": round(gbs, 2), "unit": "GB/s",
            "what": "per-sequence algorithmic bytes (shared pages counted once per sequence "
                    "that attends them) / step time: deduplicated work, not a bandwidth"}
    db.close()
    del flush
    torch.cuda.empty_cache()
    # the oracle: every sequence of every layer, all host cores; tiny and small
    # also on one thread
    dt, nb, threads, used, seqs, refs, slots = oracle_sample_run(w, w.batch, want_slots=True)
    orc = {"seconds": round(dt, 4), "threads": threads, "value": round(nb / dt / 1e9, 4),
           "unit": "GB/s", "sample": f"all {used} sequences x {w.layers} layer(s)"}
    if name in ("tiny", "small"):
        dt1, nb1, _, _, _, _ = oracle_sample_run(w, w.batch, threads=1)
        orc["single_thread_seconds"] = round(dt1, 4)
        orc["single_thread_value"] = round(nb1 / dt1 / 1e9, 4)
    rec["oracle"] = orc
    rec["speedup_vs_oracle"] = round(dt / (ms / 1e3), 1)
    par = parity_report(got, refs)
    par["appended_slots_bit_exact"] = bool(np.array_equal(rows, np.stack(slots)))
    par["sequences"] = f"all {w.batch} x {w.layers} layer(s)"
    rec["parity_vs_oracle"] = par
    rec["wall_s"] = round(time.time() - t_start, 1)
    return rec


def measure_prefill(args, dev, peak):
    """The paged prefill write (256 prompts x 2047 tokens) timed in repeated
    regions; 4 prompts' pages compared bit for bit with the oracle's write."""
    import torch
    import oracle
    from paged_kv_decode_04_gb300 import binding, synth
    t_start = time.time()
    p = synth.make_prefill(args.seed)
    B, L = p.batch, p.prompt_len
    k = synth.to_device_bf16(p.k, dev)
    v = synth.to_device_bf16(p.v, dev)
    off = torch.from_numpy(p.token_offsets).to(dev)
    st = torch.from_numpy(p.start_positions).to(dev)
    bt = torch.from_numpy(p.block_table).to(dev)
    pool = torch.full((p.num_pages, 2, 16, 8, 64), -1, dtype=torch.int16,
                      device=dev).view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        binding.kv_write_prefill(k, v, off, st, pool, bt, dev_err=err)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    def region():
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    probe = region()
    reps = int(min(MAX_REPEATS, max(args.min_repeats, math.ceil(
        min(0.5, args.repeat_seconds) / max(probe / 1e3, 1e-6)))))
    times = [region() for _ in range(reps)]
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the prefill write")
    sp = spread(times, args.steps)
    ms = sp["ms_per_step_median"]
    T = B * L
    step_bytes = T * 8 * 64 * 2 * 2 * 2 + (B + 1) * 4 + B * 4 + B * p.block_table.shape[1] * 4
    gbs = step_bytes / (ms / 1e3) / 1e9
    # oracle: the write of 4 prompts into a compact pool of their pages
    sample = [0, 1, B // 2, B - 1]
    c = synth.compact_prefill(p, sample)
    t0 = time.perf_counter()
    rc = oracle.kv_write_prefill(c.k, c.v, c.token_offsets, c.start_positions, c.pool,
                                 c.block_table)
    dt = time.perf_counter() - t0
    got = synth.bits(pool[torch.from_numpy(c.pages).to(dev)])
    exact = rc == 0 and bool(np.array_equal(got, c.pool))
    rec = {
        "workload": PREFILL_TEXT, "algorithmic_bytes_per_step": step_bytes, "ms_per_step": ms,
        "timing": sp, "value": round(gbs, 2), "unit": "GB/s",
        "l2": "inputs larger than L2: 1.07 GB of new K/V read and written per call; no flush",
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                     "frac": round(gbs / peak, 4), "unit": "GB/s",
                     "basis": "bytes of the call (new K/V read + pool write + offsets, positions, "
                              "tables) / its median CUDA-event time"},
        "dominant_kernel": {"name": "kv_write_prefill_kernel", "share": 1.0},
        "oracle": {"seconds": round(dt, 4), "threads": 1,
                   "value": round(len(sample) * L * 8 * 64 * 2 * 2 * 2 / dt / 1e9, 4),
                   "unit": "GB/s", "sample": f"{len(sample)} of {B} prompts"},
        "parity_vs_oracle": {"pages_compared": int(len(c.pages)),
                             "bit_exact": exact, "sequences": f"{len(sample)} of {B} prompts"},
        "gpu_launches": args.steps * sp["repeats"],
    }
    del pool, k, v
    torch.cuda.empty_cache()
    rec["wall_s"] = round(time.time() - t_start, 1)
    return rec


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
    from paged_kv_decode_04_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    w = synth.make_workload(args.workload, args.seed, num_pages=args.pool_pages)
    db = DecodeBench(w, args, dev, world=world)
    plan_build_us = None
    if db.planned:
        # host cost of planning one step (a serving loop builds one plan per step)
        from paged_kv_decode_04_gb300 import binding
        t = time.perf_counter()
        for _ in range(200):
            binding.Plan(w.seq_lens, w.max_blocks, **db.plan_kw)
        plan_build_us = round((time.perf_counter() - t) / 200 * 1e6, 2)
    db.warm_and_capture(args.warmup, args.graph)
    layers = w.layers

    # ---- timed: repeated regions of K whole steps, device-resident inputs
    sampler = ClockSampler(gpu_selector(local)) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    times, t_wall0, t_wall1 = db.timed(args.steps)
    if sampler:
        sampler.stop()
    db.check_err("timed runs")
    sp = spread(times, args.steps)
    ms_per_step = sp["ms_per_step_median"]
    step_bytes = algorithmic_bytes(w, "step")
    dedup = None
    if args.workload == "prefix":
        # sequences share prefix pages: the bytes DRAM must deliver count each
        # physical page once per step; the per-sequence count is kept as a
        # work rate, not a bandwidth
        dedup = {"value": round(step_bytes / (ms_per_step / 1e3) / 1e9 * world, 2),
                 "unit": "GB/s", "algorithmic_bytes_per_step": step_bytes,
                 "what": "per-sequence algorithmic bytes (shared pages counted once per "
                         "sequence that attends them) / step time: deduplicated work, not a "
                         "bandwidth"}
        step_bytes = unique_bytes(w)
    total_bytes = sum_over_ranks(step_bytes, world, dev)
    value = total_bytes / (ms_per_step / 1e3) / 1e9

    # ---- per-kernel durations: CUDA events around each launch on the same stream
    kern, dom_ms, dom_bytes, dom_name = db.per_launch(args.steps)
    if dedup is not None and db.fused:
        dom_bytes = step_bytes / layers  # the whole fused step, shared pages once
    peak, peak_kind = measured_hbm_peak()
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    duration_source = "CUDA events around each launch, in a separate pass of the same loop"
    if db.fused and db.kernels_per_layer == 1:
        # the timed steps are this one kernel, `layers` launches per step back to back: its
        # average launch duration is the timed regions' own CUDA-event time per launch (the
        # separate pass above puts an event record between launches, which keeps each launch
        # from starting before the previous one has finished)
        dom_ms = ms_per_step / layers
        kern["decode_step_timed_region"] = round(dom_ms * 1e3, 2)
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        duration_source = ("timed regions: the median of the repeated CUDA-event regions of K "
                           "steps, which are this kernel alone")

    # ---- end to end: per-step plan built on the host, inputs from pinned host
    # memory, output back to the host
    e2e = db.e2e(args.steps, args.warmup) if args.e2e else None

    # ---- CPU baseline: the oracle on a bounded sample of the same workload, and
    # the same sample set against the GPU's outputs of the timed steps
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
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
        got = db.output_bits()[:, seqs]
        cpu["parity_vs_gpu"] = parity_report(got, refs)
    launched, kernels_per_layer, split_text, splits = (db.launched, db.kernels_per_layer,
                                                       db.split_text, db.splits)
    fused = db.fused
    db.close()

    # ---- the other workloads, each the same way (N = 1 only)
    per = None
    if rank == 0 and world == 1 and args.per_workload:
        per = {}
        for name in PER_WORKLOADS:
            if name != args.workload:
                print(f"[bench] {name} ...", file=sys.stderr, flush=True)
                per[name] = measure_workload(name, args, dev, peak)
                print(f"[bench] {name}: {per[name]['ms_per_step'] * 1e3:.2f} us per step, "
                      f"{per[name]['value']} GB/s", file=sys.stderr, flush=True)
        print("[bench] prefill ...", file=sys.stderr, flush=True)
        per["prefill"] = measure_prefill(args, dev, peak)

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
        "timing": sp,
        "steps_per_s": round(1e3 / ms_per_step * world, 1),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_copy": round(100 * value / world / peak, 2),
        "algorithmic_bytes_per_step": step_bytes,
        "bytes_basis": ("every physical page once per step (shared prefix pages once)"
                        if dedup is not None else "per-sequence algorithmic bytes"),
        "dedup_work_rate": dedup,
        "kernels_us": kern,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": dom_name, "peak_kind": f"{peak_kind} copy bandwidth",
                     "bytes_per_launch": dom_bytes, "duration_source": duration_source},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": kernels_per_layer * layers * args.steps * sp["repeats"],
        "gpu_launches_note": "library kernels launched in all the repeated timed regions",
        "clocks": clocks,
    }
    if per is not None:
        line["per_workload"] = per
    print(json.dumps(line), flush=True)
    return 0


def run_prefill(args, world, rank, local):
    """Throughput of the paged prefill write alone: 256 prompts x 2047 tokens per call."""
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    peak, _ = measured_hbm_peak()
    rec = measure_prefill(args, dev, peak)
    if rank == 0:
        line = {"metric": "paged prefill write achieved HBM GB/s", "value": rec["value"],
                "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "storage_dtype": "bf16",
                "data": "synthetic", "config": {"workload": PREFILL_TEXT, "seed": args.seed}}
        line.update({k: rec[k] for k in ("timing", "algorithmic_bytes_per_step", "roofline",
                                         "parity_vs_oracle", "gpu_launches")})
        print(json.dumps(line), flush=True)
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
    ap.add_argument("--min-repeats", type=int, default=MIN_REPEATS,
                    help="fewest timed regions of K steps (the median is reported)")
    ap.add_argument("--repeat-seconds", type=float, default=MIN_TIMED_SECONDS,
                    help="shortest span of the repeated timed regions")
    ap.add_argument("--e2e", action=argparse.BooleanOptionalAction, default=True,
                    help="also measure the step end to end from pinned host memory")
    ap.add_argument("--per-workload", action=argparse.BooleanOptionalAction, default=True,
                    help="after the headline, measure the other workloads and the prefill "
                         "write the same way, each against the oracle (N = 1 only)")
    ap.add_argument("--op",choices=["decode", "prefill", "serve"], default="decode",
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
