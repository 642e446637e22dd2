"""A synthetic serving loop: the host scheduler (include/pkv_sched.h) drives the
prefill write and the fused decode step on the GPU.

Each iteration is one scheduling point: admit waiting requests, prefill at
most one admitted prompt (its K/V written into freshly allocated pages of
every layer), then run one decode step for every prefilled sequence (one new
token appended at its next position and attended over its pages, per
layer).  Request K/V/q values are synthetic (seeded N(0, 1) rounded to bf16);
there are no weights, so "tokens" are the decode steps the scheduler issues.
This mirrors the engine loop of the Tiny-vLLM README ("これまでの進捗":
static and continuous batching; "現在のスコープ": one prompt prefilled
between decode iterations).
"""
from __future__ import annotations

import time

import numpy as np
import torch

from . import binding
from .scheduler import Scheduler

HQ, HKV, D, P = 32, 8, 64, 16


class Engine:
    def __init__(self, num_pages: int, layers: int, device, *, max_context: int = 2048,
                 static_batching: bool = False, max_batch: int = 256, seed: int = 0,
                 host_inputs: bool = False, use_plan: bool = True):
        self.dev = torch.device(device)
        self.layers = layers
        self.max_batch = max_batch
        self.max_blocks = max_context // P
        self.sched = Scheduler(num_pages, layers, max_context, P, static_batching)
        self.pool = torch.full((num_pages, 2, P, HKV, D), -1, dtype=torch.int16,
                               device=self.dev).view(torch.bfloat16)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)
        # the automatic split plan depends on the batch size: size the
        # workspace for the largest need over every batch the loop may build
        need = max(binding.workspace_bytes(n, self.max_blocks) for n in range(1, max_batch + 1))
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=self.dev)
        self.host_inputs = host_inputs
        # the scheduler knows every length, so each decode step runs under a
        # work plan built from them (pkv_plan_build), shared by all layers
        self.use_plan = use_plan
        self.rng = np.random.default_rng(seed)
        self.gen = torch.Generator(device=self.dev).manual_seed(seed)

    def _normal(self, shape):
        if self.host_inputs:
            x = torch.from_numpy(self.rng.standard_normal(shape).astype(np.float32))
            return x.to(torch.bfloat16).to(self.dev)
        return torch.randn(shape, generator=self.gen, device=self.dev, dtype=torch.bfloat16)

    def _upload_i32(self, *arrays):
        """Copy int32 host arrays to the device in one transfer through pinned
        memory, without waiting for the work already queued; returns views."""
        sizes = [a.size for a in arrays]
        staged = torch.empty(sum(sizes), dtype=torch.int32, pin_memory=True)
        flat = staged.numpy()
        at = 0
        for a, k in zip(arrays, sizes):
            flat[at:at + k] = a.reshape(-1)
            at += k
        dev = staged.to(self.dev, non_blocking=True)
        views, at = [], 0
        for a, k in zip(arrays, sizes):
            views.append(dev[at:at + k].view(a.shape))
            at += k
        return views

    def step(self, on_prefill=None, on_decode=None) -> int:
        """One scheduling point; returns the decode batch size."""
        self.sched.admit()
        got = self.sched.next_prefill()
        if got is not None:
            rid, plen, bt = got
            dbt, off, st = self._upload_i32(np.ascontiguousarray(bt, dtype=np.int32)[:, None],
                                            np.array([0, plen], np.int32),
                                            np.zeros(1, np.int32))
            kv = self._normal((2, self.layers, plen, HKV, D))   # one draw per prompt
            ks, vs = kv[0], kv[1]
            binding.kv_write_prefill_layers(ks, vs, off, st, self.pool, dbt, dev_err=self.err)
            if on_prefill is not None:
                for layer in range(self.layers):
                    on_prefill(layer, rid, ks[layer], vs[layer], bt[layer])
        n = min(self.max_batch, self.sched.running())
        if n == 0:
            return 0
        # One pinned staging buffer per step: the scheduler writes every
        # layer's block table and the lengths straight into it, the plan is
        # built behind them, and one copy moves all of it to the device.
        L, mb = self.layers, self.max_blocks
        nt = L * n * mb
        plan_at = (nt + n + 3) // 4 * 4                  # 16-byte aligned
        plan_words = binding.plan_bytes(n, mb) // 4 if self.use_plan else 0
        staged = torch.empty(plan_at + plan_words, dtype=torch.int32, pin_memory=True)
        flat = staged.numpy()
        bts = flat[:nt].reshape(L, n, mb)
        lens = flat[nt:nt + n]
        ids = np.empty(n, np.int64)
        if self.sched.decode_batch_into(ids, lens, bts) != n:
            raise RuntimeError("the scheduler's decode batch does not match its running count")
        plan = None
        upto = nt + n
        if self.use_plan:
            plan = binding.Plan(lens, mb, out=flat[plan_at:])
            upto = plan_at + plan.bytes_used // 4
            if plan.workspace_bytes > self.ws.numel():
                self.ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=self.dev)
        dev = staged[:upto].to(self.dev, non_blocking=True)
        dbts = dev[:nt].view(L, n, mb)
        dlens = dev[nt:nt + n]
        if plan is not None:
            plan.dev = dev[plan_at:upto]
        a, b = L * n * HQ * D, L * n * HKV * D
        x = self._normal((a + 2 * b,))                   # one draw per step
        qs = x[:a].view(L, n, HQ, D)
        kns = x[a:a + b].view(L, n, HKV, D)
        vns = x[a + b:].view(L, n, HKV, D)
        if plan is not None:
            # every layer in one native call, launched in layer order
            outs = binding.decode_steps_planned(qs, kns, vns, self.pool, dbts, dlens, plan,
                                                workspace=self.ws, dev_err=self.err)
        else:
            outs = [binding.decode_step(qs[layer], kns[layer], vns[layer], self.pool,
                                        dbts[layer], dlens, workspace=self.ws,
                                        dev_err=self.err) for layer in range(L)]
        if on_decode is not None:
            for layer in range(L):
                on_decode(layer, ids, lens, bts[layer], qs[layer], kns[layer], vns[layer],
                          outs[layer])
        return n

    def run(self, requests, max_iters: int = 1_000_000, on_prefill=None, on_decode=None):
        """Serve `requests` [(prompt_tokens, max_new_tokens)] to completion."""
        ids = [self.sched.submit(p, n) for p, n in requests]
        tokens = 0
        iters = 0
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        while iters < max_iters:
            st = self.sched.stats()
            if st["waiting"] == 0 and st["active"] == 0:
                break
            tokens += self.step(on_prefill, on_decode)
            iters += 1
        torch.cuda.synchronize(self.dev)
        dt = time.perf_counter() - t0
        self.sched.admit()   # release what the last step finished
        if int(self.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(self.err.item())}")
        return {"request_ids": ids, "decode_tokens": tokens, "iterations": iters,
                "seconds": dt, "stats": self.sched.stats()}
