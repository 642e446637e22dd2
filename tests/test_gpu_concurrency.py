"""Concurrent calls (the header's "calls are thread-safe"): host threads, each
on its own CUDA stream with its own pool copy, workspace and plan upload,
issue planned fused steps and fixed-plan attention at the same time.  The
library's host state (per-thread tensor-map caches, per-device configuration,
the RoPE table) must give every thread the bits of a sequential run.
"""
import threading

import numpy as np
import pytest
import torch

from paged_kv_decode_04_gb300 import synth
from _gpu_util import binding, cuda_or_skip

pytestmark = pytest.mark.gpu

THREADS = 4
ITERS = 25


def test_threads_on_their_own_streams_match_a_sequential_run():
    dev = cuda_or_skip()
    b = binding()
    lens = np.random.default_rng(3).integers(0, 2049, 40).astype(np.int32)
    w = synth.make_workload("edge", 3, seq_lens=lens, num_pages=3000)

    def one_step(d, plan, ws):
        bt, sl = d["block_tables"][0], d["seq_lens"]
        out = b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], bt, sl,
                                    plan, workspace=ws)
        att = b.paged_decode_attention(d["q"][0], d["pool"], bt, sl, num_splits=0)
        return out, att

    d0 = synth.device_inputs(w, dev)
    plan0 = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    ws0 = torch.empty(max(16, plan0.workspace_bytes), dtype=torch.uint8, device=dev)
    want = [synth.bits(x) for x in one_step(d0, plan0, ws0)]
    # the fused step appends the same rows each time, so repeating it is idempotent
    want2 = [synth.bits(x) for x in one_step(d0, plan0, ws0)]
    assert all(np.array_equal(a, c) for a, c in zip(want, want2))

    inputs = [synth.device_inputs(w, dev) for _ in range(THREADS)]
    torch.cuda.synchronize(dev)        # the uploads above ran on this thread's stream
    results, errors = [None] * THREADS, []

    def worker(i):
        try:
            s = torch.cuda.Stream(dev)
            with torch.cuda.stream(s):
                plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
                ws = torch.empty(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
                for _ in range(ITERS):
                    out = one_step(inputs[i], plan, ws)
            s.synchronize()
            results[i] = [synth.bits(x) for x in out]
        except Exception as e:  # surfaced below, in the test's thread
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(THREADS)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    for i in range(THREADS):
        assert all(np.array_equal(a, c) for a, c in zip(results[i], want)), i
