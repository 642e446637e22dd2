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


def test_two_thetas_on_two_streams_interleaved_are_bit_exact():
    # Appends with two rope_theta values, never seen before in this process,
    # run interleaved on two streams with nothing ordering one stream against
    # the other: each theta's first call builds its cos/sin table on its own
    # stream while the other stream's kernels run.  Every appended K row must
    # equal the oracle's rotation with its own theta, and every V row the new
    # V, bit for bit (a table rewritten under a reader would give another
    # theta's angles).
    import oracle
    from _gpu_util import bf16_normal
    dev = cuda_or_skip()
    b = binding()
    thetas = (31415.5, 271828.25)
    iters, batch, pages = 12, 64, 64 * 12
    rng = np.random.default_rng(11)
    pos = rng.integers(0, 2048, (2, iters, batch)).astype(np.int32)
    k_new = bf16_normal(rng, (2, iters, batch, 8, 64))
    v_new = bf16_normal(rng, (2, iters, batch, 8, 64))
    # iteration i of stream s writes sequence r's token into page i * batch + r
    bt = np.full((2, iters, batch, 128), -1, np.int32)
    for i in range(iters):
        bt[:, i, np.arange(batch), pos[0, i] // 16] = i * batch + np.arange(batch)
        bt[1, i] = -1
        bt[1, i, np.arange(batch), pos[1, i] // 16] = i * batch + np.arange(batch)
    u16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
        torch.bfloat16)
    pools = [torch.full((pages, 2, 16, 8, 64), -1, dtype=torch.int16, device=dev).view(
        torch.bfloat16) for _ in range(2)]
    ks, vs = u16(k_new), u16(v_new)
    bts = torch.from_numpy(bt).to(dev)
    ps = torch.from_numpy(pos).to(dev)
    errs = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in range(2)]
    torch.cuda.synchronize(dev)
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    for i in range(iters):
        for s in range(2):
            with torch.cuda.stream(streams[s]):
                b.kv_append(ks[s, i], vs[s, i], pools[s], bts[s, i], ps[s, i],
                            rope_theta=thetas[s], dev_err=errs[s])
    torch.cuda.synchronize(dev)
    assert int(errs[0].item()) == 0 and int(errs[1].item()) == 0
    for s in range(2):
        pool = synth.bits(pools[s])
        for i in range(iters):
            for r in range(batch):
                p = i * batch + r
                slot = int(pos[s, i, r]) % 16
                want_k = np.stack([oracle.rope_rotate(k_new[s, i, r, h], int(pos[s, i, r]),
                                                      thetas[s]) for h in range(8)])
                assert np.array_equal(pool[p, 0, slot], want_k), (s, i, r)
                assert np.array_equal(pool[p, 1, slot], v_new[s, i, r]), (s, i, r)
