"""In-kernel waits that run out (GPU).

Every kernel that waits on its own copies or on another warp role gives up
after the calling thread's wait limit (pkv_set_wait_limit_ns), ORs
PKV_DEVERR_TIMEOUT into dev_err, lets what it started finish, frees what it
holds and returns.  Here the limit is 0 -- a wait whose copy has not landed at
the first look counts as timed out -- on batches that stream more K/V than L2
holds, so waits that find their copy still in flight are certain.  Nothing
faults or hangs: only the limit of the waits changes, every copy is a normal
one.  After each timed-out call the same call with the default limit must
match the FP64 oracle, i.e. the context and the pool are still good.
"""
import threading

import numpy as np
import pytest
import torch

from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip, oracle_step

pytestmark = pytest.mark.gpu


def new_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def timed_out(call, tries=3):
    """Run call(err) with the wait limit at 0 until a launch reports a
    timeout; returns the error bits and the call's result."""
    b = binding()
    for _ in range(tries):
        err = new_err()
        prev = b.set_wait_limit_ns(0)
        try:
            res = call(err)
        finally:
            b.set_wait_limit_ns(prev)
        torch.cuda.synchronize()
        bits = int(err.item())
        if bits & b.DEVERR_TIMEOUT:
            return bits, res
    return bits, res


def check_recovered(w, d, out_fn, what):
    """The same step with the default limit: no error bits, oracle outputs."""
    err = new_err()
    out = out_fn(err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{what}: error bits {int(err.item())} after the timeout"
    ref, _ = oracle_step(w, 0)
    assert_close(synth.bits(out), ref, what)


def test_default_limit_is_two_seconds_and_per_thread():
    cuda_or_skip()
    b = binding()
    assert b.set_wait_limit_ns(b.DEFAULT_WAIT_NS) == b.DEFAULT_WAIT_NS
    seen = []
    prev = b.set_wait_limit_ns(12345)
    try:
        t = threading.Thread(target=lambda: seen.append(b.set_wait_limit_ns(b.DEFAULT_WAIT_NS)))
        t.start()
        t.join()
    finally:
        assert b.set_wait_limit_ns(prev) == 12345
    assert seen == [b.DEFAULT_WAIT_NS]       # another thread keeps its own limit


def test_per_head_kernel_times_out_then_recovers():
    dev = cuda_or_skip()
    b = binding()
    # 64 sequences x 2048 tokens (256 MiB of K/V), two ranges each: the
    # per-(sequence, kv head, range) kernel and the split merge
    w = synth.make_workload("peak", 1, batch=64, num_pages=10000)
    d = synth.device_inputs(w, dev)
    assert b.attention_kernels(w.batch, w.max_blocks, 2) == \
        "paged_decode_kernel+merge_splits_kernel"
    bt, lens = d["block_tables"][0], d["seq_lens"]
    b.kv_append(d["k_new"][0], d["v_new"][0], d["pool"], bt, d["positions"])

    def call(err):
        return b.paged_decode_attention(d["q"][0], d["pool"], bt, lens, num_splits=2,
                                        dev_err=err)
    bits, out = timed_out(call)
    assert bits & b.DEVERR_TIMEOUT, f"no wait timed out (bits {bits})"
    assert torch.isfinite(out.float()).all()
    check_recovered(w, d, lambda err: b.paged_decode_attention(
        d["q"][0], d["pool"], bt, lens, num_splits=2, dev_err=err), "per-head kernel")


def test_planned_packed_kernel_times_out_then_recovers():
    dev = cuda_or_skip()
    b = binding()
    # 112 short and 16 long sequences: packed items (one sequence per warp)
    # and split ranges, the fused step under a host plan
    rng = np.random.default_rng(7)
    lens = np.concatenate([rng.integers(16, 129, 112), rng.integers(1536, 2049, 16)])
    lens = rng.permutation(lens).astype(np.int32)
    w = synth.make_workload("custom", 2, seq_lens=lens, num_pages=8192)
    d = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    assert (plan.items()[:, 0] == 1).any() and plan.num_merges > 0
    assert b.attention_kernels(w.batch, w.max_blocks, 0, plan) == \
        "paged_decode_kernel+merge_plan_kernel"

    def step(err):
        return b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                     d["block_tables"][0], d["seq_lens"], plan,
                                     rope_theta=w.rope_theta, scale=w.scale, dev_err=err)
    bits, out = timed_out(step)
    assert bits & b.DEVERR_TIMEOUT, f"no wait timed out (bits {bits})"
    assert torch.isfinite(out.float()).all()
    check_recovered(w, d, step, "planned per-head kernel")


def test_pagebox_kernel_times_out_then_recovers():
    dev = cuda_or_skip()
    b = binding()
    # 160 sequences of 512 tokens (160 MiB of K/V), one range each (fixed
    # plan): at least one CTA per SM, so the whole-page kernel runs, fused
    w = synth.make_workload("custom", 3, seq_lens=np.full(160, 512, np.int32), num_pages=8192)
    d = synth.device_inputs(w, dev)
    assert b.attention_kernels(w.batch, w.max_blocks, 1) == "paged_decode_pagebox_kernel"

    def step(err):
        return b.decode_step(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                             d["block_tables"][0], d["seq_lens"], num_splits=1,
                             rope_theta=w.rope_theta, scale=w.scale, dev_err=err)
    bits, out = timed_out(step)
    assert bits & b.DEVERR_TIMEOUT, f"no wait timed out (bits {bits})"
    assert torch.isfinite(out.float()).all()
    check_recovered(w, d, step, "whole-page kernel")


def test_segment_kernel_times_out_then_recovers():
    dev = cuda_or_skip()
    b = binding()
    # 600 sequences of 200-700 tokens (about 130 MiB of K/V): a segment plan,
    # several whole sequences and pieces per CTA, fused
    rng = np.random.default_rng(8)
    w = synth.make_workload("custom", 8, seq_lens=rng.integers(200, 701, 600).astype(np.int32),
                            num_pages=20000)
    d = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    assert plan.num_segs > 0 and plan.items()[:, 2].max() > 1
    assert b.attention_kernels(w.batch, w.max_blocks, 0, plan).startswith(
        "paged_decode_segments_kernel")

    def step(err):
        return b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                     d["block_tables"][0], d["seq_lens"], plan,
                                     rope_theta=w.rope_theta, scale=w.scale, dev_err=err)
    bits, out = timed_out(step)
    assert bits & b.DEVERR_TIMEOUT, f"no wait timed out (bits {bits})"
    assert torch.isfinite(out.float()).all()
    check_recovered(w, d, step, "segment kernel")


@pytest.mark.parametrize("share, kernels", [
    (64, "paged_decode_shared_kernel+paged_decode_segments_kernel+merge_plan_kernel"),
    (120, "paged_decode_shared_kernel+paged_decode_kernel+merge_plan_kernel")])
def test_shared_prefix_kernel_times_out_then_recovers(share, kernels):
    dev = cuda_or_skip()
    b = binding()
    # two groups of 16 sequences sharing 64 (or 120) pages, 2048 tokens each:
    # the tcgen05 shared-prefix kernel (copies, MMAs and TMEM in flight when
    # its waits give up), then segment CTAs beside it (own tails of 64 pages)
    # or the per-(item, kv head) kernel after it (tails of 8), and the merge
    w = synth.make_workload("prefix", 4, batch=32, num_pages=4096, share_group=16,
                            share_blocks=share)
    d = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, block_tables=w.block_tables[0])
    assert plan.num_shared > 0
    assert b.attention_kernels(w.batch, w.max_blocks, 0, plan) == kernels

    def step(err):
        return b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                     d["block_tables"][0], d["seq_lens"], plan,
                                     rope_theta=w.rope_theta, scale=w.scale, dev_err=err)
    bits, out = timed_out(step)
    assert bits & b.DEVERR_TIMEOUT, f"no wait timed out (bits {bits})"
    assert torch.isfinite(out.float()).all()
    check_recovered(w, d, step, "shared-prefix kernel")


@pytest.mark.parametrize("sms, layout", [(8, 0), (32, 1)])
def test_folding_segment_plan_times_out_then_recovers(sms, layout):
    dev = cuda_or_skip()
    b = binding()
    # 64 sequences in groups of 16 sharing 64 pages, 2048 tokens each: the
    # shared-prefix kernel and segment CTAs that fold each member's shared
    # partials into its output (no merge) -- both time out.  Planned as for
    # 8 SMs the shared-prefix CTAs run first (layout 0); as for 32 SMs the
    # segment CTAs run beside them and stream before their grid wait (layout 1)
    w = synth.make_workload("prefix", 7, batch=64, num_pages=8192, share_group=16,
                            share_blocks=64)
    d = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, num_sms=sms,
                  block_tables=w.block_tables[0])
    assert plan.num_shared > 0 and plan.num_segs > 0 and plan.num_merges == 0
    assert (plan.segments()[:, 5] > 0).all()
    assert plan.layout == layout

    def step(err):
        return b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                     d["block_tables"][0], d["seq_lens"], plan,
                                     rope_theta=w.rope_theta, scale=w.scale, dev_err=err)
    bits, out = timed_out(step)
    assert bits & b.DEVERR_TIMEOUT, f"no wait timed out (bits {bits})"
    assert torch.isfinite(out.float()).all()
    check_recovered(w, d, step, "folding segment plan")


def test_prefill_write_times_out_then_recovers():
    dev = cuda_or_skip()
    b = binding()
    import oracle
    # 64 prompts x 2047 tokens: 256 MiB of new K/V staged through the ring
    p = synth.make_prefill(5, batch=64, num_pages=8192)
    k = synth.to_device_bf16(p.k, dev)
    v = synth.to_device_bf16(p.v, dev)
    off = torch.from_numpy(p.token_offsets).to(dev)
    st = torch.from_numpy(p.start_positions).to(dev)
    bt = torch.from_numpy(p.block_table).to(dev)
    pool = torch.full((p.num_pages, 2, 16, 8, 64), -1, dtype=torch.int16,
                      device=dev).view(torch.bfloat16)

    def write(err):
        b.kv_write_prefill(k, v, off, st, pool, bt, dev_err=err)
    bits, _ = timed_out(write)
    assert bits & b.DEVERR_TIMEOUT, f"no wait timed out (bits {bits})"
    err = new_err()
    write(err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    c = synth.compact_prefill(p, [0, 31, 63])
    assert oracle.kv_write_prefill(c.k, c.v, c.token_offsets, c.start_positions, c.pool,
                                   c.block_table) == 0
    assert np.array_equal(synth.bits(pool[torch.from_numpy(c.pages).to(dev)]), c.pool)
