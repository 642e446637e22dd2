"""GPU parity past the 2048-token context: block tables of 2048 entries (32k
tokens) and of 8192 entries (128k tokens), so that a sequence has more pages
than one range may hold (the fixed plan caps a range at 1024 pages), work-plan
ranges grow with the table and merge up to 48 partials, and the fused append
rotates positions far past the 2048-entry cos/sin table.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip

pytestmark = pytest.mark.gpu

MAX_BLOCKS = 2048
LENS = [32768, 10000, 5, 0, 2049, 16 * 1024 + 1]


def workload():
    lens = np.asarray(LENS, np.int32)
    pages = int(sum((int(L) + 15) // 16 for L in lens))
    return synth.make_workload("edge", 41, seq_lens=lens, num_pages=pages + 64,
                               max_blocks=MAX_BLOCKS)


def oracle_step(w):
    """Append at seq_lens - 1, then attention, on a host copy of the pool."""
    pool = synth.host_pool(w)
    live = np.nonzero(w.seq_lens > 0)[0]
    assert oracle.kv_append(w.k_new[0][live], w.v_new[0][live], pool, w.block_tables[0][live],
                            w.positions[live]) == 0
    return oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens), pool


@pytest.mark.parametrize("mode", ["auto", "splits1", "splits5", "plan"])
def test_fused_step_long_context(mode):
    dev = cuda_or_skip()
    w = workload()
    ref, host_pool = oracle_step(w)
    d = synth.device_inputs(w, dev)
    b = binding()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    args = (d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], d["block_tables"][0],
            d["seq_lens"])
    if mode == "plan":
        plan = b.Plan(w.seq_lens, MAX_BLOCKS, device=dev)
        assert plan.range_pages <= 1024
        out = b.decode_step_planned(*args, plan, rope_theta=w.rope_theta, scale=w.scale,
                                    dev_err=err)
    else:
        splits = {"auto": 0, "splits1": 1, "splits5": 5}[mode]
        if splits == 1:   # 2048 pages per range would exceed the cap: two ranges of 1024
            assert b.plan_splits(len(LENS), MAX_BLOCKS, 1) == 2
        out = b.decode_step(*args, rope_theta=w.rope_theta, scale=w.scale, num_splits=splits,
                            dev_err=err)
    got = synth.bits(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got, ref, f"long context, {mode}")
    assert np.all(got[3] == 0)                     # the empty sequence
    # the appended slots, positions up to 32767, are the oracle's bits
    pool = synth.bits(d["pool"])
    for i in np.nonzero(w.seq_lens > 0)[0]:
        pos = int(w.positions[i])
        page = int(w.block_tables[0, i, pos // 16])
        assert np.array_equal(pool[page, :, pos % 16], host_pool[page, :, pos % 16]), (i, pos)


# 128k tokens: a table of 8192 entries, ranges capped at 1024 pages (fixed
# plan) or cut by the host plan into 172-page ranges merged 48 and 26 ways,
# and the append at position 131071, far past the cos/sin table
HUGE_BLOCKS = 8192
HUGE_LENS = [131072, 70000, 3]


@pytest.fixture(scope="module")
def huge():
    lens = np.asarray(HUGE_LENS, np.int32)
    pages = int(sum((int(L) + 15) // 16 for L in lens))
    w = synth.make_workload("edge", 43, seq_lens=lens, num_pages=pages + 64,
                            max_blocks=HUGE_BLOCKS)
    ref, host_pool = oracle_step(w)
    return w, ref, host_pool


@pytest.mark.parametrize("mode", ["auto", "splits1", "plan"])
def test_fused_step_128k_context(huge, mode):
    dev = cuda_or_skip()
    w, ref, host_pool = huge
    d = synth.device_inputs(w, dev)
    b = binding()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    args = (d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], d["block_tables"][0],
            d["seq_lens"])
    if mode == "plan":
        plan = b.Plan(w.seq_lens, HUGE_BLOCKS, device=dev)
        assert plan.num_merges == 2
        out = b.decode_step_planned(*args, plan, rope_theta=w.rope_theta, scale=w.scale,
                                    dev_err=err)
    else:
        splits = 0 if mode == "auto" else 1
        if splits == 1:   # 8192 pages: eight ranges of the 1024-page cap
            assert b.plan_splits(len(HUGE_LENS), HUGE_BLOCKS, 1) == 8
        out = b.decode_step(*args, rope_theta=w.rope_theta, scale=w.scale, num_splits=splits,
                            dev_err=err)
    got = synth.bits(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got, ref, f"128k context, {mode}")
    pool = synth.bits(d["pool"])
    for i in range(len(HUGE_LENS)):
        pos = int(w.positions[i])
        page = int(w.block_tables[0, i, pos // 16])
        assert np.array_equal(pool[page, :, pos % 16], host_pool[page, :, pos % 16]), (i, pos)
