"""Segment plans on the GPU: CTAs that stream several sequences' pages (whole
sequences and pieces of long ones) through one ring of whole-page boxes.

Every output is checked against the FP64 oracle, and every appended slot bit
for bit; plans made as for more SMs than the device has cut more sequences in
pieces (partials and merges), and empty sequences must give zero rows.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip

pytestmark = pytest.mark.gpu


def oracle_step(w):
    """The oracle's step (append of the live sequences, then attention) on a
    compact host copy of layer 0; empty sequences append nothing."""
    c = synth.compact(w, 0)
    live = np.nonzero(c.seq_lens > 0)[0]
    assert oracle.kv_append(c.k_new[live], c.v_new[live], c.pool, c.block_table[live],
                            c.positions[live]) == 0
    return oracle.decode_attention(c.q, c.pool, c.block_table, c.seq_lens), c


def appended_ok(w, d, c):
    pos = w.positions
    live = np.nonzero(w.seq_lens > 0)[0]
    pages = w.block_tables[0, live, pos[live] // 16]
    got = synth.bits(d["pool"][torch.from_numpy(pages).long().cuda(), :,
                               torch.from_numpy(pos[live] % 16).long().cuda()])
    want = c.pool[c.block_table[live, pos[live] // 16], :, pos[live] % 16]
    return np.array_equal(got, want)


@pytest.mark.parametrize("num_sms", [152, 400, 1000])
@pytest.mark.parametrize("seed", [0, 1])
def test_segment_plans_match_the_oracle(seed, num_sms):
    dev = cuda_or_skip()
    b = binding()
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(300, 700))
    lens = rng.integers(100, 2049, n).astype(np.int32)
    lens[rng.choice(n, 6, replace=False)] = 0
    lens[rng.choice(n, 6, replace=False)] = 1
    w = synth.make_workload("custom", 20 + seed, seq_lens=lens, num_pages=int(
        sum(-(-int(L) // 16) for L in lens) + 512))
    plan = b.Plan(w.seq_lens, w.max_blocks, num_sms=num_sms, device=dev)
    assert plan.num_segs > 0
    if num_sms > 152:
        assert plan.num_merges > 0 and plan.items()[:, 2].max() > 1
    ref, c = oracle_step(w)
    for fused in (True, False):
        d = synth.device_inputs(w, dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        if fused:
            out = b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                        d["block_tables"][0], d["seq_lens"], plan, dev_err=err)
        else:
            # (an empty sequence's position -1 is skipped and reported: no dev_err here)
            b.kv_append(d["k_new"][0], d["v_new"][0], d["pool"], d["block_tables"][0],
                        d["positions"])
            out = b.paged_decode_attention_planned(d["q"][0], d["pool"], d["block_tables"][0],
                                                   d["seq_lens"], plan, dev_err=err)
        got = synth.bits(out)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(got, ref, f"segment plan for {num_sms} SMs, fused={fused}")
        assert np.all(got[w.seq_lens == 0] == 0)
        assert appended_ok(w, d, c)


def test_segment_plan_equals_the_whole_page_kernel_bit_for_bit():
    # one whole sequence per segment CTA: the same per-page arithmetic in the
    # same order as the whole-page kernel with one range per sequence
    dev = cuda_or_skip()
    b = binding()
    w = synth.make_workload("peak", 3, batch=200, num_pages=30000)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    assert plan.num_segs == w.batch and plan.num_merges == 0
    assert b.attention_kernels(w.batch, w.max_blocks, 1) == "paged_decode_pagebox_kernel"
    outs = []
    for planned in (True, False):
        d = synth.device_inputs(w, dev)
        if planned:
            out = b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                        d["block_tables"][0], d["seq_lens"], plan)
        else:
            out = b.decode_step(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                d["block_tables"][0], d["seq_lens"], num_splits=1)
        outs.append((synth.bits(out), synth.bits(d["pool"])))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_segment_plan_with_changed_lengths_is_reported():
    # the kernels take the lengths from the plan; a device length that
    # differs from the plan's is reported as PKV_DEVERR_PLAN
    dev = cuda_or_skip()
    b = binding()
    lens = np.random.default_rng(4).integers(300, 2049, 400).astype(np.int32)
    w = synth.make_workload("custom", 24, seq_lens=lens, num_pages=int(
        sum(-(-int(L) // 16) for L in lens) + 64))
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    assert plan.num_segs > 0
    d = synth.device_inputs(w, dev)
    d["seq_lens"][7] -= 1
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    b.paged_decode_attention_planned(d["q"][0], d["pool"], d["block_tables"][0], d["seq_lens"],
                                     plan, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == b.DEVERR_PLAN
