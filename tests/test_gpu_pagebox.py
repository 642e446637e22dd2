"""GPU parity of the whole-page attention kernel (decode_pagebox.cu), which
serves batches of at least one CTA per SM: one CTA per (sequence, range) for
all kv heads, each page one 32 KiB TMA box.  Reached through the fixed plan
(S ranges per sequence, split merge for S > 1) and through work plans made of
ranges only (the planned instance, with and without split sequences).

Outputs are checked against the FP64 oracle with the attention tolerance of
_gpu_util; appended slots bit for bit; the fused step equals append +
attention bit for bit; the fixed S = 1 call and a one-range-per-sequence plan
are the same decomposition and give the same bits.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip

pytestmark = pytest.mark.gpu

B = 160            # >= the SM count (152 on GB300): the whole-page kernel's territory


def workload(lo, hi, seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, B).astype(np.int32)
    lens[:4] = [hi, lo, 16 * ((lo + hi) // 32), 16 * ((lo + hi) // 32) + 1]
    pages = int(sum((int(L) + 15) // 16 for L in lens))
    return synth.make_workload("edge", seed, seq_lens=lens, num_pages=pages + 64)


def oracle_step(w):
    pool = synth.host_pool(w)
    live = np.nonzero(w.seq_lens > 0)[0]
    assert oracle.kv_append(w.k_new[0][live], w.v_new[0][live], pool, w.block_tables[0][live],
                            w.positions[live]) == 0
    return oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens, threads=0), pool


def check_slots(w, dev_pool, host_pool):
    pool = synth.bits(dev_pool)
    for i in np.nonzero(w.seq_lens > 0)[0]:
        pos = int(w.positions[i])
        page = int(w.block_tables[0, i, pos // 16])
        assert np.array_equal(pool[page, :, pos % 16], host_pool[page, :, pos % 16]), i


@pytest.mark.parametrize("splits", [1, 2, 3])
def test_fixed_plan_fused_step(splits):
    dev = cuda_or_skip()
    w = workload(1, 700, 50 + splits)
    ref, host_pool = oracle_step(w)
    d = synth.device_inputs(w, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = binding().decode_step(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                d["block_tables"][0], d["seq_lens"], num_splits=splits,
                                dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(synth.bits(out), ref, f"whole-page kernel, S={splits}")
    check_slots(w, d["pool"], host_pool)


@pytest.mark.parametrize("num_sms", [152, 400])
def test_planned_ranges(num_sms):
    # long sequences only: a segment plan (the whole-page segment kernel);
    # planned as for 400 SMs the 128-page sequences are cut in pieces (partials
    # + merge)
    dev = cuda_or_skip()
    w = workload(1100, 2048, 60)
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, num_sms=num_sms, device=dev)
    assert not (plan.items()[:, 0] == 1).any() and plan.num_items >= 152
    assert num_sms == 152 or plan.num_merges > 0
    ref, host_pool = oracle_step(w)
    d = synth.device_inputs(w, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                d["block_tables"][0], d["seq_lens"], plan, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert b.attention_kernels(w.batch, w.max_blocks, 0, plan).startswith(
        "paged_decode_segments_kernel")
    assert_close(synth.bits(out), ref, f"segment kernel, plan for {num_sms} SMs")
    check_slots(w, d["pool"], host_pool)


def test_fused_equals_unfused_and_plan_equals_fixed():
    dev = cuda_or_skip()
    w = workload(900, 2048, 70)
    b = binding()
    # (planned: a segment plan, which may cut sequences in pieces; it equals
    # the fixed plan within tolerance, and bit for bit when every segment is
    # a whole sequence, which tests/test_gpu_segments.py checks)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    results = {}
    for mode in ("fused", "unfused", "planned"):
        d = synth.device_inputs(w, dev)
        bt, lens = d["block_tables"][0], d["seq_lens"]
        if mode == "fused":
            out = b.decode_step(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], bt, lens,
                                num_splits=1)
        elif mode == "unfused":
            b.kv_append(d["k_new"][0], d["v_new"][0], d["pool"], bt, d["positions"])
            out = b.paged_decode_attention(d["q"][0], d["pool"], bt, lens, num_splits=1)
        else:
            out = b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], bt,
                                        lens, plan)
        results[mode] = (synth.bits(out), synth.bits(d["pool"]))
    assert np.array_equal(results["unfused"][0], results["fused"][0])
    for mode in ("unfused", "planned"):
        assert np.array_equal(results[mode][1], results["fused"][1]), mode   # the pool
    if plan.num_merges == 0:
        assert np.array_equal(results["planned"][0], results["fused"][0])
    else:
        ref, _ = oracle_step(w)
        assert_close(results["planned"][0], ref, "segment plan")


def test_bad_pages_and_lengths_reported():
    dev = cuda_or_skip()
    w = workload(300, 600, 80)
    d = synth.device_inputs(w, dev)
    b = binding()
    b.kv_append(d["k_new"][0], d["v_new"][0], d["pool"], d["block_tables"][0], d["positions"])
    bt = d["block_tables"][0].clone()
    bt[5, 3] = w.num_pages + 9
    bt[6, 0] = -2
    lens = d["seq_lens"].clone()
    lens[7] = -1
    lens[8] = 128 * 16 + 3
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = b.paged_decode_attention(d["q"][0], d["pool"], bt, lens, num_splits=1, dev_err=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & b.DEVERR_PAGE and e & b.DEVERR_SEQLEN
    got = synth.bits(out)
    assert np.all(got[7] == 0)
    keep = [i for i in range(B) if i not in (5, 6, 7, 8)]
    ref, _ = oracle_step(w)
    assert_close(got[keep], ref[keep], "untouched sequences")
    # a bad page is skipped, the rest of its sequence still attended
    assert np.all(np.isfinite(oracle.bf16_to_f64(got[[5, 6]])))


def test_kernel_choice_is_reported():
    cuda_or_skip()
    b = binding()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    big = max(B, sms)                      # one CTA per SM: the whole-page kernel
    assert b.attention_kernels(big, 128, 1) == "paged_decode_pagebox_kernel"
    assert b.attention_kernels(big, 128, 2) == "paged_decode_pagebox_kernel+merge_splits_kernel"
    assert b.attention_kernels(sms - 1, 128, 1) == "paged_decode_kernel"
    assert b.attention_kernels(8, 128, 1) == "paged_decode_kernel"
    assert b.attention_kernels(1, 128, 0) == "paged_decode_kernel+merge_splits_kernel"
    lens = np.full(big, 2048, np.int32)    # planned: one whole-sequence segment per CTA
    assert b.attention_kernels(big, 128, 0, b.Plan(lens, 128)) == "paged_decode_segments_kernel"
    mixed = np.concatenate([np.full(13, 2000), np.full(115, 60)]).astype(np.int32)
    assert b.attention_kernels(128, 128, 0, b.Plan(mixed, 128)) == \
        "paged_decode_kernel+merge_plan_kernel"
