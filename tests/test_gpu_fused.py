"""GPU parity of the fused decode step (pkv_decode_step): one kernel that
appends the new token at seq_lens - 1 and attends over the pages.

It must write the same pool bits as pkv_kv_append and give bit-identical
outputs to pkv_kv_append + pkv_paged_decode_attention, and match the FP64
oracle within |err| <= 1e-3 + 8e-3 * |ref|.
"""
import functools

import numpy as np
import pytest
import torch

from paged_kv_decode_04_gb300 import synth
from _gpu_util import (appended_slots_expected, assert_close, binding, cuda_or_skip,
                       gpu_step, oracle_step)

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=2)
def workload(name, seed=0):
    return synth.make_workload(name, seed)


def fused(w, d, layer, **kw):
    return binding().decode_step(d["q"][layer], d["k_new"][layer], d["v_new"][layer], d["pool"],
                                 d["block_tables"][layer], d["seq_lens"],
                                 rope_theta=w.rope_theta, scale=w.scale, **kw)


@pytest.mark.parametrize("splits", [0, 1, 3, 32])
@pytest.mark.parametrize("name", ["tiny", "small", "long"])
def test_fused_equals_separate_bit_for_bit(name, splits):
    dev = cuda_or_skip()
    w = workload(name)
    d1 = synth.device_inputs(w, dev)
    d2 = synth.device_inputs(w, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for layer in range(w.layers):
        a = fused(w, d1, layer, num_splits=splits, dev_err=err)
        b = gpu_step(w, d2, layer, num_splits=splits)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (name, layer)
    assert torch.equal(d1["pool"].view(torch.int16), d2["pool"].view(torch.int16))
    torch.cuda.synchronize()
    assert int(err.item()) == 0


@pytest.mark.parametrize("name", ["tiny", "small", "long"])
def test_fused_matches_oracle(name):
    dev = cuda_or_skip()
    w = workload(name)
    d = synth.device_inputs(w, dev)
    for layer in range(w.layers):
        out = fused(w, d, layer)
        ref, _ = oracle_step(w, layer)
        assert_close(synth.bits(out), ref, f"fused {name} layer {layer}")
        kexp, vexp = appended_slots_expected(w, layer, range(w.batch))
        for b in range(w.batch):
            pos = int(w.positions[b])
            page = int(w.block_tables[layer, b, pos // 16])
            assert np.array_equal(synth.bits(d["pool"][page, 0, pos % 16]), kexp[b])
            assert np.array_equal(synth.bits(d["pool"][page, 1, pos % 16]), vexp[b])


def test_fused_peak_full_size_every_output():
    dev = cuda_or_skip()
    w = workload("peak")
    d = synth.device_inputs(w, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = synth.bits(fused(w, d, 0, dev_err=err))
    ref, _ = oracle_step(w, 0)             # every sequence, all host cores
    assert_close(out, ref, "fused peak, every output")
    kexp, vexp = appended_slots_expected(w, 0, range(w.batch))
    pos = torch.from_numpy(w.positions.astype(np.int64)).to(dev)
    pages = d["block_tables"][0].long().gather(1, (pos // 16)[:, None])[:, 0]
    sb = synth.bits(d["pool"][pages, :, pos % 16])
    assert np.array_equal(sb[:, 0], kexp) and np.array_equal(sb[:, 1], vexp)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the benchmark's configuration: the same step under a host work plan (one
    # whole sequence per segment CTA), on a fresh copy of the inputs
    b = binding()
    d2 = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, block_tables=w.block_tables[0])
    assert b.attention_kernels(w.batch, w.max_blocks, 0, plan) == "paged_decode_segments_kernel"
    out2 = synth.bits(b.decode_step_planned(d2["q"][0], d2["k_new"][0], d2["v_new"][0], d2["pool"],
                                            d2["block_tables"][0], d2["seq_lens"], plan,
                                            rope_theta=w.rope_theta, scale=w.scale, dev_err=err))
    assert_close(out2, ref, "fused peak, host plan, every output")
    sb2 = synth.bits(d2["pool"][pages, :, pos % 16])
    assert np.array_equal(sb2[:, 0], kexp) and np.array_equal(sb2[:, 1], vexp)
    if b.attention_kernels(w.batch, w.max_blocks, 0) == "paged_decode_pagebox_kernel":
        assert np.array_equal(out2, out)          # the same decomposition, the same bits
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_fused_mix_full_size_every_output():
    # the benchmark's configuration: the fused step under the host plan built
    # from the lengths and layer 0's tables, every layer, every sequence, and
    # every appended slot
    dev = cuda_or_skip()
    b = binding()
    w = workload("mix")
    d = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, block_tables=w.block_tables[0])
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = [synth.bits(b.decode_step_planned(
        d["q"][layer], d["k_new"][layer], d["v_new"][layer], d["pool"], d["block_tables"][layer],
        d["seq_lens"], plan, rope_theta=w.rope_theta, scale=w.scale, dev_err=err))
        for layer in range(w.layers)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    pos = w.positions
    for layer in range(w.layers):
        ref, c = oracle_step(w, layer)
        assert_close(outs[layer], ref, f"fused mix layer {layer}")
        pages = w.block_tables[layer, np.arange(w.batch), pos // 16]
        got = synth.bits(d["pool"][torch.from_numpy(pages).long().to(dev), :,
                                   torch.from_numpy(pos % 16).long().to(dev)])
        want = c.pool[c.block_table[np.arange(w.batch), pos // 16], :, pos % 16]
        assert np.array_equal(got, want), f"appended slots, layer {layer}"


@pytest.mark.parametrize("splits", [0, 2])
def test_fused_ragged_lengths_with_empty_sequences(splits):
    dev = cuda_or_skip()
    lens = [0, 1, 2, 15, 16, 17, 33, 2048, 0, 500]
    w = synth.make_workload("edge", 9, seq_lens=lens, num_pages=512)
    d = synth.device_inputs(w, dev)
    before = synth.bits(d["pool"])
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = synth.bits(fused(w, d, 0, num_splits=splits, dev_err=err))
    live = np.nonzero(w.seq_lens > 0)[0]
    ref, _ = oracle_step(w, 0, live)
    assert_close(out[live], ref, "fused ragged")
    for b in np.nonzero(w.seq_lens == 0)[0]:
        assert np.all(out[b] == 0)
    # only the appended slots changed
    after = synth.bits(d["pool"])
    changed = np.argwhere(np.any(after != before, axis=(3, 4)))
    want = {(int(w.block_tables[0, b, (L - 1) // 16]), kv, (L - 1) % 16)
            for b, L in enumerate(lens) if L > 0 for kv in (0, 1)}
    assert {tuple(map(int, c)) for c in changed} <= want
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_fused_bad_last_block_is_reported():
    dev = cuda_or_skip()
    w = synth.make_workload("edge", 10, seq_lens=[40, 20], num_pages=64)
    d = synth.device_inputs(w, dev)
    bt = d["block_tables"][0].clone()
    bt[0, 2] = 1000          # the block holding position 39
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    b = binding()
    out = b.decode_step(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], bt, d["seq_lens"],
                        dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & b.DEVERR_PAGE
    ref, _ = oracle_step(w, 0, [1])
    assert_close(synth.bits(out)[1:], ref, "untouched sequence")
