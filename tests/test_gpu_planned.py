"""GPU parity of the planned calls (pkv_*_planned): attention and the fused
step under a work plan built on the host from the lengths.

Outputs are checked against the FP64 oracle with the attention tolerance of
_gpu_util.  A plan that reproduces the fixed one-range-per-sequence split must
give the same bits as the unplanned call; the fused step must equal append +
attention bit for bit under the same plan; repeated calls give identical bits.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip

pytestmark = pytest.mark.gpu


def case(lens, seed=13, max_blocks=128):
    lens = np.asarray(lens, np.int32)
    pages = int(sum((int(L) + 15) // 16 for L in lens))
    w = synth.make_workload("edge", seed, seq_lens=lens, num_pages=max(64, pages + 16),
                            max_blocks=max_blocks)
    pool = synth.host_pool(w)
    live = np.nonzero(w.seq_lens > 0)[0]
    if len(live):
        assert oracle.kv_append(w.k_new[0][live], w.v_new[0][live], pool,
                                w.block_tables[0][live], w.positions[live]) == 0
    return w, pool


def dev_bf16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def planned_attention(w, pool_dev, dev, plan, lens=None, err=None):
    lens = w.seq_lens if lens is None else lens
    return binding().paged_decode_attention_planned(
        dev_bf16(w.q[0], dev), pool_dev, torch.from_numpy(w.block_tables[0]).to(dev),
        torch.from_numpy(np.asarray(lens, np.int32)).to(dev), plan, dev_err=err)


def mixed_lengths(rng, n_short, n_long):
    lens = np.concatenate([rng.integers(16, 129, n_short), rng.integers(1536, 2049, n_long)])
    return rng.permutation(lens).astype(np.int32)


@pytest.mark.parametrize("seed", [0, 1])
def test_mixed_batch_every_output(seed):
    dev = cuda_or_skip()
    lens = mixed_lengths(np.random.default_rng(seed), 115, 13)
    w, pool = case(lens, seed=seed)
    plan = binding().Plan(w.seq_lens, w.max_blocks, device=dev)
    assert plan.num_merges > 0 and any(plan.items()[:, 0] == 1)   # both item kinds
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pool_dev = dev_bf16(pool, dev)
    got = synth.bits(planned_attention(w, pool_dev, dev, plan, err=err))
    assert_close(got, ref, f"planned mixed batch seed {seed}")
    again = synth.bits(planned_attention(w, pool_dev, dev, plan, err=err))
    assert np.array_equal(got, again)
    assert int(err.item()) == 0


@pytest.mark.parametrize("lens", [
    [0, 0, 0, 0, 0],
    [1],
    [37],
    [2048],
    [2048] + [0] * 30,
    [128 * 16, 8 * 16, 8 * 16 + 1, 16 * 16 - 1, 16 * 16, 16 * 16 + 1, 3],
    [0, 2048, 0, 1, 2047, 0],
    list(range(1, 200, 7)),
])
def test_edge_batches(lens):
    dev = cuda_or_skip()
    w, pool = case(lens)
    plan = binding().Plan(w.seq_lens, w.max_blocks, device=dev)
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    got = synth.bits(planned_attention(w, dev_bf16(pool, dev), dev, plan, err=err))
    assert_close(got, ref, f"lens={lens}")
    for i, L in enumerate(lens):
        if L == 0:
            assert np.all(got[i] == 0)
    assert int(err.item()) == 0


def test_fused_step_equals_append_then_attention():
    dev = cuda_or_skip()
    lens = mixed_lengths(np.random.default_rng(5), 40, 6)
    w = synth.make_workload("edge", 5, seq_lens=lens, num_pages=2048)
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    outs, pools = [], []
    for fused in (False, True):
        d = synth.device_inputs(w, dev)
        bt = d["block_tables"][0]
        if fused:
            out = b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], bt,
                                        d["seq_lens"], plan, rope_theta=w.rope_theta,
                                        scale=w.scale)
        else:
            b.kv_append(d["k_new"][0], d["v_new"][0], d["pool"], bt, d["positions"],
                        rope_theta=w.rope_theta)
            out = b.paged_decode_attention_planned(d["q"][0], d["pool"], bt, d["seq_lens"], plan,
                                                   scale=w.scale)
        outs.append(synth.bits(out))
        pools.append(synth.bits(d["pool"]))
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(pools[0], pools[1])
    # and the appended slots are the oracle's
    c_pool = synth.host_pool(w)
    assert oracle.kv_append(w.k_new[0], w.v_new[0], c_pool, w.block_tables[0], w.positions) == 0
    live = w.block_tables[0][np.arange(w.batch), w.positions // 16]
    slots = w.positions % 16
    assert np.array_equal(pools[1][live, :, slots], c_pool[live, :, slots])


def test_uniform_plan_matches_the_unplanned_call_bit_for_bit():
    # 160 x 2048, planned as for a 16-SM part: a segment plan of whole
    # sequences, four per CTA (a plan made for another SM count is still
    # valid).  Each segment is attended exactly as the whole-page kernel
    # attends one sequence, which the fixed S = 1 split runs for this batch.
    dev = cuda_or_skip()
    w = synth.make_workload("edge", 21, seq_lens=np.full(160, 2048, np.int32), num_pages=20480)
    d = synth.device_inputs(w, dev)
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, num_sms=16, device=dev)
    assert plan.num_merges == 0 and plan.num_segs == 160 and plan.items()[:, 2].max() == 4
    assert b.attention_kernels(w.batch, w.max_blocks, 1) == "paged_decode_pagebox_kernel"
    bt = d["block_tables"][0]
    want = b.paged_decode_attention(d["q"][0], d["pool"], bt, d["seq_lens"], num_splits=1)
    got = b.paged_decode_attention_planned(d["q"][0], d["pool"], bt, d["seq_lens"], plan)
    assert np.array_equal(synth.bits(got), synth.bits(want))


def test_plan_mismatch_and_bad_pages_are_reported():
    dev = cuda_or_skip()
    w, pool = case([600, 40, 2048, 7])
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    pool_dev = dev_bf16(pool, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lens = w.seq_lens.copy()
    lens[1] += 1                                   # the device disagrees with the plan
    got = synth.bits(planned_attention(w, pool_dev, dev, plan, lens=lens, err=err))
    assert int(err.item()) & b.DEVERR_PLAN
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    assert_close(got, ref, "outputs follow the plan's lengths")
    err.zero_()
    bt = w.block_tables[0].copy()
    bt[2, 5] = w.num_pages + 3
    bt[3, 0] = -7
    out = b.paged_decode_attention_planned(
        dev_bf16(w.q[0], dev), pool_dev, torch.from_numpy(bt).to(dev),
        torch.from_numpy(w.seq_lens).to(dev), plan, dev_err=err)
    assert int(err.item()) & b.DEVERR_PAGE
    got = synth.bits(out)
    assert_close(got[:2], ref[:2], "untouched sequences")
    assert np.all(np.isfinite(oracle.bf16_to_f64(got)))


def test_plan_must_match_the_batch():
    dev = cuda_or_skip()
    w, pool = case([100, 200])
    b = binding()
    plan = b.Plan([100, 200, 300], w.max_blocks, device=dev)   # built for another batch
    with pytest.raises(b.PkvError):
        planned_attention(w, dev_bf16(pool, dev), dev, plan)


def test_mix_workload_planned_sampled():
    # the 16-layer mix workload in its benchmark form: one plan for all layers
    dev = cuda_or_skip()
    w = synth.make_workload("mix", 0)
    d = synth.device_inputs(w, dev)
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = []
    for layer in range(w.layers):
        outs.append(synth.bits(b.decode_step_planned(
            d["q"][layer], d["k_new"][layer], d["v_new"][layer], d["pool"],
            d["block_tables"][layer], d["seq_lens"], plan, rope_theta=w.rope_theta,
            scale=w.scale, dev_err=err)))
    from _gpu_util import oracle_step
    long_seqs = np.nonzero(w.seq_lens >= 1536)[0]
    short_seqs = np.nonzero(w.seq_lens <= 128)[0][:8]
    seqs = np.sort(np.concatenate([long_seqs, short_seqs]))
    for layer in (0, 15):
        ref, _ = oracle_step(w, layer, seqs)
        assert_close(outs[layer][seqs], ref, f"mix layer {layer}")
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_graph_replays_reuse_the_plan():
    # a captured planned call (attention + merge) replays to the eager result
    dev = cuda_or_skip()
    lens = mixed_lengths(np.random.default_rng(8), 60, 8)
    w = synth.make_workload("edge", 8, seq_lens=lens, num_pages=4096)
    d = synth.device_inputs(w, dev)
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    assert plan.num_merges > 0
    bt = d["block_tables"][0]
    ws = torch.empty(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
    want = b.paged_decode_attention_planned(d["q"][0], d["pool"], bt, d["seq_lens"], plan,
                                            workspace=ws)
    want_bits = synth.bits(want)
    out = torch.zeros_like(want)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.paged_decode_attention_planned(d["q"][0], d["pool"], bt, d["seq_lens"], plan, out,
                                         workspace=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(synth.bits(out), want_bits)


def test_all_layers_in_one_call_equal_per_layer_calls():
    # pkv_decode_steps_planned: the mix workload's 16 layers in one native call
    # give the bits of 16 single-layer calls, outputs and appended pages alike
    dev = cuda_or_skip()
    w = synth.make_workload("mix", 1)
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    d = synth.device_inputs(w, dev)
    one = [b.decode_step_planned(d["q"][layer], d["k_new"][layer], d["v_new"][layer], d["pool"],
                                 d["block_tables"][layer], d["seq_lens"], plan,
                                 rope_theta=w.rope_theta, scale=w.scale, dev_err=err)
           for layer in range(w.layers)]
    one = np.stack([synth.bits(o) for o in one])
    pool_one = synth.bits(d["pool"])
    del d
    d = synth.device_inputs(w, dev)
    many = b.decode_steps_planned(d["q"], d["k_new"], d["v_new"], d["pool"], d["block_tables"],
                                  d["seq_lens"], plan, rope_theta=w.rope_theta, scale=w.scale,
                                  dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(synth.bits(many), one)
    assert np.array_equal(synth.bits(d["pool"]), pool_one)
    from _gpu_util import oracle_step
    seqs = np.sort(np.concatenate([np.nonzero(w.seq_lens >= 1536)[0][:4],
                                   np.nonzero(w.seq_lens <= 128)[0][:4]]))
    ref, _ = oracle_step(w, 7, seqs)
    assert_close(one[7][seqs], ref, "mix layer 7 through the multi-layer call")


def test_multi_layer_call_checks_its_shapes():
    dev = cuda_or_skip()
    w = synth.make_workload("edge", 3, seq_lens=np.array([40, 17], np.int32), layers=2,
                            num_pages=64)
    d = synth.device_inputs(w, dev)
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    with pytest.raises(ValueError):
        b.decode_steps_planned(d["q"], d["k_new"][:1].contiguous(), d["v_new"], d["pool"],
                               d["block_tables"], d["seq_lens"], plan)
    with pytest.raises(b.PkvError):                 # a plan built for another batch
        b.decode_steps_planned(d["q"], d["k_new"], d["v_new"], d["pool"], d["block_tables"],
                               d["seq_lens"], b.Plan([40, 17, 5], w.max_blocks, device=dev))


def test_one_layer_multi_call_equals_the_single_layer_call():
    dev = cuda_or_skip()
    lens = mixed_lengths(np.random.default_rng(9), 30, 3)
    w = synth.make_workload("edge", 9, seq_lens=lens, num_pages=2048)
    b = binding()
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev)
    outs = []
    for multi in (False, True):
        d = synth.device_inputs(w, dev)
        if multi:
            out = b.decode_steps_planned(d["q"][:1], d["k_new"][:1], d["v_new"][:1], d["pool"],
                                         d["block_tables"][:1], d["seq_lens"], plan)[0]
        else:
            out = b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"],
                                        d["block_tables"][0], d["seq_lens"], plan)
        outs.append((synth.bits(out), synth.bits(d["pool"])))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("shape", ["per_head", "segments"])
def test_plans_swapped_by_copies_between_calls(shape):
    # The planned kernels read their plan before the grid dependency wait: a
    # plan's device copy is filled by a copy, which has finished before the
    # next kernel on the stream can start.  Two plans for different lengths
    # take turns in one device buffer, each copied in (with its lengths)
    # right before its call on the same stream; every call must give the
    # oracle's outputs for its own lengths.
    dev = cuda_or_skip()
    b = binding()
    rng = np.random.default_rng(21 if shape == "per_head" else 22)
    if shape == "per_head":
        lens_a = mixed_lengths(rng, 115, 13)
    else:
        lens_a = rng.integers(200, 1400, 320).astype(np.int32)
    lens_b = np.maximum(1, lens_a - rng.integers(0, 200, len(lens_a))).astype(np.int32)
    w, pool = case(lens_a, seed=23)
    plans = [b.Plan(lens, w.max_blocks) for lens in (lens_a, lens_b)]
    if shape == "per_head":
        assert all(p.num_segs == 0 and p.num_merges > 0 for p in plans)
    else:
        assert all(p.num_segs > 0 for p in plans)
    refs = [oracle.decode_attention(w.q[0], pool, w.block_tables[0], lens)
            for lens in (lens_a, lens_b)]
    staged = [torch.from_numpy(p.host.copy()).pin_memory() for p in plans]
    lens_pin = [torch.from_numpy(lens.copy()).pin_memory() for lens in (lens_a, lens_b)]
    dbuf = torch.empty(max(p.bytes_used for p in plans) // 4, dtype=torch.int32, device=dev)
    lens_dev = torch.empty(len(lens_a), dtype=torch.int32, device=dev)
    ws = torch.empty(max(16, max(p.workspace_bytes for p in plans)), dtype=torch.uint8,
                     device=dev)
    q, pool_dev = dev_bf16(w.q[0], dev), dev_bf16(pool, dev)
    bt = torch.from_numpy(w.block_tables[0]).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = []
    for i in range(6):
        k = i % 2
        p = plans[k]
        words = p.bytes_used // 4
        dbuf[:words].copy_(staged[k], non_blocking=True)
        lens_dev.copy_(lens_pin[k], non_blocking=True)
        p.dev = dbuf[:words]
        outs.append(b.paged_decode_attention_planned(q, pool_dev, bt, lens_dev, p, workspace=ws,
                                                     dev_err=err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for i, out in enumerate(outs):
        assert_close(synth.bits(out), refs[i % 2], f"{shape} call {i}")
