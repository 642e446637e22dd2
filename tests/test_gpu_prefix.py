"""Prefix-shared pages: block tables of several sequences alias the same
physical pages for a common prompt prefix (GPU).

The decode step must (1) match the oracle, which walks the same aliased
tables, (2) give bit-identical outputs to a batch where every sequence owns
private copies of those pages, and (3) leave the shared pages untouched (the
append only writes each sequence's private last page)."""
import numpy as np
import pytest
import torch

from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip, oracle_step

pytestmark = pytest.mark.gpu


def fused(w, d, bt, layer=0, **kw):
    return binding().decode_step(d["q"][layer], d["k_new"][layer], d["v_new"][layer], d["pool"],
                                 bt, d["seq_lens"], rope_theta=w.rope_theta, scale=w.scale, **kw)


def unshare(w, d):
    """A pool and table in which every follower has its own copy of the prefix pages."""
    S = synth.PREFIX_BLOCKS if w.name == "prefix" else None
    bt = d["block_tables"][0].clone()
    used = torch.zeros(w.num_pages, dtype=torch.bool, device=bt.device)
    used[bt[bt >= 0].long()] = True
    free = torch.nonzero(~used)[:, 0]
    pool = d["pool"].clone()
    cur = 0
    G = synth.PREFIX_GROUP
    for b in range(w.batch):
        if b % G == 0:
            continue
        new = free[cur:cur + S]
        cur += S
        pool[new] = d["pool"][bt[b, :S].long()]
        bt[b, :S] = new.int()
    return pool, bt


@pytest.mark.parametrize("splits", [0, 3])
def test_shared_prefix_matches_oracle_and_private_copies(splits):
    dev = cuda_or_skip()
    w = synth.make_workload("prefix", 1, batch=48, num_pages=12000)
    d = synth.device_inputs(w, dev)
    shared = torch.from_numpy(np.unique(w.block_tables[0, :, :synth.PREFIX_BLOCKS])).long().to(dev)
    before = d["pool"][shared].clone()
    pool2, bt2 = unshare(w, d)
    d2 = dict(d, pool=pool2)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    a = fused(w, d, d["block_tables"][0], num_splits=splits, dev_err=err)
    b = fused(w, d2, bt2, num_splits=splits, dev_err=err)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(d["pool"][shared].view(torch.int16), before.view(torch.int16))
    ref, _ = oracle_step(w, 0)
    assert_close(synth.bits(a), ref, f"shared prefix, splits={splits}")
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_prefix_full_size_every_output():
    dev = cuda_or_skip()
    w = synth.make_workload("prefix", 0)
    d = synth.device_inputs(w, dev)
    out = synth.bits(fused(w, d, d["block_tables"][0]))
    ref, _ = oracle_step(w, 0)
    assert_close(out, ref, "prefix 256 x 2048, every sequence")


# ------------------------------------------------ shared-prefix work plans --

def planned(w, d, plan, fused_step=True, **kw):
    b = binding()
    bt = d["block_tables"][0]
    if fused_step:
        return b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], bt,
                                     d["seq_lens"], plan, rope_theta=w.rope_theta, scale=w.scale,
                                     **kw)
    return b.paged_decode_attention_planned(d["q"][0], d["pool"], bt, d["seq_lens"], plan,
                                            scale=w.scale, **kw)


def test_shared_plan_matches_oracle_fused_and_unfused():
    # 48 sequences in groups of 16 sharing 96 pages: the plan makes groups of 8
    dev = cuda_or_skip()
    b = binding()
    w = synth.make_workload("prefix", 2, batch=48, num_pages=12000)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, block_tables=w.block_tables[0])
    assert plan.num_shared > 0
    assert b.attention_kernels(w.batch, w.max_blocks, 0, plan).startswith(
        "paged_decode_shared_kernel+")
    ref, c = oracle_step(w, 0)
    outs = []
    for fused_step in (True, False):
        d = synth.device_inputs(w, dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        if not fused_step:
            binding().kv_append(d["k_new"][0], d["v_new"][0], d["pool"], d["block_tables"][0],
                                d["positions"], rope_theta=w.rope_theta, dev_err=err)
        out = synth.bits(planned(w, d, plan, fused_step, dev_err=err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out, ref, f"shared plan, fused={fused_step}")
        outs.append(out)
    assert np.array_equal(outs[0], outs[1])
    # repeated calls give the same bits
    d = synth.device_inputs(w, dev)
    again = [synth.bits(planned(w, d, plan)) for _ in range(3)]
    assert all(np.array_equal(x, outs[0]) for x in again)


def test_shared_plan_full_size_every_output():
    # the prefix workload itself, in the benchmark's launch configuration:
    # 256 x 2048, 16-way shared 1536-token prefixes, the fused step under the
    # shared-prefix plan; every output and every appended slot
    dev = cuda_or_skip()
    b = binding()
    w = synth.make_workload("prefix", 0)
    d = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, block_tables=w.block_tables[0])
    assert plan.num_shared > 0
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = synth.bits(planned(w, d, plan, dev_err=err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, c = oracle_step(w, 0)
    assert_close(out, ref, "prefix 256 x 2048 under a shared plan, every sequence")
    pos = w.positions
    pages = w.block_tables[0, np.arange(w.batch), pos // 16]
    got = synth.bits(d["pool"][torch.from_numpy(pages).long().to(dev), :,
                               torch.from_numpy(pos % 16).long().to(dev)])
    want = c.pool[c.block_table[np.arange(w.batch), pos // 16], :, pos % 16]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("seq,page", [(5, 10), (15, 63), (17, 0), (30, 37)])
def test_shared_plan_with_a_diverging_member_table_is_reported(seq, page):
    # A shared plan says that every member's table holds the leader's page ids
    # over the shared ranges.  A member whose table says otherwise (a plan
    # built from another layer's tables, or tables changed since) would attend
    # the leader's pages; the kernel compares the tables, batch by batch, and
    # reports it -- for any member and any shared page (the first and last
    # member of a group, the first and last shared page).
    dev = cuda_or_skip()
    b = binding()
    w = synth.make_workload("prefix", 6, batch=32, num_pages=4096, share_group=16,
                            share_blocks=64)
    d = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, block_tables=w.block_tables[0])
    assert plan.num_shared > 0
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    planned(w, d, plan, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bt = d["block_tables"][0]
    bt[seq, page] = bt[20, 100]      # a valid page, but not the leader's shared one
    planned(w, d, plan, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & b.DEVERR_PLAN
    assert not int(err.item()) & (b.DEVERR_PAGE | b.DEVERR_TIMEOUT)


def test_shared_plan_ragged_groups():
    # groups of different sizes and prefix lengths, sequences in no group,
    # short own tails: every output against the oracle, fused
    import oracle
    from _gpu_util import bf16_normal
    dev = cuda_or_skip()
    b = binding()
    rng = np.random.default_rng(5)
    lens, rows, nxt = [], [], 0
    for size, k in [(3, 20), (1, 0), (8, 40), (2, 16), (5, 17), (1, 0)]:
        common = list(range(nxt, nxt + k))
        nxt += k
        for _ in range(size):
            o = int(rng.integers(1, 30))
            rows.append(common + list(range(nxt, nxt + o)))
            nxt += o
            lens.append(16 * (k + o) - int(rng.integers(0, 16)))
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    perm = rng.permutation(nxt + 32).astype(np.int32)
    bt = np.full((B, 128), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = perm[r]
    pool = bf16_normal(rng, (nxt + 32, 2, 16, 8, 64))
    q = bf16_normal(rng, (B, 32, 64))
    kn = bf16_normal(rng, (B, 8, 64))
    vn = bf16_normal(rng, (B, 8, 64))
    ref_pool = pool.copy()
    assert oracle.kv_append(kn, vn, ref_pool, bt, lens - 1) == 0
    ref = oracle.decode_attention(q, ref_pool, bt, lens)
    u16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
        torch.bfloat16)
    plan = b.Plan(lens, 128, device=dev, block_tables=bt)
    assert plan.num_shared > 0
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dpool = u16(pool)
    out = b.decode_step_planned(u16(q), u16(kn), u16(vn), dpool, torch.from_numpy(bt).to(dev),
                                torch.from_numpy(lens).to(dev), plan, dev_err=err)
    got = synth.bits(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got, ref, "ragged shared groups")
    assert np.array_equal(synth.bits(dpool), ref_pool)    # appended slots, nothing else


def test_folding_segment_plan_over_several_layers_in_one_call():
    # the prefix workload with 3 layers under one shared plan of member
    # segments that fold their shared partials (no merge): every layer's
    # shared-prefix kernel rewrites the partial slots the previous layer's
    # segments folded, so the multi-layer call must give the bits of one call
    # per layer, and the oracle's outputs
    dev = cuda_or_skip()
    b = binding()
    w = synth.make_workload("prefix", 6, layers=3)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, block_tables=w.block_tables[0])
    assert plan.num_segs > 0 and plan.num_merges == 0
    assert (plan.segments()[:, 5] > 0).sum() == w.batch
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    d = synth.device_inputs(w, dev)
    one = np.stack([synth.bits(b.decode_step_planned(
        d["q"][layer], d["k_new"][layer], d["v_new"][layer], d["pool"],
        d["block_tables"][layer], d["seq_lens"], plan, rope_theta=w.rope_theta, scale=w.scale,
        dev_err=err)) for layer in range(w.layers)])
    pool_one = synth.bits(d["pool"])
    del d
    d = synth.device_inputs(w, dev)
    many = synth.bits(b.decode_steps_planned(
        d["q"], d["k_new"], d["v_new"], d["pool"], d["block_tables"], d["seq_lens"], plan,
        rope_theta=w.rope_theta, scale=w.scale, dev_err=err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(many, one)
    assert np.array_equal(synth.bits(d["pool"]), pool_one)
    for layer in (1, 2):
        ref, _ = oracle_step(w, layer)
        assert_close(one[layer], ref, f"prefix layer {layer} under a folding segment plan")


@pytest.mark.parametrize("sms, layout", [(24, 0), (48, 1)])
def test_layers_of_folding_and_merged_members_in_both_layouts(sms, layout):
    # 48 sequences in 4 groups (16 members sharing 48 pages, 8 sharing 30),
    # own tails of 8..70 pages: planned as for 24 SMs the shared-prefix CTAs
    # run first (layout 0); as for 48 SMs the segment CTAs run beside them
    # (layout 1).  Either way some members fold their shared partial in their
    # one segment and others, cut into pieces, go through the merge kernel.
    # Three layers in one call (each layer's kernels reuse the partial slots
    # the previous layer's merge and folds read) must give the bits of one
    # call per layer, and the oracle's outputs.
    import oracle
    from _gpu_util import bf16_normal
    dev = cuda_or_skip()
    b = binding()
    rng = np.random.default_rng(1)
    lens, rows, nxt = [], [], 0
    for size, k in [(16, 48)] * 2 + [(8, 30)] * 2:
        common = list(range(nxt, nxt + k))
        nxt += k
        for _ in range(size):
            o = int(rng.integers(8, 71))
            rows.append(common + list(range(nxt, nxt + o)))
            nxt += o
            lens.append(16 * (k + o) - int(rng.integers(0, 16)))
    lens = np.asarray(lens, np.int32)
    B, L, P = len(lens), 3, nxt + 16
    bt = np.full((L, B, 128), -1, np.int32)
    for layer in range(L):                 # each layer: the same sharing, its own pages
        perm = rng.permutation(P).astype(np.int32) + layer * P
        for i, r in enumerate(rows):
            bt[layer, i, :len(r)] = perm[r]
    pool = bf16_normal(rng, (L * P, 2, 16, 8, 64))
    q = bf16_normal(rng, (L, B, 32, 64))
    kn = bf16_normal(rng, (L, B, 8, 64))
    vn = bf16_normal(rng, (L, B, 8, 64))
    plan = b.Plan(lens, 128, device=dev, num_sms=sms, block_tables=bt[0])
    assert plan.layout == layout and plan.num_segs > 0 and plan.num_merges > 0
    assert (plan.segments()[:, 5] > 0).any()

    def u16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
            torch.bfloat16)
    dbt, dl = torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pool_one = u16(pool)
    one = np.stack([synth.bits(b.decode_step_planned(
        u16(q[layer]), u16(kn[layer]), u16(vn[layer]), pool_one, dbt[layer], dl, plan,
        dev_err=err)) for layer in range(L)])
    pool_many = u16(pool)
    many = synth.bits(b.decode_steps_planned(u16(q), u16(kn), u16(vn), pool_many, dbt, dl, plan,
                                             dev_err=err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(many, one)
    ref_pool = pool.copy()
    for layer in range(L):
        assert oracle.kv_append(kn[layer], vn[layer], ref_pool, bt[layer], lens - 1) == 0
        ref = oracle.decode_attention(q[layer], ref_pool, bt[layer], lens)
        assert_close(one[layer], ref, f"layer {layer}, layout {layout}")
    assert np.array_equal(synth.bits(pool_one), ref_pool)
    assert np.array_equal(synth.bits(pool_many), ref_pool)


@pytest.mark.parametrize("sms", [24, 48, 152])
def test_long_shared_prefixes_beside(sms):
    # 1024-entry tables: groups of 8, 8 and 6 sequences sharing 400, 250 and
    # 600 pages, own tails of 100..300 pages (up to 14,208 tokens).  Planned as
    # for 24, 48 and 152 SMs these are beside-layout plans with shared ranges
    # of 600, 300 and 100 pages and segment CTAs of up to 258 pages; some
    # members fold, others are merged.  Fused step against the oracle.
    import oracle
    from _gpu_util import bf16_normal
    dev = cuda_or_skip()
    b = binding()
    mb = 1024
    rng = np.random.default_rng(3)
    lens, rows, nxt = [], [], 0
    for size, k in [(8, 400), (8, 250), (6, 600)]:
        common = list(range(nxt, nxt + k))
        nxt += k
        for _ in range(size):
            o = int(rng.integers(100, 301))
            rows.append(common + list(range(nxt, nxt + o)))
            nxt += o
            lens.append(16 * (k + o) - int(rng.integers(0, 16)))
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    bt = np.full((B, mb), -1, np.int32)
    perm = np.random.default_rng(4).permutation(nxt + 16).astype(np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = perm[r]
    pool = bf16_normal(rng, (nxt + 16, 2, 16, 8, 64))
    q = bf16_normal(rng, (B, 32, 64))
    kn = bf16_normal(rng, (B, 8, 64))
    vn = bf16_normal(rng, (B, 8, 64))
    ref_pool = pool.copy()
    assert oracle.kv_append(kn, vn, ref_pool, bt, lens - 1) == 0
    ref = oracle.decode_attention(q, ref_pool, bt, lens)
    plan = b.Plan(lens, mb, device=dev, num_sms=sms, block_tables=bt)
    assert plan.layout == 1 and plan.num_shared > 0 and plan.num_merges > 0

    def u16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
            torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dpool = u16(pool)
    out = b.decode_step_planned(u16(q), u16(kn), u16(vn), dpool, torch.from_numpy(bt).to(dev),
                                torch.from_numpy(lens).to(dev), plan, dev_err=err)
    got = synth.bits(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got, ref, f"long shared prefixes, sms={sms}")
    assert np.array_equal(synth.bits(dpool), ref_pool)
