"""Seeded fuzz parity of shared-prefix plans (GPU).

Each case draws groups of consecutive sequences whose block tables start with
the same physical pages: group sizes 2..16, shared prefixes of 16..100 pages
(so shared ranges end on any page of a 4-page batch), singletons between the
groups, private tails of 1..27 pages whose last page is partly filled, and a
random minimum shared extent.  The decode step runs fused and as append +
attention under the plan built from the lengths and tables, for this device
and as for 8 SMs (mostly segment plans: folding members and merged ones).  Every output is
checked against the FP64 oracle, every appended slot bit for bit, and fused
against unfused bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, bf16_normal, binding, cuda_or_skip

pytestmark = pytest.mark.gpu

MAX_BLOCKS = 128


def draw_case(seed):
    rng = np.random.default_rng(7000 + seed)
    min_shared = int(rng.choice([16, 24, 32]))
    lens, rows, nxt, expect_shared = [], [], 0, False
    for _ in range(int(rng.integers(1, 6))):
        groups = [(1, 0)] if rng.random() < 0.5 else []
        groups.append((int(rng.integers(2, 17)), int(rng.integers(16, 101))))
        for size, k in groups:
            expect_shared |= size >= 2 and k >= min_shared
            common = list(range(nxt, nxt + k))
            nxt += k
            for _ in range(size):
                o = int(rng.integers(1, 28))
                rows.append(common + list(range(nxt, nxt + o)))
                nxt += o
                lens.append(16 * (k + o) - int(rng.integers(0, 16)))
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    perm = rng.permutation(nxt + 16).astype(np.int32)
    bt = np.full((B, MAX_BLOCKS), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = perm[r]
    pool = bf16_normal(rng, (nxt + 16, 2, 16, 8, 64))
    q = bf16_normal(rng, (B, 32, 64))
    kn = bf16_normal(rng, (B, 8, 64))
    vn = bf16_normal(rng, (B, 8, 64))
    return lens, bt, pool, q, kn, vn, min_shared, expect_shared


@pytest.mark.parametrize("sms", [0, 8])
@pytest.mark.parametrize("seed", range(8))
def test_random_shared_groups(seed, sms):
    # sms 8: the plan made as for 8 SMs is mostly a segment plan, in which
    # members whose own pages are one segment fold their shared partials and
    # members cut into several pieces are merged
    dev = cuda_or_skip()
    b = binding()
    lens, bt, pool, q, kn, vn, min_shared, expect_shared = draw_case(seed)
    ref_pool = pool.copy()
    assert oracle.kv_append(kn, vn, ref_pool, bt, lens - 1) == 0
    ref = oracle.decode_attention(q, ref_pool, bt, lens)

    def u16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
            torch.bfloat16)

    plan = b.Plan(lens, MAX_BLOCKS, device=dev, num_sms=sms, block_tables=bt,
                  min_shared_pages=min_shared)
    assert (plan.num_shared > 0) == expect_shared
    if expect_shared:
        assert b.attention_kernels(len(lens), MAX_BLOCKS, 0, plan).startswith(
            "paged_decode_shared_kernel+")
    dbt, dl = torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev)
    outs, pools = [], []
    for fused in (True, False):
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        dpool = u16(pool)
        if fused:
            out = b.decode_step_planned(u16(q), u16(kn), u16(vn), dpool, dbt, dl, plan,
                                        dev_err=err)
        else:
            b.kv_append(u16(kn), u16(vn), dpool, dbt, dl - 1, dev_err=err)
            out = b.paged_decode_attention_planned(u16(q), dpool, dbt, dl, plan, dev_err=err)
        got = synth.bits(out)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(got, ref, f"shared fuzz seed {seed}, sms={sms}, fused={fused}")
        outs.append(got)
        pools.append(synth.bits(dpool))
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(pools[0], ref_pool)  # appended slots, nothing else
    assert np.array_equal(pools[1], ref_pool)


def test_bad_page_in_shared_prefix_is_reported():
    # every member of a group names the same out-of-range page inside the
    # shared prefix: the shared-prefix kernel records PKV_DEVERR_PAGE, skips
    # that page and finishes (no timeout); outputs stay finite
    dev = cuda_or_skip()
    b = binding()
    lens, bt, pool, q, kn, vn, min_shared, _ = draw_case(3)
    plan0 = b.Plan(lens, MAX_BLOCKS, block_tables=bt, min_shared_pages=min_shared)
    sh = plan0.shared()
    assert len(sh) > 0
    members, p_begin = int(sh[0][0]), int(sh[0][1])
    seqs = [int(x) for x in sh[0][4:4 + members]]
    bad = bt.copy()
    for s in seqs:
        bad[s, p_begin + 2] = pool.shape[0] + 5
    plan = b.Plan(lens, MAX_BLOCKS, device=dev, block_tables=bad, min_shared_pages=min_shared)
    assert plan.num_shared == plan0.num_shared

    def u16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
            torch.bfloat16)

    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = b.paged_decode_attention_planned(u16(q), u16(pool), torch.from_numpy(bad).to(dev),
                                           torch.from_numpy(lens).to(dev), plan, dev_err=err)
    got = synth.bits(out)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & b.DEVERR_PAGE
    assert not e & b.DEVERR_TIMEOUT
    assert np.all(np.isfinite(oracle.bf16_to_f64(got)))


def draw_segment_case(seed):
    """Groups of 2..16 members sharing 16..60 pages with own tails of 16..60
    pages, singletons between them: large enough for segment plans."""
    rng = np.random.default_rng(9100 + seed)
    lens, rows, nxt = [], [], 0
    for _ in range(int(rng.integers(2, 6))):
        groups = [(1, 0)] if rng.random() < 0.3 else []
        groups.append((int(rng.integers(2, 17)), int(rng.integers(16, 61))))
        for size, k in groups:
            common = list(range(nxt, nxt + k))
            nxt += k
            for _ in range(size):
                o = int(rng.integers(16, 61))
                rows.append(common + list(range(nxt, nxt + o)))
                nxt += o
                lens.append(16 * (k + o) - int(rng.integers(0, 16)))
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    perm = rng.permutation(nxt + 16).astype(np.int32)
    bt = np.full((B, MAX_BLOCKS), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = perm[r]
    pool = bf16_normal(rng, (nxt + 16, 2, 16, 8, 64))
    q = bf16_normal(rng, (B, 32, 64))
    kn = bf16_normal(rng, (B, 8, 64))
    vn = bf16_normal(rng, (B, 8, 64))
    return lens, bt, pool, q, kn, vn


@pytest.mark.parametrize("sms", [16, 32, 48])
@pytest.mark.parametrize("seed", range(8))
def test_random_segment_plans_in_both_layouts(seed, sms):
    # planned as for 16, 32 and 48 SMs these are segment plans, some with
    # their segment CTAs beside the shared-prefix CTAs (layout 1) and some
    # with the shared-prefix CTAs first (layout 0); members fold or merge
    dev = cuda_or_skip()
    b = binding()
    lens, bt, pool, q, kn, vn = draw_segment_case(seed)
    ref_pool = pool.copy()
    assert oracle.kv_append(kn, vn, ref_pool, bt, lens - 1) == 0
    ref = oracle.decode_attention(q, ref_pool, bt, lens)

    def u16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
            torch.bfloat16)

    plan = b.Plan(lens, MAX_BLOCKS, device=dev, num_sms=sms, block_tables=bt)
    assert plan.num_shared > 0
    dbt, dl = torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev)
    outs = []
    for fused in (True, False):
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        dpool = u16(pool)
        if fused:
            out = b.decode_step_planned(u16(q), u16(kn), u16(vn), dpool, dbt, dl, plan,
                                        dev_err=err)
        else:
            b.kv_append(u16(kn), u16(vn), dpool, dbt, dl - 1, dev_err=err)
            out = b.paged_decode_attention_planned(u16(q), dpool, dbt, dl, plan, dev_err=err)
        got = synth.bits(out)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(got, ref, f"segment fuzz seed {seed}, sms={sms}, layout {plan.layout}, "
                               f"fused={fused}")
        assert np.array_equal(synth.bits(dpool), ref_pool)
        outs.append(got)
    assert np.array_equal(outs[0], outs[1])
