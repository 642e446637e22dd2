"""GPU parity at the largest batch the C ABI accepts (65535 sequences: the
grid's y limit), through the automatic fixed plan and a host work plan.

Attention only: the block tables alias a small 64-page pool (attention only
reads), so the whole batch is cheap; every output of the sampled sequences
and of the edge-case ones is checked against the FP64 oracle.  The fused
step: each sequence owns one page (so the appends never collide), the pool
is filled on the device, and the sampled sequences' pages are copied into a
small host pool (their block tables remapped) for the oracle; their appended
slots must match it bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_util import assert_close, bf16_normal, binding, cuda_or_skip

pytestmark = pytest.mark.gpu

B = 65535
SAMPLE = 2000


def dev_u16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def sample_of(rng, special):
    pick = rng.choice(B, SAMPLE, replace=False)
    return np.unique(np.concatenate([pick, np.asarray(special), np.arange(B - 8, B)]))


def test_max_batch_attention_fixed_and_planned():
    dev = cuda_or_skip()
    b = binding()
    rng = np.random.default_rng(65535)
    mb, P = 4, 64
    lens = rng.integers(0, mb * 16 + 1, B).astype(np.int32)
    special = np.arange(8)
    lens[special] = [0, 1, 15, 16, 17, 63, 64, 48]
    bt = rng.integers(0, P, (B, mb)).astype(np.int32)
    pool = bf16_normal(rng, (P, 2, 16, 8, 64))
    q = bf16_normal(rng, (B, 32, 64))
    dq, dpool = dev_u16(q, dev), dev_u16(pool, dev)
    dbt, dl = torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out_fixed = b.paged_decode_attention(dq, dpool, dbt, dl, num_splits=0, dev_err=err)
    plan = b.Plan(lens, mb, device=dev)
    assert plan.num_items <= 65535
    out_plan = b.paged_decode_attention_planned(dq, dpool, dbt, dl, plan, dev_err=err)
    got_fixed, got_plan = bits(out_fixed), bits(out_plan)
    assert int(err.item()) == 0
    seqs = sample_of(rng, special)
    ref = oracle.decode_attention(q[seqs], pool, bt[seqs], lens[seqs])
    assert_close(got_fixed[seqs], ref, "max batch, fixed plan")
    assert_close(got_plan[seqs], ref, "max batch, host plan")
    assert np.all(got_fixed[lens == 0] == 0) and np.all(got_plan[lens == 0] == 0)


def test_max_batch_fused_step_appends_and_attends():
    dev = cuda_or_skip()
    b = binding()
    rng = np.random.default_rng(65536)
    lens = rng.integers(1, 17, B).astype(np.int32)          # one page per sequence
    lens[:4] = [1, 16, 2, 15]
    pages = rng.permutation(B + 1)[:B].astype(np.int32)      # a distinct page each
    bt = pages[:, None].copy()
    g = torch.Generator(device=dev).manual_seed(7)
    dpool = torch.randn((B + 1, 2, 16, 8, 64), generator=g, device=dev, dtype=torch.bfloat16)
    dq = torch.randn((B, 32, 64), generator=g, device=dev, dtype=torch.bfloat16)
    dk = torch.randn((B, 8, 64), generator=g, device=dev, dtype=torch.bfloat16)
    dv = torch.randn((B, 8, 64), generator=g, device=dev, dtype=torch.bfloat16)
    seqs = sample_of(rng, np.arange(4))
    # the sampled sequences' pages before the append, in a small host pool
    rows = torch.from_numpy(pages[seqs].astype(np.int64)).to(dev)
    small = bits(dpool[rows])
    small_bt = np.arange(len(seqs), dtype=np.int32)[:, None]
    dbt, dl = torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = [b.decode_step(dq, dk, dv, dpool, dbt, dl, num_splits=0, dev_err=err)]
    plan = b.Plan(lens, 1, device=dev)
    # the second call appends the same rows to the same slots again
    outs.append(b.decode_step_planned(dq, dk, dv, dpool, dbt, dl, plan, dev_err=err))
    got = [bits(o)[seqs] for o in outs]
    after = bits(dpool[rows])
    assert int(err.item()) == 0
    q_h, k_h, v_h = bits(dq)[seqs], bits(dk)[seqs], bits(dv)[seqs]
    pos = lens[seqs] - 1
    assert oracle.kv_append(k_h, v_h, small, small_bt, pos) == 0
    ref = oracle.decode_attention(q_h, small, small_bt, lens[seqs])
    assert_close(got[0], ref, "max batch fused, fixed plan")
    assert_close(got[1], ref, "max batch fused, host plan")
    slot = pos % 16
    idx = np.arange(len(seqs))
    assert np.array_equal(after[idx, :, slot], small[idx, :, slot])
