"""GPU parity of the shared-prefix kernel where its online softmax is
stressed: the shared pages' keys are built along each member's query
direction with a magnitude that rises (or spikes, or alternates) along the
prefix, so a row's running maximum keeps moving inside a shared range and the
kernel rescales its O rows in TMEM again and again, in both copies of the
rows (the copy weighing pages 0, 1 of each 4-page batch and the one weighing
pages 2, 3).  Private tails are ragged and moderate, so each member's result
merges shared and private partials of very different maxima.

Every value is a bf16 input that the FP64 oracle reads too.  Routes: the
shared plan (attention only and the fused step) and, as a control, the plan
from the lengths alone.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_util import assert_close, binding, cuda_or_skip

pytestmark = pytest.mark.gpu

POISON = 0xFFFF
GROUPS = 3                  # groups of 16 members
MEMBERS = 16
SHARED = [64, 37, 96]       # shared pages per group
PATTERNS = ["ramp_up", "spike", "alternate"]


def to_bf16_bits(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def shared_keys(rng, pattern, L, u):
    """[L][64] keys along unit direction u (scores ~ strength * a(t) / 8)."""
    t = np.arange(L, dtype=np.float64)
    if pattern == "ramp_up":
        a = -40 + 100 * t / max(L - 1, 1)
    elif pattern == "spike":
        a = np.full(L, -10.0)
        a[(7 * L) // 9] = 50.0
    else:
        a = np.where(t % 3 == 0, 45.0, -45.0) * (t / L)
    return a[:, None] * u[None, :] + 0.05 * rng.standard_normal((L, 64))


def build(seed):
    rng = np.random.default_rng(seed)
    B, mb = GROUPS * MEMBERS, 128
    own = rng.integers(1, 20 * 16, B)                    # private tail tokens, ragged
    lens = np.zeros(B, np.int32)
    for gi in range(GROUPS):
        for m in range(MEMBERS):
            b = gi * MEMBERS + m
            lens[b] = SHARED[gi] * 16 + own[b]
    pages = [(int(L) + 15) // 16 for L in lens]
    num_pages = sum(SHARED) + sum(p - SHARED[b // MEMBERS] for b, p in enumerate(pages)) + 16
    perm = rng.permutation(num_pages)
    bt = np.full((B, mb), -1, np.int32)
    pool = np.full((num_pages, 2, 16, 8, 64), POISON, np.uint16)
    q = np.zeros((B, 32, 64))
    at = 0
    for gi in range(GROUPS):
        S = SHARED[gi]
        shared_ids = perm[at:at + S]
        at += S
        dirs = rng.standard_normal((8, 64))
        dirs /= np.linalg.norm(dirs, axis=1, keepdims=True)
        k = np.zeros((S * 16, 8, 64))
        for h in range(8):
            k[:, h] = shared_keys(rng, PATTERNS[gi], S * 16, dirs[h])
        v = rng.standard_normal((S * 16, 8, 64))
        t = np.arange(S * 16)
        pool[shared_ids[t // 16], 0, t % 16] = to_bf16_bits(k)
        pool[shared_ids[t // 16], 1, t % 16] = to_bf16_bits(v)
        for m in range(MEMBERS):
            b = gi * MEMBERS + m
            n_own = pages[b] - S
            own_ids = perm[at:at + n_own]
            at += n_own
            bt[b, :S] = shared_ids
            bt[b, S:pages[b]] = own_ids
            L_own = int(lens[b]) - S * 16
            to = np.arange(L_own)
            pool[own_ids[to // 16], 0, to % 16] = to_bf16_bits(rng.standard_normal((L_own, 8, 64)))
            pool[own_ids[to // 16], 1, to % 16] = to_bf16_bits(rng.standard_normal((L_own, 8, 64)))
            for h in range(8):                           # 4 query rows of different strength
                for r in range(4):
                    s = 3.0 + 1.5 * r + 0.25 * m
                    q[b, 4 * h + r] = dirs[h] * s + 0.05 * rng.standard_normal(64)
    k_new = to_bf16_bits(rng.standard_normal((B, 8, 64)))
    v_new = to_bf16_bits(rng.standard_normal((B, 8, 64)))
    return to_bf16_bits(q), pool, bt, lens, k_new, v_new


def dev_u16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("shared_plan,sms", [(True, 0), (False, 0), (True, 8)])
@pytest.mark.parametrize("fused", [False, True])
def test_shared_prefix_softmax_extremes(shared_plan, sms, fused):
    # sms 8: the plan made as for 8 SMs is a segment plan, in which every
    # member's one own segment folds its shared partials into its output
    dev = cuda_or_skip()
    b = binding()
    q, pool, bt, lens, k_new, v_new = build(505)
    ref_pool = pool.copy()
    if fused:
        assert oracle.kv_append(k_new, v_new, ref_pool, bt, lens - 1) == 0
    else:
        # attention only reads what is there: the last slot holds a real token
        assert oracle.kv_append(k_new, v_new, pool, bt, lens - 1) == 0
        ref_pool = pool
    ref = oracle.decode_attention(q, ref_pool, bt, lens)
    assert np.all(np.isfinite(ref))
    dq, dpool = dev_u16(q, dev), dev_u16(pool, dev)
    dbt, dl = torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    plan = b.Plan(lens, bt.shape[1], device=dev, num_sms=sms,
                  block_tables=bt if shared_plan else None)
    if shared_plan:
        assert plan.num_shared >= GROUPS
        assert b.attention_kernels(len(lens), bt.shape[1], 0, plan).startswith(
            "paged_decode_shared_kernel+")
    else:
        assert plan.num_shared == 0
    if sms:
        assert plan.num_segs > 0 and plan.num_merges == 0
        assert (plan.segments()[:, 5] > 0).sum() == len(lens)
    if fused:
        out = b.decode_step_planned(dq, dev_u16(k_new, dev), dev_u16(v_new, dev), dpool, dbt, dl,
                                    plan, dev_err=err)
    else:
        out = b.paged_decode_attention_planned(dq, dpool, dbt, dl, plan, dev_err=err)
    got = bits(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got, ref, f"shared-prefix softmax extremes, shared_plan={shared_plan}, "
                           f"sms={sms}, fused={fused}")
