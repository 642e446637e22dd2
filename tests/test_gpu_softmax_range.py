"""GPU parity where the online softmax is stressed: scores whose maximum keeps
rising along the sequence (the running maximum is updated again and again,
across pages and across split ranges), falling scores, one dominant token,
identical keys, large random logits, alternating signs and a one-token
sequence.  Within one sequence the scores span up to ~150 in natural-log
units, beyond FP32's exp range (~88) without the running maximum.

The keys are built along one direction per (sequence, kv head) so that the
scores follow the wanted shape; every value is a bf16 input that the FP64
oracle reads too.  Routes: the automatic fixed plan, fixed plans of 4 and 16
splits, and a host work plan; attention only and the fused step (its appended
key is rotated by RoPE, so its score is whatever the rotation makes it).
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu_util import assert_close, binding, cuda_or_skip

pytestmark = pytest.mark.gpu

POISON = 0xFFFF
LENS = [2048, 2048, 1000, 513, 37, 16, 2048, 1]
PATTERNS = ["ramp_up", "ramp_down", "spike", "flat", "large", "alternate", "ramp_up", "large"]


def to_bf16_bits(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def key_rows(rng, pattern, L, u):
    """[L][64] float keys for one kv head along unit direction u (scores ~ q.k / 8)."""
    t = np.arange(L, dtype=np.float64)
    noise = 0.05 * rng.standard_normal((L, 64))
    if pattern == "ramp_up":
        a = -60 + 120 * t / max(L - 1, 1)        # q.k from -60*|q| to +60*|q|
    elif pattern == "ramp_down":
        a = 60 - 120 * t / max(L - 1, 1)
    elif pattern == "spike":
        a = np.full(L, -20.0)
        a[L // 2] = 60.0
    elif pattern == "flat":
        return np.tile(u * 3.0, (L, 1))          # identical keys: the mean of V
    elif pattern == "alternate":
        a = np.where(t % 2 == 0, 50.0, -50.0)
    else:                                        # large random logits
        return 12.0 * rng.standard_normal((L, 64))
    return a[:, None] * u[None, :] + noise


def build(seed):
    rng = np.random.default_rng(seed)
    B, mb = len(LENS), 128
    lens = np.asarray(LENS, np.int32)
    pages = [(L + 15) // 16 for L in LENS]
    num_pages = sum(pages) + 24
    perm = rng.permutation(num_pages)
    bt = np.full((B, mb), -1, np.int32)
    pool = np.full((num_pages, 2, 16, 8, 64), POISON, np.uint16)
    q = np.zeros((B, 32, 64), np.float64)
    at = 0
    for b, (L, pat) in enumerate(zip(LENS, PATTERNS)):
        bt[b, :pages[b]] = perm[at:at + pages[b]]
        at += pages[b]
        t = np.arange(L)
        k = np.zeros((L, 8, 64))
        for g in range(8):
            u = rng.standard_normal(64)
            u /= np.linalg.norm(u)
            k[:, g] = key_rows(rng, pat, L, u)
            for r in range(4):                   # 4 query rows of different strength
                q[b, 4 * g + r] = u * (4.0 + 2.0 * r) + 0.05 * rng.standard_normal(64)
        v = rng.standard_normal((L, 8, 64))
        page, slot = bt[b, t // 16], t % 16
        pool[page, 0, slot] = to_bf16_bits(k)
        pool[page, 1, slot] = to_bf16_bits(v)
    q = to_bf16_bits(q)
    k_new = to_bf16_bits(rng.standard_normal((B, 8, 64)))
    v_new = to_bf16_bits(rng.standard_normal((B, 8, 64)))
    return q, pool, bt, lens, k_new, v_new


def dev_u16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("route", ["auto", "S=4", "S=16", "plan"])
@pytest.mark.parametrize("fused", [False, True])
def test_softmax_extremes(route, fused):
    dev = cuda_or_skip()
    b = binding()
    q, pool, bt, lens, k_new, v_new = build(404)
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
    if route == "plan":
        plan = b.Plan(lens, 128, device=dev)
        if fused:
            out = b.decode_step_planned(dq, dev_u16(k_new, dev), dev_u16(v_new, dev), dpool, dbt,
                                        dl, plan, dev_err=err)
        else:
            out = b.paged_decode_attention_planned(dq, dpool, dbt, dl, plan, dev_err=err)
    else:
        ns = 0 if route == "auto" else int(route[2:])
        if fused:
            out = b.decode_step(dq, dev_u16(k_new, dev), dev_u16(v_new, dev), dpool, dbt, dl,
                                num_splits=ns, dev_err=err)
        else:
            out = b.paged_decode_attention(dq, dpool, dbt, dl, num_splits=ns, dev_err=err)
    got = bits(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got, ref, f"softmax extremes, {route}, fused={fused}")
