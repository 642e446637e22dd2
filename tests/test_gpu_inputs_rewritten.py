"""Inputs rewritten on the stream right before each call.  The attention
kernels read the lengths and block tables before griddepcontrol.wait (only
to prefetch pages into L2) and again after it; what they compute must come
from the values the preceding kernel wrote.  (A plan's device copy is filled
by a copy, never by the kernel just before the call, so the kernels use it
before the wait.)

The pool holds two copies of every sequence's pages with different K/V;
table variant A points at the first, variant B at the second.  A torch copy
kernel writes A or B (and, for the fixed plan, one of two length vectors)
into the table the call reads, alternating between calls.  Each output must
be the oracle's output for the variant written just before it.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, bf16_normal, binding, cuda_or_skip

pytestmark = pytest.mark.gpu


def two_variants(seed, whole_page_kernel=False):
    rng = np.random.default_rng(seed)
    if whole_page_kernel:           # a batch that fills the SMs: one CTA per sequence
        lens = np.full(160, 256, np.int32)
    else:
        lens = np.concatenate([rng.integers(1, 200, 40), rng.integers(1500, 2049, 6)])
        lens = rng.permutation(lens).astype(np.int32)
    B, mb = len(lens), 128
    pages = [(int(L) + 15) // 16 for L in lens]
    n = sum(pages)
    perm = rng.permutation(2 * n + 8)
    bt_a = np.full((B, mb), -1, np.int32)
    bt_b = np.full((B, mb), -1, np.int32)
    at = 0
    for b, p in enumerate(pages):
        bt_a[b, :p] = perm[at:at + p]
        bt_b[b, :p] = perm[n + at:n + at + p]
        at += p
    pool = bf16_normal(rng, (2 * n + 8, 2, 16, 8, 64))     # every slot a real value
    q = bf16_normal(rng, (B, 32, 64))
    lens_short = np.maximum(lens - rng.integers(0, 16, B).astype(np.int32), 1)
    return q, pool, lens, lens_short, bt_a, bt_b


def dev_u16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


@pytest.mark.parametrize("route", ["fixed", "plan", "whole_page"])
def test_tables_and_lengths_written_just_before_each_call(route):
    dev = cuda_or_skip()
    b = binding()
    q, pool, lens, lens_short, bt_a, bt_b = two_variants(12, route == "whole_page")
    if route == "whole_page":
        assert b.attention_kernels(len(lens), 128, 0) == "paged_decode_pagebox_kernel"
    variants = [(bt_a, lens), (bt_b, lens)]
    if route != "plan":             # the fixed plan reads the lengths on the device too
        variants += [(bt_a, lens_short), (bt_b, lens_short)]
    refs = [oracle.decode_attention(q, pool, bt, ln) for bt, ln in variants]
    dq, dpool = dev_u16(q, dev), dev_u16(pool, dev)
    src = [(torch.from_numpy(bt).to(dev), torch.from_numpy(ln).to(dev)) for bt, ln in variants]
    dbt = torch.empty_like(src[0][0])
    dl = torch.empty_like(src[0][1])
    plan = b.Plan(lens, 128, device=dev) if route == "plan" else None
    ws = torch.empty(max(16, b.workspace_bytes(len(lens), 128, 0),
                         plan.workspace_bytes if plan else 0), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    order = [i % len(variants) for i in range(24)]
    outs = []
    for i in order:
        dbt.copy_(src[i][0])        # a kernel on this stream, right before the call
        dl.copy_(src[i][1])
        if plan is None:
            out = b.paged_decode_attention(dq, dpool, dbt, dl, num_splits=0, workspace=ws,
                                           dev_err=err)
        else:
            out = b.paged_decode_attention_planned(dq, dpool, dbt, dl, plan, workspace=ws,
                                                   dev_err=err)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for k, (i, out) in enumerate(zip(order, outs)):
        assert_close(synth.bits(out), refs[i], f"{route} call {k} (variant {i})")
