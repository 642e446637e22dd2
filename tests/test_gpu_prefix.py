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


def test_prefix_full_size_sampled():
    dev = cuda_or_skip()
    w = synth.make_workload("prefix", 0)
    d = synth.device_inputs(w, dev)
    out = synth.bits(fused(w, d, d["block_tables"][0]))
    seqs = np.array([0, 1, 15, 16, 130, 255])
    ref, _ = oracle_step(w, 0, seqs)
    assert_close(out[seqs], ref, "prefix 256 x 2048 sampled")
