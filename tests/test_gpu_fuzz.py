"""Seeded fuzz parity: random ragged batches through every attention route.

Each case draws a batch size, a table width and lengths (zeros, partial pages,
exact page multiples and full tables included), then runs the decode step
fused and as append + attention under the fixed automatic plan, a random
fixed split count and a host work plan.  Every output is checked against the
FP64 oracle, every appended slot bit for bit, and fused against unfused bit
for bit under the same plan.  The batch sizes straddle the SM count, so both
attention kernels and both merge kernels are reached.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip

pytestmark = pytest.mark.gpu


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    batch = [1, 3, 17, 64, 151, 152, 153, 200][seed % 8]   # straddling 152 SMs
    # large batches take narrower tables so the oracle stays within seconds
    max_blocks = int(rng.choice([8, 32] if batch >= 150 else [8, 32, 64, 128]))
    lmax = max_blocks * 16
    kind = rng.integers(0, 4)
    if kind == 0:
        lens = rng.integers(0, lmax + 1, batch)
    elif kind == 1:                                 # mostly short, a few full
        lens = rng.integers(0, min(lmax, 200) + 1, batch)
        lens[rng.choice(batch, max(1, batch // 10), replace=False)] = lmax
    elif kind == 2:                                 # page multiples and their neighbours
        lens = 16 * rng.integers(0, max_blocks + 1, batch) + rng.integers(-1, 2, batch)
    else:                                           # equal lengths
        lens = np.full(batch, int(rng.integers(1, lmax + 1)))
    lens = np.clip(lens, 0, lmax).astype(np.int32)
    splits = int(rng.integers(1, max(2, max_blocks // 4) + 1))
    return lens, max_blocks, splits


def case_inputs(lens, max_blocks, seed):
    pages = int(sum((int(L) + 15) // 16 for L in lens))
    w = synth.make_workload("edge", 2000 + seed, seq_lens=lens, num_pages=max(64, pages + 16),
                            max_blocks=max_blocks)
    pool = synth.host_pool(w)
    live = np.nonzero(w.seq_lens > 0)[0]
    if len(live):
        assert oracle.kv_append(w.k_new[0][live], w.v_new[0][live], pool,
                                w.block_tables[0][live], w.positions[live]) == 0
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    return w, pool, ref


@pytest.mark.parametrize("seed", range(12))
def test_random_batches_every_route(seed):
    dev = cuda_or_skip()
    lens, max_blocks, splits = draw_case(seed)
    w, host_pool, ref = case_inputs(lens, max_blocks, seed)
    b = binding()
    plan = b.Plan(w.seq_lens, max_blocks, device=dev)
    live = np.nonzero(w.seq_lens > 0)[0]
    for route in ("auto", f"S={splits}", "plan"):
        outs = {}
        for fused in (True, False):
            d = synth.device_inputs(w, dev)
            bt, sl = d["block_tables"][0], d["seq_lens"]
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            if not fused and len(live):
                # an empty sequence has no position to append at (kv_append would
                # skip and report it); the fused step appends nothing for it
                ix = torch.from_numpy(live).to(dev)
                b.kv_append(d["k_new"][0][ix].contiguous(), d["v_new"][0][ix].contiguous(),
                            d["pool"], bt[ix].contiguous(), d["positions"][ix].contiguous(),
                            dev_err=err)
            if route == "plan":
                if fused:
                    out = b.decode_step_planned(d["q"][0], d["k_new"][0], d["v_new"][0],
                                                d["pool"], bt, sl, plan, dev_err=err)
                else:
                    out = b.paged_decode_attention_planned(d["q"][0], d["pool"], bt, sl, plan,
                                                           dev_err=err)
            else:
                ns = 0 if route == "auto" else splits
                if fused:
                    out = b.decode_step(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], bt,
                                        sl, num_splits=ns, dev_err=err)
                else:
                    out = b.paged_decode_attention(d["q"][0], d["pool"], bt, sl, num_splits=ns,
                                                   dev_err=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0, (route, fused)
            outs[fused] = synth.bits(out)
            what = f"seed {seed} {route} fused={fused} B={len(lens)} max_blocks={max_blocks}"
            assert_close(outs[fused], ref, what)
            if fused and len(live):
                pool = synth.bits(d["pool"])
                pages = w.block_tables[0][live, w.positions[live] // 16]
                slots = w.positions[live] % 16
                assert np.array_equal(pool[pages, :, slots], host_pool[pages, :, slots]), what
        assert np.array_equal(outs[True], outs[False]), (seed, route)
