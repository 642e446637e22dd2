"""GPU parity of the split plans on ragged batches: the automatic plan
(num_splits = 0) and explicit ones with short ranges (deep per-warp page
ring, 3 CTAs per SM) and long ranges (shallow ring, 4 CTAs per SM).

Outputs are checked against the FP64 oracle with the attention tolerance of
_gpu_util; the fused step must equal append + attention bit for bit under the
same plan, and repeated calls must give identical bits.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip

pytestmark = pytest.mark.gpu


def case(lens, seed=11, num_pages=None, max_blocks=128):
    """Host pool holding every token of every sequence, plus device copies."""
    lens = np.asarray(lens, np.int32)
    pages = int(sum((int(L) + 15) // 16 for L in lens))
    w = synth.make_workload("edge", seed, seq_lens=lens,
                            num_pages=num_pages or max(64, pages + 16), max_blocks=max_blocks)
    pool = synth.host_pool(w)
    live = np.nonzero(w.seq_lens > 0)[0]
    if len(live):
        assert oracle.kv_append(w.k_new[0][live], w.v_new[0][live], pool,
                                w.block_tables[0][live], w.positions[live]) == 0
    return w, pool


def dev_bf16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def attend(w, pool_dev, dev, lens=None, err=None, num_splits=0):
    lens = w.seq_lens if lens is None else lens
    return binding().paged_decode_attention(
        dev_bf16(w.q[0], dev), pool_dev, torch.from_numpy(w.block_tables[0]).to(dev),
        torch.from_numpy(np.asarray(lens, np.int32)).to(dev), num_splits=num_splits,
        dev_err=err)


def mixed_lengths(rng, n_short, n_long):
    lens = np.concatenate([rng.integers(16, 129, n_short), rng.integers(1536, 2049, n_long)])
    return rng.permutation(lens).astype(np.int32)


@pytest.mark.parametrize("seed,splits", [(0, 0), (1, 0), (0, 3), (0, 16)])
def test_mixed_batch_every_output(seed, splits):
    # 115 short (16..128 tokens) and 13 long (1536..2048) sequences, shuffled
    dev = cuda_or_skip()
    lens = mixed_lengths(np.random.default_rng(seed), 115, 13)
    w, pool = case(lens, seed=seed)
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pool_dev = dev_bf16(pool, dev)
    got = synth.bits(attend(w, pool_dev, dev, err=err, num_splits=splits))
    assert_close(got, ref, f"mixed batch seed {seed} splits {splits}")
    again = synth.bits(attend(w, pool_dev, dev, err=err, num_splits=splits))
    assert np.array_equal(got, again)
    assert int(err.item()) == 0


def test_fused_step_equals_append_then_attention():
    dev = cuda_or_skip()
    lens = mixed_lengths(np.random.default_rng(5), 40, 6)
    w = synth.make_workload("edge", 5, seq_lens=lens, num_pages=2048)
    b = binding()
    outs, pools = [], []
    for fused in (False, True):
        d = synth.device_inputs(w, dev)
        bt = d["block_tables"][0]
        if fused:
            out = b.decode_step(d["q"][0], d["k_new"][0], d["v_new"][0], d["pool"], bt,
                                d["seq_lens"], rope_theta=w.rope_theta, scale=w.scale)
        else:
            b.kv_append(d["k_new"][0], d["v_new"][0], d["pool"], bt, d["positions"],
                        rope_theta=w.rope_theta)
            out = b.paged_decode_attention(d["q"][0], d["pool"], bt, d["seq_lens"],
                                           scale=w.scale)
        outs.append(synth.bits(out))
        pools.append(synth.bits(d["pool"]))
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(pools[0], pools[1])


@pytest.mark.parametrize("lens", [
    [0, 0, 0, 0, 0],                       # nothing to attend: zero rows
    [1],
    [2048],                                # one sequence over the whole table
    [2048] + [0] * 30,                     # one long sequence among empty ones
    [128 * 16, 8 * 16, 8 * 16 + 1, 16 * 16 - 1, 16 * 16, 16 * 16 + 1, 3],
    [0, 2048, 0, 1, 2047, 0],
])
@pytest.mark.parametrize("splits", [0, 2, 16])
def test_edge_batches(lens, splits):
    dev = cuda_or_skip()
    w, pool = case(lens)
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    got = synth.bits(attend(w, dev_bf16(pool, dev), dev, err=err, num_splits=splits))
    assert_close(got, ref, f"lens={lens} splits={splits}")
    for i, L in enumerate(lens):
        if L == 0:
            assert np.all(got[i] == 0)
    assert int(err.item()) == 0


@pytest.mark.parametrize("batch", [1024, 1025])
def test_large_ragged_batch(batch):
    # mostly short sequences plus a few long ones
    dev = cuda_or_skip()
    rng = np.random.default_rng(batch)
    lens = rng.integers(0, 65, batch).astype(np.int32)
    lens[rng.choice(batch, 6, replace=False)] = rng.integers(1024, 2049, 6)
    w, pool = case(lens, seed=batch)
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    got = synth.bits(attend(w, dev_bf16(pool, dev), dev, err=err))
    assert_close(got, ref, f"batch {batch}")
    assert int(err.item()) == 0


def test_bad_lengths_are_reported_and_clamped():
    dev = cuda_or_skip()
    w, pool = case([2048, 5, 700, 300])
    lens = w.seq_lens.copy()
    lens[0] = 128 * 16 + 9         # past the table: clamped to 2048
    lens[1] = -4                   # negative: an empty sequence
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    got = synth.bits(attend(w, dev_bf16(pool, dev), dev, lens=lens, err=err))
    assert int(err.item()) & binding().DEVERR_SEQLEN
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    assert_close(got[[0, 2, 3]], ref[[0, 2, 3]], "clamped and untouched sequences")
    assert np.all(got[1] == 0)


def test_static_scratch_automatic_plan_on_a_large_batch():
    # the allocation-free entry point with num_splits = 0 on 1024 sequences
    dev = cuda_or_skip()
    b = binding()
    batch = 1024
    assert b.workspace_bytes(batch, 128, 0) <= (4 << 20)
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 40, batch).astype(np.int32)
    w, pool = case(lens, seed=3)
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    f = b.lib().pkv_paged_decode_attention_static_ws
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [vp, vp, i64, vp, i32, vp, i32, i32, i32, i32, i32, ctypes.c_float, vp, i32,
                  vp, vp]
    f.restype = i32
    q = dev_bf16(w.q[0], dev)
    pool_dev = dev_bf16(pool, dev)
    bt = torch.from_numpy(w.block_tables[0]).to(dev)
    ln = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = f(p(q), p(pool_dev), w.num_pages, p(bt), 128, p(ln), batch, 32, 8, 64, 16, w.scale,
           p(out), 0, p(err), stream)
    assert rc == 0, b.strerror(rc)
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0
    assert_close(synth.bits(out), ref, "static scratch, batch 1024")
