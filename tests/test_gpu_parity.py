"""GPU parity of the decode step (KV append + paged decode attention) against the
FP64 CPU oracle, through the C-ABI binding.

Appended K/V slots must match the oracle bit for bit; attention outputs must be
within |err| <= 1e-3 + 8e-3 * |ref| element-wise, on every output, the
full-size workloads (256 x 2048, and the 16-layer 8 GiB-pool mix) included.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import (appended_slots_expected, assert_close, binding, cuda_or_skip,
                       equal_but_nan_payload, gpu_step, oracle_step, special_bf16)

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=2)
def workload(name, seed=0):
    return synth.make_workload(name, seed)


def upload(w):
    return synth.device_inputs(w, cuda_or_skip())


def new_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------- small, exhaustive --

@pytest.mark.parametrize("name", ["tiny", "small", "long"])
def test_step_matches_oracle_everywhere(name):
    w = workload(name)
    d = upload(w)
    err = new_err()
    for layer in range(w.layers):
        out = gpu_step(w, d, layer, dev_err=err)
        ref, _ = oracle_step(w, layer)
        assert_close(synth.bits(out), ref, f"{name} layer {layer}")
        kexp, vexp = appended_slots_expected(w, layer, range(w.batch))
        pool = d["pool"]
        for b in range(w.batch):
            pos = int(w.positions[b])
            page = int(w.block_tables[layer, b, pos // 16])
            assert np.array_equal(synth.bits(pool[page, 0, pos % 16]), kexp[b]), (layer, b)
            assert np.array_equal(synth.bits(pool[page, 1, pos % 16]), vexp[b]), (layer, b)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


@pytest.mark.parametrize("name", ["tiny", "small", "long"])
def test_append_touches_nothing_else(name):
    w = workload(name)
    d = upload(w)
    for layer in range(w.layers):
        gpu_step(w, d, layer)
    expect = synth.host_pool(w)
    for layer in range(w.layers):
        kexp, vexp = appended_slots_expected(w, layer, range(w.batch))
        for b in range(w.batch):
            pos = int(w.positions[b])
            page = int(w.block_tables[layer, b, pos // 16])
            expect[page, 0, pos % 16] = kexp[b]
            expect[page, 1, pos % 16] = vexp[b]
    assert np.array_equal(synth.bits(d["pool"]), expect)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8, 16, 32, 128])
@pytest.mark.parametrize("name", ["small", "long"])
def test_every_split_count_matches_oracle(name, splits):
    w = workload(name)
    d = upload(w)
    layer = 0
    out = gpu_step(w, d, layer, num_splits=splits)
    ref, _ = oracle_step(w, layer)
    assert_close(synth.bits(out), ref, f"{name} splits={splits}")


@pytest.mark.parametrize("splits", [0, 1, 4, 32])
def test_same_inputs_give_identical_bits(splits):
    w = workload("small")
    d = upload(w)
    b = binding()
    gpu_step(w, d, 0)  # append once; attention is then re-run on a fixed pool
    outs = [b.paged_decode_attention(d["q"][0], d["pool"], d["block_tables"][0], d["seq_lens"],
                                     num_splits=splits) for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_page_permutation_is_bit_invisible():
    w = workload("small")
    d = upload(w)
    b = binding()
    gpu_step(w, d, 0)
    base = b.paged_decode_attention(d["q"][0], d["pool"], d["block_tables"][0], d["seq_lens"])
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(w.num_pages, generator=g).to("cuda")  # new id of page p
    pool2 = torch.empty_like(d["pool"])
    pool2[perm] = d["pool"]
    bt = d["block_tables"][0]
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    for splits in (0, 1, 7):
        a = b.paged_decode_attention(d["q"][0], d["pool"], bt, d["seq_lens"], num_splits=splits)
        c = b.paged_decode_attention(d["q"][0], pool2, bt2, d["seq_lens"], num_splits=splits)
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
    assert torch.equal(base.view(torch.int16),
                       b.paged_decode_attention(d["q"][0], pool2, bt2, d["seq_lens"]).view(torch.int16))


# ------------------------------------------------------------ full size, sampled --

def test_peak_full_size_every_output():
    w = workload("peak")
    d = upload(w)
    err = new_err()
    out = gpu_step(w, d, 0, dev_err=err)   # 256 x 2048, the two-kernel path, automatic split plan
    got = synth.bits(out)
    ref, _ = oracle_step(w, 0)             # every sequence, all host cores
    assert_close(got, ref, "peak, every output")
    # the appended slots of all 256 sequences, bit for bit
    kexp, vexp = appended_slots_expected(w, 0, range(w.batch))
    pos = torch.from_numpy(w.positions.astype(np.int64)).cuda()
    pages = d["block_tables"][0].long().gather(1, (pos // 16)[:, None])[:, 0]
    slots = d["pool"][pages, :, pos % 16]     # [B][2][Hkv][D]
    sb = synth.bits(slots)
    assert np.array_equal(sb[:, 0], kexp) and np.array_equal(sb[:, 1], vexp)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_mix_full_size_every_output():
    w = workload("mix")
    d = upload(w)
    err = new_err()
    outs = [synth.bits(gpu_step(w, d, layer, dev_err=err)) for layer in range(w.layers)]
    for layer in range(w.layers):          # every sequence of every layer
        ref, _ = oracle_step(w, layer)
        assert_close(outs[layer], ref, f"mix layer {layer}")
    torch.cuda.synchronize()
    assert int(err.item()) == 0


# ------------------------------------------------------------------ edge cases --

def attention_only_case(lens, seed=3, num_pages=512):
    """Host pool already holding every token (oracle append applied on the host)."""
    w = synth.make_workload("edge", seed, seq_lens=lens, num_pages=num_pages)
    pool = synth.host_pool(w)
    live = np.nonzero(w.seq_lens > 0)[0]
    if len(live):
        rc = oracle.kv_append(w.k_new[0][live], w.v_new[0][live], pool,
                              w.block_tables[0][live], w.positions[live])
        assert rc == 0
    return w, pool


@pytest.mark.parametrize("lens", [[0], [1], [15], [16], [17], [2048], [0, 1, 2, 31, 32, 33, 47, 2048],
                                  [1] * 40, [2048, 3, 1999, 64, 65]])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_ragged_and_degenerate_lengths(lens, splits):
    dev = cuda_or_skip()
    w, pool = attention_only_case(lens)
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    b = binding()
    err = new_err()
    out = b.paged_decode_attention(
        torch.from_numpy(w.q[0].view(np.int16)).to(dev).view(torch.bfloat16),
        torch.from_numpy(pool.view(np.int16)).to(dev).view(torch.bfloat16),
        torch.from_numpy(w.block_tables[0]).to(dev), torch.from_numpy(w.seq_lens).to(dev),
        num_splits=splits, dev_err=err)
    got = synth.bits(out)
    assert_close(got, ref, f"lens={lens} splits={splits}")
    for i, L in enumerate(lens):
        if L == 0:
            assert np.all(got[i] == 0)        # defined as a zero row, never NaN
    assert int(err.item()) == 0


def test_bad_page_id_is_reported_and_skipped():
    dev = cuda_or_skip()
    w, pool = attention_only_case([40, 33, 20])
    bt = w.block_tables[0].copy()
    bt[1, 1] = w.num_pages + 5     # out of range
    bt[2, 0] = -3                  # negative
    b = binding()
    err = new_err()
    out = b.paged_decode_attention(
        torch.from_numpy(w.q[0].view(np.int16)).to(dev).view(torch.bfloat16),
        torch.from_numpy(pool.view(np.int16)).to(dev).view(torch.bfloat16),
        torch.from_numpy(bt).to(dev), torch.from_numpy(w.seq_lens).to(dev), dev_err=err)
    got = synth.bits(out)
    assert int(err.item()) & b.DEVERR_PAGE
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    assert_close(got[:1], ref[:1], "untouched sequence")
    assert np.all(np.isfinite(oracle.bf16_to_f64(got)))


def test_bad_seq_len_is_reported_and_clamped():
    dev = cuda_or_skip()
    w, pool = attention_only_case([2048, 5])
    lens = w.seq_lens.copy()
    lens[0] = 128 * 16 + 1
    lens[1] = -4
    b = binding()
    err = new_err()
    out = b.paged_decode_attention(
        torch.from_numpy(w.q[0].view(np.int16)).to(dev).view(torch.bfloat16),
        torch.from_numpy(pool.view(np.int16)).to(dev).view(torch.bfloat16),
        torch.from_numpy(w.block_tables[0]).to(dev), torch.from_numpy(lens).to(dev),
        dev_err=err)
    assert int(err.item()) & b.DEVERR_SEQLEN
    got = synth.bits(out)
    ref = oracle.decode_attention(w.q[0], pool, w.block_tables[0], w.seq_lens)
    assert_close(got[:1], ref[:1], "clamped to the table width")
    assert np.all(got[1] == 0)


def test_append_bad_position_and_page_are_skipped():
    dev = cuda_or_skip()
    w = workload("small")
    d = upload(w)
    b = binding()
    before = synth.bits(d["pool"])
    pos = d["positions"].clone()
    pos[0] = -1
    pos[1] = 128 * 16
    bt = d["block_tables"][0].clone()
    bt[2, int(w.positions[2]) // 16] = w.num_pages
    keep = torch.tensor([0, 1, 2], device=dev)
    err = new_err()
    b.kv_append(d["k_new"][0][keep].contiguous(), d["v_new"][0][keep].contiguous(), d["pool"],
                bt[keep].contiguous(), pos[keep].contiguous(), dev_err=err)
    e = int(err.item())
    assert e & b.DEVERR_POSITION and e & b.DEVERR_PAGE
    assert np.array_equal(synth.bits(d["pool"]), before)


def test_query_rotation_bit_exact():
    dev = cuda_or_skip()
    w = workload("small")
    d = upload(w)
    b = binding()
    q_out = torch.empty_like(d["q"][0])
    b.kv_append(d["k_new"][0], d["v_new"][0], d["pool"], d["block_tables"][0], d["positions"],
                q_in=d["q"][0], q_out=q_out)
    want = oracle.rope_queries(w.q[0], w.positions, w.rope_theta)
    assert np.array_equal(synth.bits(q_out), want)


def test_rope_over_every_position_bit_exact():
    # One sequence per position 0..2047 (each in its own page), so every
    # (position, frequency) pair of the 2048-token context is exercised.
    dev = cuda_or_skip()
    B = 2048
    rng = np.random.default_rng(17)
    k = torch.from_numpy(rng.standard_normal((B, 8, 64)).astype(np.float32)).to(torch.bfloat16)
    kb = k.view(torch.int16).numpy().view(np.uint16)
    bt = np.full((B, 128), -1, np.int32)
    pos = np.arange(B, dtype=np.int32)
    bt[np.arange(B), pos // 16] = np.arange(B)
    pool = torch.full((B, 2, 16, 8, 64), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
    b = binding()
    kd = k.to(dev)
    b.kv_append(kd, kd, pool, torch.from_numpy(bt).to(dev), torch.from_numpy(pos).to(dev))
    got = synth.bits(pool[torch.arange(B, device=dev), 0, torch.from_numpy(pos % 16).long().to(dev)])
    want = np.stack([np.stack([oracle.rope_rotate(kb[i, h], i, 500000.0) for h in range(8)])
                     for i in range(B)])
    mism = np.argwhere(got != want)
    assert mism.size == 0, f"{len(mism)} mismatches, first {mism[:4].tolist()}"


def test_rope_beyond_the_table_and_theta_switch_bit_exact():
    # positions 2048..4095 (past the per-device cos/sin table) take the
    # in-kernel sincos path; switching theta rebuilds the table in between.
    dev = cuda_or_skip()
    B = 512
    rng = np.random.default_rng(23)
    k = torch.from_numpy(rng.standard_normal((B, 8, 64)).astype(np.float32)).to(torch.bfloat16)
    kb = k.view(torch.int16).numpy().view(np.uint16)
    b = binding()
    for theta, base in ((500000.0, 2048), (10000.0, 0), (500000.0, 1536), (10000.0, 3000)):
        pos = (base + np.arange(B) * 2).astype(np.int32)
        bt = np.full((B, 256), -1, np.int32)
        bt[np.arange(B), pos // 16] = np.arange(B)
        pool = torch.full((B, 2, 16, 8, 64), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
        kd = k.to(dev)
        b.kv_append(kd, kd, pool, torch.from_numpy(bt).to(dev), torch.from_numpy(pos).to(dev),
                    rope_theta=theta)
        got = synth.bits(pool[torch.arange(B, device=dev), 0,
                              torch.from_numpy(pos % 16).long().to(dev)])
        want = np.stack([np.stack([oracle.rope_rotate(kb[i, h], int(pos[i]), theta)
                                   for h in range(8)]) for i in range(B)])
        assert np.array_equal(got, want), (theta, base)


@pytest.mark.parametrize("fused", [False, True])
def test_append_special_values_bit_exact(fused):
    # zeros, subnormals, tiny/huge normals, inf, NaN and cancelling pairs in the
    # new keys, at positions inside and past the cos/sin table; the fused step
    # appends through its own copy of the rotation.  NaN payloads are not compared.
    dev = cuda_or_skip()
    rng = np.random.default_rng(31)
    B = 640
    pos = np.concatenate([rng.integers(0, 2048, B - 64), rng.integers(2048, 4096, 64)])
    pos = pos.astype(np.int32)
    k = special_bf16(rng, (B, 8, 64))
    v = special_bf16(rng, (B, 8, 64))
    # sequence i appends into page i; the fused step also attends over the
    # earlier blocks, which all point at one extra zero page (index B)
    bt = np.full((B, 256), -1, np.int32)
    for i in range(B):
        bt[i, :pos[i] // 16] = B
    bt[np.arange(B), pos // 16] = np.arange(B)
    pool = torch.full((B + 1, 2, 16, 8, 64), 0x1234, dtype=torch.int16,
                      device=dev).view(torch.bfloat16)
    pool[B] = 0
    b = binding()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kd = torch.from_numpy(k.view(np.int16)).to(dev).view(torch.bfloat16)
    vd = torch.from_numpy(v.view(np.int16)).to(dev).view(torch.bfloat16)
    btd = torch.from_numpy(bt).to(dev)
    if fused:
        q = torch.zeros((B, 32, 64), dtype=torch.bfloat16, device=dev)
        b.decode_step(q, kd, vd, pool, btd, torch.from_numpy(pos + 1).to(dev), dev_err=err)
    else:
        b.kv_append(kd, vd, pool, btd, torch.from_numpy(pos).to(dev), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = synth.bits(pool[torch.arange(B, device=dev), :,
                          torch.from_numpy(pos % 16).long().to(dev)])
    for i in range(B):
        want_k = np.stack([oracle.rope_rotate(k[i, h], int(pos[i]), 500000.0) for h in range(8)])
        assert equal_but_nan_payload(got[i, 0], want_k).all(), (i, int(pos[i]))
        assert np.array_equal(got[i, 1], v[i]), i
