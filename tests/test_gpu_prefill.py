"""GPU parity of the paged prefill write (pkv_kv_write_prefill) against the
oracle, bit for bit, and of prefill followed by a fused decode step."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, binding, cuda_or_skip, is_nan_bf16, special_bf16

pytestmark = pytest.mark.gpu

POISON = 0xFFFF


def bf16_normal(rng, shape):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def ragged_case(seed, counts, starts, num_pages=256, max_blocks=128, extents=None):
    rng = np.random.default_rng(seed)
    B = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(off[-1])
    k = bf16_normal(rng, (T, 8, 64))
    v = bf16_normal(rng, (T, 8, 64))
    bt = np.full((B, max_blocks), -1, np.int32)
    perm = rng.permutation(num_pages)
    cur = 0
    extents = counts if extents is None else extents
    for b in range(B):            # map only the blocks [start, start + extent) touches
        if extents[b] == 0:
            continue
        first, last = starts[b] // 16, (starts[b] + extents[b] - 1) // 16
        bt[b, first:last + 1] = perm[cur:cur + last - first + 1]
        cur += last - first + 1
    return k, v, off, np.asarray(starts, np.int32), bt


def to_dev(a, dev, bf=False):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf else np.ascontiguousarray(a))
    t = t.to(dev)
    return t.view(torch.bfloat16) if bf else t


@pytest.mark.parametrize("counts,starts", [
    ([37], [0]),
    ([20, 0, 5, 16, 1], [0, 3, 15, 16, 2047]),
    ([1] * 64, list(range(0, 64 * 31, 31))),
    ([300, 700, 2048, 1], [100, 0, 0, 900]),
])
def test_prefill_bit_exact(counts, starts):
    dev = cuda_or_skip()
    k, v, off, st, bt = ragged_case(len(counts), counts, starts)
    pool = np.full((256, 2, 16, 8, 64), POISON, dtype=np.uint16)
    want = pool.copy()
    assert oracle.kv_write_prefill(k, v, off, st, want, bt) == 0
    dpool = to_dev(pool, dev, bf=True)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding().kv_write_prefill(to_dev(k, dev, True), to_dev(v, dev, True), to_dev(off, dev),
                               to_dev(st, dev), dpool, to_dev(bt, dev), dev_err=err)
    got = synth.bits(dpool)
    mism = np.argwhere(got != want)
    assert mism.size == 0, f"{len(mism)} mismatching elements, first {mism[:3].tolist()}"
    assert int(err.item()) == 0


def test_prefill_full_size_sampled():
    """256 prompts x 2047 tokens into a 40000-page pool (1 GiB written)."""
    dev = cuda_or_skip()
    B, L = 256, 2047
    rng = np.random.default_rng(7)
    perm = rng.permutation(40000)
    bt = np.full((B, 128), -1, np.int32)
    bt[:, :128] = perm[:B * 128].reshape(B, 128)
    g = torch.Generator(device=dev).manual_seed(7)
    k = torch.randn((B * L, 8, 64), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((B * L, 8, 64), generator=g, device=dev).to(torch.bfloat16)
    off = torch.arange(0, B * L + 1, L, dtype=torch.int32, device=dev)
    st = torch.zeros(B, dtype=torch.int32, device=dev)
    pool = torch.full((40000, 2, 16, 8, 64), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding().kv_write_prefill(k, v, off, st, pool, to_dev(bt, dev), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in (0, 77, 255):
        kb = synth.bits(k[b * L:(b + 1) * L])
        vb = synth.bits(v[b * L:(b + 1) * L])
        hp = np.full((128, 2, 16, 8, 64), POISON, dtype=np.uint16)
        lbt = np.arange(128, dtype=np.int32)[None]
        assert oracle.kv_write_prefill(kb, vb, np.array([0, L], np.int32),
                                       np.array([0], np.int32), hp, lbt) == 0
        got = synth.bits(pool[torch.from_numpy(bt[b]).long().to(dev)])
        assert np.array_equal(got, hp), b


def test_prefill_then_decode_matches_oracle():
    dev = cuda_or_skip()
    lens = np.array([37, 16, 17, 1, 500], np.int32)     # lengths after the decode token
    prompt = lens - 1
    k, v, off, st, bt = ragged_case(3, list(prompt), [0] * len(lens), extents=list(lens))
    rng = np.random.default_rng(4)
    q = bf16_normal(rng, (len(lens), 32, 64))
    kn = bf16_normal(rng, (len(lens), 8, 64))
    vn = bf16_normal(rng, (len(lens), 8, 64))
    hp = np.full((256, 2, 16, 8, 64), POISON, dtype=np.uint16)
    assert oracle.kv_write_prefill(k, v, off, st, hp, bt) == 0
    assert oracle.kv_append(kn, vn, hp, bt, lens - 1) == 0
    ref = oracle.decode_attention(q, hp, bt, lens)

    b = binding()
    dpool = to_dev(np.full((256, 2, 16, 8, 64), POISON, dtype=np.uint16), dev, bf=True)
    dbt = to_dev(bt, dev)
    b.kv_write_prefill(to_dev(k, dev, True), to_dev(v, dev, True), to_dev(off, dev),
                       to_dev(st, dev), dpool, dbt)
    out = b.decode_step(to_dev(q, dev, True), to_dev(kn, dev, True), to_dev(vn, dev, True), dpool,
                        dbt, to_dev(lens, dev))
    assert_close(synth.bits(out), ref, "prefill + decode")
    assert np.array_equal(synth.bits(dpool), hp)


def test_prefill_reports_bad_offsets_and_pages():
    dev = cuda_or_skip()
    k, v, off, st, bt = ragged_case(5, [4, 4], [0, 0])
    b = binding()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    bad_off = np.array([2, 3, 5], np.int32)          # tokens 0 and 1 belong to no sequence
    dpool = to_dev(np.full((256, 2, 16, 8, 64), POISON, dtype=np.uint16), dev, bf=True)
    b.kv_write_prefill(to_dev(k[:5], dev, True), to_dev(v[:5], dev, True), to_dev(bad_off, dev),
                       to_dev(st, dev), dpool, to_dev(bt, dev), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & b.DEVERR_OFFSETS
    err.zero_()
    bt2 = bt.copy()
    bt2[1, 0] = 10 ** 6
    b.kv_write_prefill(to_dev(k, dev, True), to_dev(v, dev, True), to_dev(off, dev),
                       to_dev(st, dev), dpool, to_dev(bt2, dev), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & b.DEVERR_PAGE


@pytest.mark.parametrize("theta", [500000.0, 10000.0])
def test_prefill_special_values_bit_exact(theta):
    # positions 0..2739 (the last sequence runs past the 2048-entry cos/sin
    # table), values that send pairs down the FP64 redo path; NaN payload and
    # sign are not compared, every other bit is
    dev = cuda_or_skip()
    counts, starts = [700, 300, 700], [0, 1021, 2040]
    rng = np.random.default_rng(29)
    k0, v0, off, st, bt = ragged_case(31, counts, starts, num_pages=512, max_blocks=256)
    k = special_bf16(rng, k0.shape)
    v = special_bf16(rng, v0.shape)
    pool = np.full((512, 2, 16, 8, 64), 0x1234, dtype=np.uint16)   # a finite poison
    want = pool.copy()
    assert oracle.kv_write_prefill(k, v, off, st, want, bt, theta=theta) == 0
    dpool = to_dev(pool, dev, bf=True)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding().kv_write_prefill(to_dev(k, dev, True), to_dev(v, dev, True), to_dev(off, dev),
                               to_dev(st, dev), dpool, to_dev(bt, dev), rope_theta=theta,
                               dev_err=err)
    got = synth.bits(dpool)
    both_nan = is_nan_bf16(got) & is_nan_bf16(want)
    mism = np.argwhere((got != want) & ~both_nan)
    assert mism.size == 0, f"{len(mism)} mismatching elements, first {mism[:3].tolist()}"
    assert int(err.item()) == 0
    assert is_nan_bf16(want).any() and (want == 0).any()


def test_multi_layer_prefill_equals_per_layer_calls():
    # pkv_kv_write_prefill_layers: 3 layers of the same ragged prompts through
    # their own tables, in one call, write the bits the oracle writes
    dev = cuda_or_skip()
    counts, starts = [20, 0, 5, 300], [0, 3, 15, 100]
    layers = 3
    rng = np.random.default_rng(77)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(off[-1])
    ks = bf16_normal(rng, (layers, T, 8, 64))
    vs = bf16_normal(rng, (layers, T, 8, 64))
    bts = np.full((layers, len(counts), 128), -1, np.int32)
    perm = rng.permutation(512)
    cur = 0
    for layer in range(layers):
        for b, (c, s0) in enumerate(zip(counts, starts)):
            if c:
                first, last = s0 // 16, (s0 + c - 1) // 16
                bts[layer, b, first:last + 1] = perm[cur:cur + last - first + 1]
                cur += last - first + 1
    st = np.asarray(starts, np.int32)
    want = np.full((512, 2, 16, 8, 64), POISON, dtype=np.uint16)
    for layer in range(layers):
        assert oracle.kv_write_prefill(ks[layer], vs[layer], off, st, want, bts[layer]) == 0
    dpool = to_dev(np.full((512, 2, 16, 8, 64), POISON, dtype=np.uint16), dev, bf=True)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding().kv_write_prefill_layers(to_dev(ks, dev, True), to_dev(vs, dev, True),
                                      to_dev(off, dev), to_dev(st, dev), dpool, to_dev(bts, dev),
                                      dev_err=err)
    assert np.array_equal(synth.bits(dpool), want)
    assert int(err.item()) == 0
