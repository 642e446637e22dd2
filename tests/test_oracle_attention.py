"""Pins for the oracle's paged decode attention and KV append (CPU only).

What is pinned, and by what (none of these re-type the oracle's own loops):
  * brute force: gather each sequence's K/V with numpy fancy indexing on the
    5-D pool and use scipy's softmax on the contiguous copy;
  * closed forms: identical keys give the mean of V, a dominant key gives its
    V, one token gives V_0, zero tokens give 0, two tokens give a logistic
    weight;
  * invariants: permuting physical pages with a remapped table, the online
    recurrence vs the two-pass form, split partials merged vs the whole;
  * structure: the GQA head map, poison never read, the append touching only
    its slot;
  * aliasing: sequences whose tables share prefix pages equal the same batch
    with private copies, and an append never writes the shared pages.
Source of the computation: "Hours of YouTube and 85 handtyped pages of notes on
LLM Inference - Start here", section "これまでの進捗" (paged decode attention
item; KV page pool item).
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle

HQ, HKV, D, P = 32, 8, 64, 16
THETA = 500000.0
SCALE = 0.125
POISON = 0xFFFF


def bf16(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def make_case(seed, lens, num_pages=64, max_blocks=8, hq=HQ, hkv=HKV):
    """Random K/V in randomly chosen pages, poison elsewhere."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    pool = np.full((num_pages, 2, P, hkv, D), POISON, dtype=np.uint16)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    perm = rng.permutation(num_pages)
    cur = 0
    for b, L in enumerate(lens):
        n = -(-L // P)
        bt[b, :n] = perm[cur:cur + n]
        cur += n
        for k in range(n):
            valid = min(P, L - k * P)
            pool[bt[b, k], :, :valid] = bf16(rng.standard_normal((2, valid, hkv, D)))
    q = bf16(rng.standard_normal((B, hq, D)))
    return q, pool, bt, np.asarray(lens, dtype=np.int32)


def brute_force(q, pool, bt, lens, hq=HQ, hkv=HKV, scale=SCALE):
    B = q.shape[0]
    out = np.zeros((B, hq, D))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        pages = bt[b, t // P]
        slots = t % P
        for j in range(hq):
            g = j // (hq // hkv)
            K = oracle.bf16_to_f64(pool[pages, 0, slots, g, :])   # [L, D]
            V = oracle.bf16_to_f64(pool[pages, 1, slots, g, :])
            w = scipy.special.softmax(scale * (K @ oracle.bf16_to_f64(q[b, j])))
            out[b, j] = w @ V
    return out


@pytest.mark.parametrize("seed,lens", [(0, [1]), (1, [37]), (2, [16, 17]), (3, [40, 5]),
                                       (4, [33, 0, 12])])
def test_matches_brute_force(seed, lens):
    q, pool, bt, L = make_case(seed, lens)
    got, rc = oracle.decode_attention(q, pool, bt, L, return_status=True)
    assert rc == 0
    want = brute_force(q, pool, bt, L)
    assert np.all(np.isfinite(got))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14)


def test_identical_keys_give_mean_of_values():
    q, pool, bt, L = make_case(5, [29])
    # copy token 0's key into every other token of the sequence
    for t in range(1, 29):
        pool[bt[0, t // P], 0, t % P] = pool[bt[0, 0], 0, 0]
    got = oracle.decode_attention(q, pool, bt, L)
    t = np.arange(29)
    for j in range(HQ):
        V = oracle.bf16_to_f64(pool[bt[0, t // P], 1, t % P, j // 4, :])
        assert np.allclose(got[0, j], V.mean(axis=0), rtol=1e-12, atol=1e-14)


def test_dominant_key_selects_its_value():
    q, pool, bt, L = make_case(6, [40])
    # q = e_0 * 8 for head 0; key t* has k_0 = 40 (score +40), every other key 0
    q[0, 0] = bf16(np.eye(D)[0] * 8.0)
    tstar = 23
    for t in range(40):
        pool[bt[0, t // P], 0, t % P, 0] = bf16(np.zeros(D))
    pool[bt[0, tstar // P], 0, tstar % P, 0, 0] = bf16([40.0])[0]
    got = oracle.decode_attention(q, pool, bt, L)
    v_star = oracle.bf16_to_f64(pool[bt[0, tstar // P], 1, tstar % P, 0])
    assert np.allclose(got[0, 0], v_star, rtol=0, atol=1e-15 * 40 * 8)


def test_single_token_is_v0_and_empty_is_zero():
    q, pool, bt, L = make_case(7, [1, 0])
    got = oracle.decode_attention(q, pool, bt, L)
    for j in range(HQ):
        assert np.array_equal(got[0, j], oracle.bf16_to_f64(pool[bt[0, 0], 1, 0, j // 4]))
    assert np.array_equal(got[1], np.zeros((HQ, D)))


def test_two_tokens_logistic_weight():
    q, pool, bt, L = make_case(8, [2])
    q[0, 5] = bf16(np.eye(D)[3] * 2.0)             # head 5 -> kv head 1
    pool[bt[0, 0], 0, 0, 1] = bf16(np.eye(D)[3] * 3.0)  # score s0 = 0.125 * 6 = 0.75
    pool[bt[0, 0], 0, 1, 1] = bf16(np.zeros(D))         # score s1 = 0
    got = oracle.decode_attention(q, pool, bt, L)
    w0 = 1.0 / (1.0 + math.exp(-0.75))
    v0 = oracle.bf16_to_f64(pool[bt[0, 0], 1, 0, 1])
    v1 = oracle.bf16_to_f64(pool[bt[0, 0], 1, 1, 1])
    assert np.allclose(got[0, 5], w0 * v0 + (1 - w0) * v1, rtol=1e-13, atol=1e-15)


def test_gqa_head_map_consecutive_heads_share_a_kv_head():
    q, pool, bt, L = make_case(9, [19])
    for g in range(HKV):                 # V of kv head g is the constant g + 1 for every token
        for t in range(19):
            pool[bt[0, t // P], 1, t % P, g] = bf16(np.full(D, g + 1.0))
    got = oracle.decode_attention(q, pool, bt, L)
    for j in range(HQ):
        assert np.allclose(got[0, j], j // 4 + 1.0, rtol=1e-13)


def test_page_permutation_is_invisible():
    q, pool, bt, L = make_case(10, [45, 31, 7], num_pages=40)
    base = oracle.decode_attention(q, pool, bt, L)
    perm = np.random.default_rng(99).permutation(pool.shape[0])   # new id of physical page p
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    assert np.array_equal(oracle.decode_attention(q, pool2, bt2, L), base)


def test_online_equals_two_pass():
    q, pool, bt, L = make_case(11, [128, 77, 1, 16], num_pages=64, max_blocks=8)
    a = oracle.decode_attention(q, pool, bt, L)
    b = oracle.decode_attention_online(q, pool, bt, L)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("cuts", [[0, 50, 100], [0, 16, 32, 48, 64, 100], [0, 0, 7, 100, 100],
                                  [0, 100]])
def test_merged_partials_equal_whole(cuts):
    q, pool, bt, L = make_case(12, [100], num_pages=16, max_blocks=8)
    whole = oracle.decode_attention(q, pool, bt, L)
    for j in (0, 13, 31):
        parts = [oracle.attention_partial(q, pool, bt, 0, j, a, b)
                 for a, b in zip(cuts[:-1], cuts[1:])]
        m = [p[0] for p in parts]
        l = [p[1] for p in parts]
        acc = np.stack([p[2] for p in parts])
        assert np.allclose(oracle.merge_partials(m, l, acc), whole[0, j], rtol=1e-12, atol=1e-15)


def test_poison_is_never_read():
    # make_case fills every non-live slot with NaN; a stray read would make NaN.
    q, pool, bt, L = make_case(13, [3, 18, 31, 32, 33], num_pages=64)
    got = oracle.decode_attention(q, pool, bt, L)
    assert np.all(np.isfinite(got))


def test_thread_count_does_not_change_results():
    q, pool, bt, L = make_case(14, [60, 5, 33], num_pages=32)
    a = oracle.decode_attention(q, pool, bt, L, threads=1)
    b = oracle.decode_attention(q, pool, bt, L, threads=7)
    assert np.array_equal(a, b)


def test_bad_page_and_length_are_reported():
    q, pool, bt, L = make_case(15, [20], num_pages=8)
    bt_bad = bt.copy(); bt_bad[0, 1] = 8
    _, rc = oracle.decode_attention(q, pool, bt_bad, L, return_status=True)
    assert rc & oracle.ORC_EBADPAGE
    _, rc = oracle.decode_attention(q, pool, bt, np.array([8 * 16 + 1], np.int32),
                                    return_status=True)
    assert rc & oracle.ORC_EBADLEN


# ------------------------------------------------------------------ append --

def test_append_writes_exactly_one_slot_per_sequence():
    rng = np.random.default_rng(20)
    q, pool, bt, L = make_case(20, [37, 16, 1], num_pages=32)
    pos = (L - 1).astype(np.int32)
    k_new = bf16(rng.standard_normal((3, HKV, D)))
    v_new = bf16(rng.standard_normal((3, HKV, D)))
    before = pool.copy()
    assert oracle.kv_append(k_new, v_new, pool, bt, pos) == 0
    expect = before.copy()
    for b in range(3):
        page, slot = bt[b, pos[b] // P], pos[b] % P
        for h in range(HKV):
            expect[page, 0, slot, h] = oracle.rope_rotate(k_new[b, h], int(pos[b]), THETA)
            expect[page, 1, slot, h] = v_new[b, h]
    assert np.array_equal(pool, expect)
    # sequence 2 was appended at position 0: RoPE is the identity there
    assert np.array_equal(pool[bt[2, 0], 0, 0], k_new[2])


def test_append_then_attend_one_token_returns_new_value():
    rng = np.random.default_rng(21)
    pool = np.full((4, 2, P, HKV, D), POISON, dtype=np.uint16)
    bt = np.array([[2, -1]], dtype=np.int32)
    k_new = bf16(rng.standard_normal((1, HKV, D)))
    v_new = bf16(rng.standard_normal((1, HKV, D)))
    q = bf16(rng.standard_normal((1, HQ, D)))
    oracle.kv_append(k_new, v_new, pool, bt, np.array([0], np.int32))
    got = oracle.decode_attention(q, pool, bt, np.array([1], np.int32))
    for j in range(HQ):
        assert np.array_equal(got[0, j], oracle.bf16_to_f64(v_new[0, j // 4]))


def test_append_bad_position_or_page_is_skipped():
    rng = np.random.default_rng(22)
    pool = np.full((4, 2, P, HKV, D), POISON, dtype=np.uint16)
    bt = np.array([[1, 9], [3, -1]], dtype=np.int32)
    k = bf16(rng.standard_normal((2, HKV, D)))
    before = pool.copy()
    rc = oracle.kv_append(k, k, pool, bt, np.array([17, 2 * P], np.int32))
    assert rc & oracle.ORC_EBADPAGE and rc & oracle.ORC_EBADPOS
    assert np.array_equal(pool, before)


def test_query_rotation_matches_single_vector_rotation():
    rng = np.random.default_rng(23)
    q = bf16(rng.standard_normal((2, HQ, D)))
    pos = np.array([5, 1999], np.int32)
    out = oracle.rope_queries(q, pos, THETA)
    for b in range(2):
        for j in (0, 17, 31):
            assert np.array_equal(out[b, j], oracle.rope_rotate(q[b, j], int(pos[b]), THETA))


# ----------------------------------------------------------------- prefill --

def _complex_rope_bits(x_bits, pos, theta=THETA):
    """RoPE through complex multiplication (independent of the oracle's loop),
    rounded once to bf16 with the separately pinned converter."""
    xv = oracle.bf16_to_f64(x_bits)
    z = (xv[:32] + 1j * xv[32:]) * np.exp(1j * pos * np.power(theta, -np.arange(32) / 32.0))
    return oracle.f64_to_bf16(np.concatenate([z.real, z.imag]))


def test_prefill_writes_rotated_tokens_at_consecutive_positions():
    rng = np.random.default_rng(30)
    starts = np.array([0, 5, 30, 0], np.int32)
    counts = np.array([20, 11, 3, 0], np.int32)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(off[-1])
    k = bf16(rng.standard_normal((T, HKV, D)))
    v = bf16(rng.standard_normal((T, HKV, D)))
    pool = np.full((16, 2, P, HKV, D), POISON, dtype=np.uint16)
    bt = np.full((4, 8), -1, np.int32)
    bt[0, :2] = [3, 7]
    bt[1, :1] = [9]
    bt[2, :3] = [1, 2, 11]
    before = pool.copy()
    assert oracle.kv_write_prefill(k, v, off, starts, pool, bt) == 0
    expect = before.copy()
    for b in range(4):
        for i in range(counts[b]):
            t = off[b] + i
            pos = starts[b] + i
            page, slot = bt[b, pos // P], pos % P
            for h in range(HKV):
                expect[page, 0, slot, h] = _complex_rope_bits(k[t, h], pos)
            expect[page, 1, slot] = v[t]
    assert np.array_equal(pool, expect)


def test_prefill_then_attention_equals_brute_force_on_rotated_keys():
    rng = np.random.default_rng(31)
    L = 37
    k = bf16(rng.standard_normal((L, HKV, D)))
    v = bf16(rng.standard_normal((L, HKV, D)))
    q = bf16(rng.standard_normal((1, HQ, D)))
    pool = np.full((8, 2, P, HKV, D), POISON, dtype=np.uint16)
    bt = np.array([[4, 0, 6, -1]], np.int32)
    assert oracle.kv_write_prefill(k, v, np.array([0, L], np.int32), np.array([0], np.int32),
                                   pool, bt) == 0
    got = oracle.decode_attention(q, pool, bt, np.array([L], np.int32))
    for j in (0, 9, 31):
        g = j // 4
        K = np.stack([oracle.bf16_to_f64(_complex_rope_bits(k[t, g], t)) for t in range(L)])
        V = oracle.bf16_to_f64(v[:, g])
        w = scipy.special.softmax(SCALE * (K @ oracle.bf16_to_f64(q[0, j])))
        assert np.allclose(got[0, j], w @ V, rtol=1e-12, atol=1e-14)


def test_prefill_bad_positions_are_skipped():
    rng = np.random.default_rng(32)
    k = bf16(rng.standard_normal((3, HKV, D)))
    pool = np.full((4, 2, P, HKV, D), POISON, dtype=np.uint16)
    bt = np.array([[1, -1]], np.int32)          # block 1 is unmapped
    before = pool.copy()
    rc = oracle.kv_write_prefill(k, k, np.array([0, 3], np.int32), np.array([15], np.int32),
                                 pool, bt)
    assert rc & oracle.ORC_EBADPAGE
    # position 15 was written, 16 and 17 (block 1) were not
    assert not np.array_equal(pool[1, :, 15], before[1, :, 15])
    changed = np.argwhere(np.any(pool != before, axis=(3, 4)))
    assert {tuple(c) for c in changed.tolist()} == {(1, 0, 15), (1, 1, 15)}


def aliased_prefix_case(seed, group=3, shared_pages=2, own=(5, 20, 33)):
    """`group` sequences whose tables name the same `shared_pages` physical
    pages first (a common prompt prefix), then pages of their own."""
    rng = np.random.default_rng(seed)
    num_pages = shared_pages + sum(-(-o // P) for o in own) + 4
    pool = np.full((num_pages, 2, P, HKV, D), POISON, dtype=np.uint16)
    perm = rng.permutation(num_pages)
    shared = perm[:shared_pages]
    pool[shared] = bf16(rng.standard_normal((shared_pages, 2, P, HKV, D)))
    bt = np.full((group, 8), -1, dtype=np.int32)
    cur = shared_pages
    lens = []
    for b in range(group):
        n_own = -(-own[b] // P)
        bt[b, :shared_pages] = shared
        bt[b, shared_pages:shared_pages + n_own] = perm[cur:cur + n_own]
        for k in range(n_own):
            valid = min(P, own[b] - k * P)
            pool[perm[cur + k], :, :valid] = bf16(rng.standard_normal((2, valid, HKV, D)))
        cur += n_own
        lens.append(shared_pages * P + own[b])
    q = bf16(rng.standard_normal((group, HQ, D)))
    return q, pool, bt, np.asarray(lens, dtype=np.int32), shared


def test_aliased_prefix_equals_private_copies():
    # prefix sharing is pure aliasing: copying the shared pages out to private
    # pages for every follower changes no output bit, and both agree with the
    # brute-force gather
    q, pool, bt, L, shared = aliased_prefix_case(21)
    base = oracle.decode_attention(q, pool, bt, L)
    S = len(shared)
    pool2 = np.concatenate([pool, np.empty((S * (len(L) - 1),) + pool.shape[1:], pool.dtype)])
    bt2 = bt.copy()
    nxt = pool.shape[0]
    for b in range(1, len(L)):
        for k in range(S):
            pool2[nxt] = pool[shared[k]]
            bt2[b, k] = nxt
            nxt += 1
    assert np.array_equal(oracle.decode_attention(q, pool2, bt2, L), base)
    np.testing.assert_allclose(base, brute_force(q, pool, bt, L), rtol=1e-12, atol=1e-12)


def test_append_to_an_aliased_batch_leaves_the_shared_pages():
    q, pool, bt, L, shared = aliased_prefix_case(22)
    rng = np.random.default_rng(23)
    kn = bf16(rng.standard_normal((len(L), HKV, D)))
    vn = bf16(rng.standard_normal((len(L), HKV, D)))
    before = pool[shared].copy()
    assert oracle.kv_append(kn, vn, pool, bt, L - 1) == 0
    assert np.array_equal(pool[shared], before)
