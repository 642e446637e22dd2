"""The host scheduler (include/pkv_sched.h) against its plain-Python oracle and
the admission rules' closed forms (CPU only).

Sources of the rules: "Hours of YouTube and 85 handtyped pages of notes on LLM
Inference - Start here", section "現在のスコープ" (page-credit admission, FIFO
wait, rejection, lazy pages, --stats) and the batching item of "これまでの進捗".
"""

import numpy as np
import pytest

from oracle.scheduler import REJECTED, OracleScheduler
from paged_kv_decode_04_gb300.scheduler import Scheduler

LAYERS = 16
CTX = 2048


@pytest.mark.parametrize("prompt,new,pages", [
    (10, 7, 1),        # 16 tokens processed at most -> one page
    (16, 1, 1),        # the only output token is never processed
    (16, 2, 2),        # 17 tokens -> two pages
    (1, 2048, 128),    # 2048 tokens fill the context exactly
    (2000, 500, 128),  # budget clamped to 49 new tokens: 2048 processed
    (2048, 10, 128),   # a full-context prompt leaves one new token
    (33, 64, 6),       # 96 tokens -> 6 pages
])
def test_budget_closed_form(prompt, new, pages):
    s = Scheduler(4096, LAYERS, CTX)
    assert s.budget_pages(prompt, new) == pages * LAYERS
    assert OracleScheduler(4096, LAYERS, CTX, 16, False).budget(prompt, new) == pages * LAYERS


@pytest.mark.parametrize("prompt,new", [(0, 5), (2049, 1), (5, 0)])
def test_budget_rejects_bad_sizes(prompt, new):
    s = Scheduler(4096, LAYERS, CTX)
    assert s.budget_pages(prompt, new) == -1
    with pytest.raises(ValueError):
        s.submit(prompt, new)


def test_small_pool_queues_the_request_that_does_not_fit():
    # 8 MiB pool of 32 KiB pages = 256 pages; three prompts of ~20 tokens with a
    # 64-token budget need 6 pages x 16 layers = 96 credits each: two fit.
    s = Scheduler(256, LAYERS, CTX)
    ids = [s.submit(20, 64) for _ in range(3)]
    assert s.admit() == 2
    st = s.stats()
    assert st["waiting"] == 1 and st["free_credits"] == 256 - 192
    s.finish(ids[0])
    assert s.admit() == 1            # credits came back at this scheduling point
    assert s.stats()["admission_wait_max"] == 1


def test_request_larger_than_pool_is_rejected():
    s = Scheduler(64, LAYERS, CTX)
    assert s.submit(100, 100) is None   # 13 pages x 16 layers > 64
    st = s.stats()
    assert st["rejected"] == 1 and st["waiting"] == 0


def test_fifo_head_blocks_later_requests():
    s = Scheduler(100, 1, CTX)
    a = s.submit(16 * 60, 1)      # 60 pages
    b = s.submit(16 * 50, 1)      # 50 pages: does not fit beside a
    c = s.submit(16, 1)           # 1 page: would fit, but must not overtake b
    assert s.admit() == 1
    assert s.stats()["waiting"] == 2
    s.finish(a)
    assert s.admit() == 2         # b and then c


def test_static_batching_waits_for_the_whole_group():
    s = Scheduler(1000, 1, CTX, static_batching=True)
    first = [s.submit(16, 3) for _ in range(2)]
    assert s.admit() == 2
    late = s.submit(16, 3)
    assert s.admit() == 0         # group still running
    s.finish(first[0])
    assert s.admit() == 0         # one member left
    s.finish(first[1])
    assert s.admit() == 1
    assert late == 2


def test_lazy_pages_follow_the_sequence_length():
    s = Scheduler(100, 2, CTX)
    rid = s.submit(15, 40)        # 54 tokens processed at most -> 4 pages per layer
    s.admit()
    got = s.next_prefill()
    assert got[0] == rid and got[1] == 15
    assert np.all(got[2][:, 0] >= 0) and np.all(got[2][:, 1:] == -1)
    assert s.stats()["free_pages"] == 100 - 2
    ids, lens, bt = s.decode_batch(8)      # appends position 15: still page 0
    assert lens.tolist() == [16] and np.all(bt[:, 0, 1] == -1)
    ids, lens, bt = s.decode_batch(8)      # appends position 16: a new page per layer
    assert lens.tolist() == [17] and np.all(bt[:, 0, 1] >= 0)
    assert s.stats()["free_pages"] == 100 - 4


def test_budget_is_exhausted_exactly():
    s = Scheduler(100, 1, CTX)
    rid = s.submit(10, 5)         # prefill + 4 decode batches
    s.admit()
    s.next_prefill()
    for k in range(4):
        ids, lens, _ = s.decode_batch(4)
        assert ids.tolist() == [rid] and lens.tolist() == [11 + k]
    assert s.decode_batch(4)[0].size == 0
    s.admit()
    assert s.stats()["free_pages"] == 100 and s.stats()["finished"] == 1


def run_trace(seed, static, num_pages=600, layers=2, steps=300):
    rng = np.random.default_rng(seed)
    cxx = Scheduler(num_pages, layers, CTX, static_batching=static)
    ref = OracleScheduler(num_pages, layers, CTX, 16, static)
    live = []
    for it in range(steps):
        for _ in range(rng.integers(0, 3)):
            p = int(rng.integers(1, 400))
            n = int(rng.integers(1, 300))
            a, b = cxx.submit(p, n), ref.submit(p, n)
            assert (a is None) == (b == REJECTED)
            if a is not None:
                assert a == b
                live.append(a)
        assert cxx.admit() == ref.admit()
        got = cxx.next_prefill()
        want = ref.next_prefill()
        assert (got is None) == (want is None)
        if got is not None:
            assert got[0] == want[0] and got[1] == want[1]
            assert np.array_equal(got[2], np.array(want[2]))
        mb = int(rng.integers(1, 16))
        ids, lens, bt = cxx.decode_batch(mb)
        w = ref.decode_batch(mb)
        assert ids.tolist() == [x[0] for x in w] and lens.tolist() == [x[1] for x in w]
        for i, x in enumerate(w):
            assert np.array_equal(bt[:, i], np.array(x[2]))
        # live block tables never share a page, and every live entry is a pool page
        used = bt[bt >= 0]
        assert len(np.unique(used)) == len(used)
        if ids.size:
            from paged_kv_decode_04_gb300 import binding
            for layer in range(bt.shape[0]):
                binding.check_tables(bt[layer], lens, num_pages)
        if live and rng.random() < 0.2:
            victim = int(rng.choice(live))
            assert cxx.finish(victim) == ref.finish(victim)
    # drain: everything admitted eventually finishes, no deadlock
    for _ in range(10000):
        cxx.admit()
        ref.admit()
        if cxx.next_prefill() is not None:
            ref.next_prefill()
        ids, _, _ = cxx.decode_batch(64)
        ref.decode_batch(64)
        st = cxx.stats()
        if st["waiting"] == 0 and st["active"] == 0:
            break
    cxx.admit()
    ref.admit()
    st = cxx.stats()
    assert st["waiting"] == 0 and st["active"] == 0
    assert st["free_pages"] == num_pages and st["free_credits"] == num_pages
    for k, v in ref.stats.items():
        assert st[k] == v, k
    return st


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("static", [False, True])
def test_matches_oracle_on_random_traces(seed, static):
    st = run_trace(seed, static)
    assert st["peak_allocated_pages"] <= 600
    # every accepted request ends finished (after admission, or cancelled while waiting)
    assert st["finished"] + st["rejected"] == st["submitted"]
    assert st["admitted"] <= st["finished"]


def test_running_count_and_decode_batch_into_match_decode_batch():
    # two schedulers fed the same trace: decode_batch_into (caller arrays sized
    # by running()) fills exactly what decode_batch returns
    rng = np.random.default_rng(21)
    reqs = [(int(rng.integers(1, 80)), int(rng.integers(1, 60))) for _ in range(12)]
    a, b = Scheduler(400, 3, CTX), Scheduler(400, 3, CTX)
    for p, n in reqs:
        a.submit(p, n)
        b.submit(p, n)
    for _ in range(200):
        a.admit()
        b.admit()
        ga, gb = a.next_prefill(), b.next_prefill()
        assert (ga is None) == (gb is None)
        n = min(5, b.running())
        ids_a, lens_a, bt_a = a.decode_batch(5)
        ids = np.empty(n, np.int64)
        lens = np.empty(n, np.int32)
        bt = np.empty((3, n, CTX // 16), np.int32)
        assert b.decode_batch_into(ids, lens, bt) == n == len(ids_a)
        assert np.array_equal(ids, ids_a) and np.array_equal(lens, lens_a)
        assert np.array_equal(bt, bt_a)
        if a.stats()["finished"] == len(reqs):
            break
    assert b.stats()["finished"] == len(reqs) and b.running() == 0


def test_decode_batch_into_rejects_bad_arrays():
    s = Scheduler(100, 2, CTX)
    with pytest.raises(ValueError):
        s.decode_batch_into(np.empty(2, np.int32), np.empty(2, np.int32),
                            np.empty((2, 2, CTX // 16), np.int32))
    with pytest.raises(ValueError):
        s.decode_batch_into(np.empty(2, np.int64), np.empty(2, np.int32),
                            np.empty((3, 2, CTX // 16), np.int32))
    assert s.decode_batch_into(np.empty(0, np.int64), np.empty(0, np.int32),
                               np.empty((2, 0, CTX // 16), np.int32)) == 0
