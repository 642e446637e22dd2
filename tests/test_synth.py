"""The seeded workload generator draws what the workload recipes say (CPU only)."""
import numpy as np

from paged_kv_decode_04_gb300 import synth


def _check_structure(w):
    assert w.block_tables.shape == (w.layers, w.batch, w.max_blocks)
    # every live page is used exactly once, all ids are in the pool
    live = w.block_tables[w.block_tables >= 0]
    assert len(np.unique(live)) == len(live) == len(w.live_pages)
    assert live.min() >= 0 and live.max() < w.num_pages
    for layer in range(w.layers):
        for b in range(w.batch):
            n = -(-int(w.seq_lens[b]) // w.page_size)
            assert np.all(w.block_tables[layer, b, :n] >= 0)
            assert np.all(w.block_tables[layer, b, n:] == -1)
    assert np.array_equal(w.positions, w.seq_lens - 1)


def test_tiny_and_small_shapes():
    w = synth.make_workload("tiny", 0)
    assert w.batch == 1 and w.seq_lens.tolist() == [37] and w.num_pages == 64
    assert w.page_data.shape == (3, 2, 16, 8, 64)
    _check_structure(w)
    # the last page holds 5 tokens: slots 0..3 live, slot 4 (the appended position) onward poison
    last = w.page_data[2]
    assert np.all(last[:, 4:] == synth.POISON)
    assert not np.any(last[:, :4] == synth.POISON)
    s = synth.make_workload("small", 0)
    assert s.batch == 8 and s.seq_lens.min() >= 1 and s.seq_lens.max() <= 2048
    _check_structure(s)


def test_mix_length_recipe():
    w = synth.make_workload("mix", 3, layers=2, num_pages=8192)
    short = (w.seq_lens >= 16) & (w.seq_lens <= 128)
    long_ = (w.seq_lens >= 1536) & (w.seq_lens <= 2048)
    assert short.sum() == 115 and long_.sum() == 13
    _check_structure(w)


def test_seeded_and_reproducible():
    a = synth.make_workload("small", 5)
    b = synth.make_workload("small", 5)
    c = synth.make_workload("small", 6)
    assert np.array_equal(a.page_data, b.page_data) and np.array_equal(a.q, b.q)
    assert not np.array_equal(a.seq_lens, c.seq_lens)


def test_values_are_standard_normal_bf16():
    w = synth.make_workload("long", 1, layers=1)
    vals = (w.page_data[:, :, :].astype(np.uint32) << 16).view(np.float32)
    vals = vals[np.isfinite(vals)]
    assert abs(vals.mean()) < 0.01 and abs(vals.std() - 1.0) < 0.01


def test_compact_is_a_relabelling():
    w = synth.make_workload("small", 2)
    c = synth.compact(w, 0, [1, 5])
    pool = synth.host_pool(w)
    for r, b in enumerate([1, 5]):
        n = -(-int(w.seq_lens[b]) // 16)
        assert np.array_equal(c.pool[c.block_table[r, :n]], pool[w.block_tables[0, b, :n]])


def test_prefix_workload_aliases_group_prefixes():
    w = synth.make_workload("prefix", 0, batch=32, num_pages=4096)
    bt = w.block_tables[0]
    G, S = synth.PREFIX_GROUP, synth.PREFIX_BLOCKS
    for b in range(32):
        lead = b - b % G
        assert np.array_equal(bt[b, :S], bt[lead, :S])
    assert not np.any(np.isin(bt[0, :S], bt[G, :S]))          # groups do not share
    private = bt[:, S:][bt[:, S:] >= 0]
    assert len(np.unique(private)) == len(private)              # tails are private
    assert len(np.unique(bt[bt >= 0])) == len(w.live_pages)
    # shared pages hold no poison; each private last page holds poison from slot 15 on
    pool = synth.host_pool(w)
    assert not np.any(pool[bt[0, :S]] == synth.POISON)
    assert np.all(pool[bt[:, 127], :, 15:] == synth.POISON)
