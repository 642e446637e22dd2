"""The benchmark's byte accounting (CPU only), against closed forms.

A decode step must read every live token's K and V rows once per kv head
(2 KiB a token for 8 heads x 64 dims x K and V in bf16), q and write out
(8 KiB a sequence), read the live table entries and the lengths, and read
and write the appended token's rows.  With shared prompt prefixes, DRAM
must deliver each physical page once per step.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_decode_04_gb300 import synth  # noqa: E402

KV_PER_TOKEN = 8 * 64 * 2 * 2        # K and V rows of 8 heads, bf16


def per_sequence(L):
    """Bytes one sequence of L tokens (after the append) needs in one layer."""
    pages = -(-L // 16)
    return (L * KV_PER_TOKEN          # its K/V
            + 32 * 64 * 2 * 2         # q read, out written
            + 4 * pages + 4           # live table entries, seq_lens
            + 8 * 64 * 2 * 2 * 2      # new K/V read, then written to the pool
            + 4)                      # position


def test_peak_step_bytes():
    w = synth.make_workload("peak", 0)
    assert per_sequence(2048) == 4_207_112
    assert bench.algorithmic_bytes(w) == 256 * 4_207_112 == 1_077_020_672
    # nothing is shared: every page is attended by one sequence
    assert bench.unique_bytes(w) == bench.algorithmic_bytes(w)


def test_prefix_step_counts_each_shared_page_once():
    w = synth.make_workload("prefix", 0)
    assert bench.algorithmic_bytes(w) == 1_077_020_672          # the same 256 x 2048 tokens
    # 16 groups of 16 share 96 full pages (1536 tokens); each sequence owns 512
    groups, members, shared_tokens, own_tokens = 16, 16, 96 * 16, 2048 - 96 * 16
    kv_unique = (groups * shared_tokens + groups * members * own_tokens) * KV_PER_TOKEN
    non_kv = 1_077_020_672 - 256 * 2048 * KV_PER_TOKEN
    assert bench.unique_bytes(w) == kv_unique + non_kv == 322_045_952


def test_mixed_batch_bytes_follow_the_lengths():
    w = synth.make_workload("mix", 0)
    want = w.layers * sum(per_sequence(int(L)) for L in w.seq_lens)
    assert bench.algorithmic_bytes(w) == want
    # attention and append parts add up to the step
    assert (bench.algorithmic_bytes(w, "attention") + bench.algorithmic_bytes(w, "append")
            == want)
    assert np.all(w.seq_lens >= 16) and w.layers == 16
