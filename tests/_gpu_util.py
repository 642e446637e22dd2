"""Shared helpers of the GPU parity tests: run the decode step through the C-ABI
binding and compute the same step with the FP64 CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_04_gb300 import synth

# Output tolerance of the decode attention: |got - ref| <= 1e-3 + 8e-3 * |ref|.
TOL_ABS = 1e-3
TOL_REL = 8e-3


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch.device("cuda", 0)


def binding():
    from paged_kv_decode_04_gb300 import binding as b
    return b


def assert_close(got_bits, ref, what=""):
    got = oracle.bf16_to_f64(got_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {idx}: "
            f"got {got[idx]!r} ref {ref[idx]!r}")


def oracle_step(w, layer, seqs=None, threads=0):
    """Append (RoPE K, V) then attention for `seqs` of one layer, on a compact host copy."""
    c = synth.compact(w, layer, seqs)
    rc = oracle.kv_append(c.k_new, c.v_new, c.pool, c.block_table, c.positions,
                          page_size=w.page_size, theta=w.rope_theta)
    assert rc == 0
    out = oracle.decode_attention(c.q, c.pool, c.block_table, c.seq_lens,
                                  num_kv_heads=w.num_kv_heads, page_size=w.page_size,
                                  scale=w.scale, threads=threads)
    return out, c


def gpu_step(w, d, layer, *, num_splits=0, dev_err=None, out=None, workspace=None):
    """One decode step of one layer on the device tensors `d` (append, then attention)."""
    b = binding()
    bt = d["block_tables"][layer]
    b.kv_append(d["k_new"][layer], d["v_new"][layer], d["pool"], bt, d["positions"],
                rope_theta=w.rope_theta, dev_err=dev_err)
    return b.paged_decode_attention(d["q"][layer], d["pool"], bt, d["seq_lens"], out,
                                    scale=w.scale, workspace=workspace, num_splits=num_splits,
                                    dev_err=dev_err)


def appended_slots_expected(w, layer, seqs):
    """Oracle K and V rows (uint16 [n][Hkv][D]) that the append writes for `seqs`."""
    ks, vs = [], []
    for b in seqs:
        pos = int(w.positions[b])
        ks.append(np.stack([oracle.rope_rotate(w.k_new[layer, b, h], pos, w.rope_theta)
                            for h in range(w.num_kv_heads)]))
        vs.append(w.v_new[layer, b])
    return np.stack(ks), np.stack(vs)
