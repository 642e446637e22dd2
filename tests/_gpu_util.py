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


def bf16_normal(rng, shape):
    """N(0, 1) drawn in FP32 and rounded to bf16 bit patterns."""
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def special_bf16(rng, shape):
    """bf16 bit patterns mixing normal values with zeros, subnormals, tiny and
    huge normals, infinities, NaNs and exact x1 == x2 pairs (cancellation) along
    the last axis of 64 dims."""
    x = bf16_normal(rng, shape)
    kind = rng.integers(0, 10, size=shape)
    sign = (rng.integers(0, 2, size=shape) << 15).astype(np.uint16)
    mant = rng.integers(0, 128, size=shape).astype(np.uint16)
    x = np.where(kind == 1, sign, x)                                            # +-0
    x = np.where(kind == 2, sign | np.maximum(mant, 1), x)                      # subnormal
    tiny = (rng.integers(1, 31, size=shape).astype(np.uint16) << 7) | mant
    x = np.where(kind == 3, sign | tiny, x)                                     # tiny normal
    huge = (rng.integers(220, 255, size=shape).astype(np.uint16) << 7) | mant
    x = np.where(kind == 4, sign | huge, x)                                     # huge normal
    x = np.where((kind == 5) & (mant < 16), sign | 0x7F80, x)                   # +-inf
    x = np.where((kind == 5) & (mant >= 120), 0x7FC1 | sign, x)                 # NaN
    x = x.astype(np.uint16)
    pair = kind[..., :32] == 6                                                  # x2 := x1
    x[..., 32:] = np.where(pair, x[..., :32], x[..., 32:])
    return x


def is_nan_bf16(x):
    return ((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0)


def equal_but_nan_payload(got, want):
    """Bit equality, except that any two NaNs are equal (payload and sign free)."""
    return (got == want) | (is_nan_bf16(got) & is_nan_bf16(want))
