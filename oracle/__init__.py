"""FP64 CPU oracle for the paged-KV decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline arm
may import this package.  The product path (``paged_kv_decode_04_gb300``) never
imports it and shares no code with it.

The arithmetic lives in ``pkv_oracle.c`` (plain C, FP64, built by
``oracle/build.py``); this module only marshals numpy arrays into it.  bf16
tensors are passed as ``uint16`` arrays holding the raw bits.

What each function computes, and the readings taken where the source pages
are silent, are stated in the header of ``pkv_oracle.c``.  Sources: the
Tiny-vLLM README translation "Hours of YouTube and 85 handtyped pages of notes
on LLM Inference - Start here", section "これまでの進捗" (KV page pool item;
paged decode attention item).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

ORC_OK = 0
ORC_EINVAL = 1
ORC_ENOMEM = 2
ORC_EBADPAGE = 4
ORC_EBADLEN = 8
ORC_EBADPOS = 16

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_version.restype = ctypes.c_int
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_rope_inv_freq.argtypes = [ctypes.c_double, ctypes.c_int, _f64p]
        L.orc_rope_inv_freq.restype = None
        L.orc_rope_rotate_f64.argtypes = [_u16p, ctypes.c_int, ctypes.c_int32, ctypes.c_double, _f64p]
        L.orc_rope_rotate_f64.restype = None
        L.orc_rope_rotate.argtypes = [_u16p, ctypes.c_int, ctypes.c_int32, ctypes.c_double, _u16p]
        L.orc_rope_rotate.restype = None
        L.orc_kv_append.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, _i32p, ctypes.c_int,
                                    _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_double]
        L.orc_kv_append.restype = ctypes.c_int
        L.orc_kv_write_prefill.argtypes = [_u16p, _u16p, _i32p, _i32p, _u16p, ctypes.c_int64,
                                           _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_double]
        L.orc_kv_write_prefill.restype = ctypes.c_int
        L.orc_rope_queries.argtypes = [_u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double]
        L.orc_rope_queries.restype = None
        att = [_u16p, _u16p, ctypes.c_int64, _i32p, ctypes.c_int, _i32p, ctypes.c_int,
               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, _f64p,
               ctypes.c_int]
        L.orc_decode_attention.argtypes = att
        L.orc_decode_attention.restype = ctypes.c_int
        L.orc_decode_attention_online.argtypes = att
        L.orc_decode_attention_online.restype = ctypes.c_int
        L.orc_attention_partial.argtypes = [_u16p, _u16p, ctypes.c_int64, _i32p, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, _f64p, _f64p, _f64p]
        L.orc_attention_partial.restype = ctypes.c_int
        L.orc_merge_partials.argtypes = [ctypes.c_int, _f64p, _f64p, _f64p, ctypes.c_int, _f64p]
        L.orc_merge_partials.restype = None
        _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


# ------------------------------------------------------------------ bf16 --

def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16)
    f = (b.astype(np.uint32) << 16).view(np.float32)
    with np.errstate(invalid="ignore"):
        return f.astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round-to-nearest-even bf16 bits of float64 values (one rounding step)."""
    L = lib()
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, v in enumerate(flat):
        out[i] = L.orc_f64_to_bf16(float(v))
    return out.reshape(x.shape)


# ------------------------------------------------------------------ RoPE --

def rope_inv_freq(theta: float, head_dim: int) -> np.ndarray:
    out = np.empty(head_dim // 2, dtype=np.float64)
    lib().orc_rope_inv_freq(theta, head_dim, _ptr(out, ctypes.c_double))
    return out


def rope_rotate_f64(x_bits, pos: int, theta: float) -> np.ndarray:
    x = _u16(x_bits)
    y = np.empty(x.shape, dtype=np.float64)
    lib().orc_rope_rotate_f64(_ptr(x, ctypes.c_uint16), x.shape[-1], int(pos), theta,
                              _ptr(y, ctypes.c_double))
    return y


def rope_rotate(x_bits, pos: int, theta: float) -> np.ndarray:
    x = _u16(x_bits)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_rope_rotate(_ptr(x, ctypes.c_uint16), x.shape[-1], int(pos), theta,
                          _ptr(y, ctypes.c_uint16))
    return y


def rope_queries(q_bits, positions, theta: float) -> np.ndarray:
    q = _u16(q_bits)
    B, Hq, D = q.shape
    pos = _i32(positions)
    out = np.empty_like(q)
    lib().orc_rope_queries(_ptr(q, ctypes.c_uint16), _ptr(out, ctypes.c_uint16),
                           _ptr(pos, ctypes.c_int32), B, Hq, D, theta)
    return out


# ---------------------------------------------------------------- append --

def kv_append(k_new, v_new, pool, block_table, positions, *, page_size: int = 16,
              theta: float = 500000.0) -> int:
    """Write RoPE(k_new) and v_new into ``pool`` (modified in place).

    pool: uint16 array [num_pages][2][page_size][Hkv][D];
    block_table: int32 [B][max_blocks]; positions: int32 [B].
    Returns the oracle's status bit set (0 = every entry written).
    """
    k = _u16(k_new)
    v = _u16(v_new)
    assert pool.dtype == np.uint16 and pool.flags["C_CONTIGUOUS"]
    bt = _i32(block_table)
    pos = _i32(positions)
    B, Hkv, D = k.shape
    num_pages = pool.shape[0]
    return lib().orc_kv_append(_ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                               _ptr(pool, ctypes.c_uint16), num_pages,
                               _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(pos, ctypes.c_int32),
                               B, Hkv, D, page_size, theta)


def kv_write_prefill(k, v, token_offsets, start_positions, pool, block_table, *,
                     page_size: int = 16, theta: float = 500000.0) -> int:
    """Write every sequence's new tokens (ragged, [num_tokens][Hkv][D]) into ``pool``."""
    ka = _u16(k)
    va = _u16(v)
    assert pool.dtype == np.uint16 and pool.flags["C_CONTIGUOUS"]
    off = _i32(token_offsets)
    st = _i32(start_positions)
    bt = _i32(block_table)
    B = st.shape[0]
    return lib().orc_kv_write_prefill(_ptr(ka, ctypes.c_uint16), _ptr(va, ctypes.c_uint16),
                                      _ptr(off, ctypes.c_int32), _ptr(st, ctypes.c_int32),
                                      _ptr(pool, ctypes.c_uint16), pool.shape[0],
                                      _ptr(bt, ctypes.c_int32), bt.shape[1], B, ka.shape[1],
                                      ka.shape[2], page_size, theta)


# ------------------------------------------------------------- attention --

def _attention(fn, q, pool, block_table, seq_lens, *, num_kv_heads, page_size, scale,
               threads):
    qa = _u16(q)
    B, Hq, D = qa.shape
    pl = _u16(pool)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = fn(_ptr(qa, ctypes.c_uint16), _ptr(pl, ctypes.c_uint16), pl.shape[0],
            _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32), B, Hq,
            num_kv_heads, D, page_size, scale, _ptr(out, ctypes.c_double),
            threads if threads else default_threads())
    return out, rc


def decode_attention(q, pool, block_table, seq_lens, *, num_kv_heads: int = 8,
                     page_size: int = 16, scale: float = 0.125, threads: int = 0,
                     return_status: bool = False):
    """Two-pass FP64 paged decode attention; returns float64 [B][Hq][D]."""
    out, rc = _attention(lib().orc_decode_attention, q, pool, block_table, seq_lens,
                         num_kv_heads=num_kv_heads, page_size=page_size, scale=scale,
                         threads=threads)
    return (out, rc) if return_status else out


def decode_attention_online(q, pool, block_table, seq_lens, *, num_kv_heads: int = 8,
                            page_size: int = 16, scale: float = 0.125, threads: int = 0,
                            return_status: bool = False):
    """One-pass (online softmax) FP64 variant of :func:`decode_attention`."""
    out, rc = _attention(lib().orc_decode_attention_online, q, pool, block_table, seq_lens,
                         num_kv_heads=num_kv_heads, page_size=page_size, scale=scale,
                         threads=threads)
    return (out, rc) if return_status else out


def attention_partial(q, pool, block_table, b: int, j: int, t_begin: int, t_end: int, *,
                      num_kv_heads: int = 8, page_size: int = 16, scale: float = 0.125):
    """(m, l, acc) of one (b, j) over tokens [t_begin, t_end)."""
    qa = _u16(q)
    B, Hq, D = qa.shape
    pl = _u16(pool)
    bt = _i32(block_table)
    m = np.zeros(1, dtype=np.float64)
    l = np.zeros(1, dtype=np.float64)
    acc = np.zeros(D, dtype=np.float64)
    rc = lib().orc_attention_partial(_ptr(qa, ctypes.c_uint16), _ptr(pl, ctypes.c_uint16),
                                     pl.shape[0], _ptr(bt, ctypes.c_int32), bt.shape[1], Hq,
                                     num_kv_heads, D, page_size, scale, b, j, t_begin, t_end,
                                     _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double),
                                     _ptr(acc, ctypes.c_double))
    if rc:
        raise RuntimeError(f"oracle partial failed: status {rc}")
    return float(m[0]), float(l[0]), acc


def merge_partials(m, l, acc) -> np.ndarray:
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    S, D = acc.shape
    out = np.zeros(D, dtype=np.float64)
    lib().orc_merge_partials(S, _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double),
                             _ptr(acc, ctypes.c_double), D, _ptr(out, ctypes.c_double))
    return out
