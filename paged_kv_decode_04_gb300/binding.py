"""Thin ctypes binding of libpkv.so (include/pkv.h).

Argument marshalling only: tensors are checked for dtype, shape, device and
contiguity, then their device pointers go to the C entry points with the
current CUDA stream.  Every step of the decode path runs in the library's
kernels; there is no Python or CPU fallback -- importing this module without
the built library raises ImportError, and a failing call raises PkvError.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_EINVAL = 1
PKV_EUNSUPPORTED = 2
PKV_EWORKSPACE = 3
PKV_ECUDA = 4
PKV_EALIGN = 5

DEVERR_PAGE = 1
DEVERR_SEQLEN = 2
DEVERR_POSITION = 4
DEVERR_TIMEOUT = 8
DEVERR_OFFSETS = 16
DEVERR_PLAN = 32
PLAN_MAGIC = 0x32564B50
PLAN_HEADER_WORDS = 12

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
PAGE_SIZE = 16


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)} (status {status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libpkv.so not found at {LIB_PATH}; build it with "
            "`python -m paged_kv_decode_04_gb300.build` (needs nvcc for sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                  ctypes.c_float, ctypes.c_double, ctypes.c_size_t)
    L.pkv_abi_version.argtypes = []
    L.pkv_abi_version.restype = i32
    L.pkv_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    L.pkv_set_wait_limit_ns.restype = ctypes.c_ulonglong
    L.pkv_strerror.argtypes = [i32]
    L.pkv_strerror.restype = ctypes.c_char_p
    L.pkv_plan_splits.argtypes = [i32, i32, i32, i32]
    L.pkv_plan_splits.restype = i32
    L.pkv_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.pkv_workspace_bytes.restype = sz
    L.pkv_kv_append.argtypes = [vp, vp, vp, i64, vp, i32, vp, i32, i32, i32, i32, f64, vp, vp,
                                i32, vp, vp]
    L.pkv_kv_append.restype = i32
    L.pkv_paged_decode_attention.argtypes = [vp, vp, i64, vp, i32, vp, i32, i32, i32, i32, i32,
                                             f32, vp, vp, sz, i32, vp, vp]
    L.pkv_paged_decode_attention.restype = i32
    L.pkv_decode_step.argtypes = [vp, vp, vp, vp, i64, vp, i32, vp, i32, i32, i32, i32, i32, f64,
                                  f32, vp, vp, sz, i32, vp, vp]
    L.pkv_decode_step.restype = i32
    L.pkv_kv_write_prefill.argtypes = [vp, vp, i32, vp, vp, vp, i64, vp, i32, i32, i32, i32, i32,
                                       f64, vp, vp]
    L.pkv_kv_write_prefill.restype = i32
    L.pkv_attention_kernels.argtypes = [i32, i32, i32, vp]
    L.pkv_attention_kernels.restype = ctypes.c_char_p
    L.pkv_check_tables.argtypes = [vp, i32, vp, i32, i64, i32, vp, vp]
    L.pkv_check_tables.restype = i32
    L.pkv_plan_bytes.argtypes = [i32, i32]
    L.pkv_plan_bytes.restype = sz
    L.pkv_plan_build.argtypes = [vp, i32, i32, i32, vp, sz]
    L.pkv_plan_build.restype = i32
    L.pkv_plan_build_shared.argtypes = [vp, vp, i32, i32, i32, i32, vp, sz]
    L.pkv_plan_build_shared.restype = i32
    L.pkv_plan_workspace_bytes.argtypes = [vp]
    L.pkv_plan_workspace_bytes.restype = sz
    L.pkv_paged_decode_attention_planned.argtypes = [vp, vp, i64, vp, i32, vp, i32, i32, i32,
                                                     i32, i32, f32, vp, vp, vp, vp, sz, vp, vp]
    L.pkv_paged_decode_attention_planned.restype = i32
    L.pkv_decode_step_planned.argtypes = [vp, vp, vp, vp, i64, vp, i32, vp, i32, i32, i32, i32,
                                          i32, f64, f32, vp, vp, vp, vp, sz, vp, vp]
    L.pkv_decode_step_planned.restype = i32
    L.pkv_decode_steps_planned.argtypes = [i32] + L.pkv_decode_step_planned.argtypes
    L.pkv_decode_steps_planned.restype = i32
    L.pkv_kv_write_prefill_layers.argtypes = [i32] + L.pkv_kv_write_prefill.argtypes
    L.pkv_kv_write_prefill_layers.restype = i32
    return L


_lib = _load()


def lib():
    return _lib


def abi_version() -> int:
    return _lib.pkv_abi_version()


def strerror(status: int) -> str:
    return _lib.pkv_strerror(status).decode()


DEFAULT_WAIT_NS = 2_000_000_000


def set_wait_limit_ns(ns: int) -> int:
    """Limit of each in-kernel wait for the kernels this thread launches from
    now on (pkv_set_wait_limit_ns); returns the previous limit."""
    if ns < 0:
        raise ValueError("the wait limit is a number of nanoseconds >= 0")
    return int(_lib.pkv_set_wait_limit_ns(int(ns)))


def plan_splits(batch: int, max_blocks: int, num_splits: int = 0,
                num_kv_heads: int = NUM_KV_HEADS) -> int:
    return _lib.pkv_plan_splits(batch, num_kv_heads, max_blocks, num_splits)


def workspace_bytes(batch: int, max_blocks: int, num_splits: int = 0, *,
                    num_q_heads: int = NUM_Q_HEADS, num_kv_heads: int = NUM_KV_HEADS,
                    head_dim: int = HEAD_DIM) -> int:
    n = _lib.pkv_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks,
                                 num_splits)
    if n == ctypes.c_size_t(-1).value:
        raise PkvError(PKV_EINVAL, "pkv_workspace_bytes")
    return n


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _pool_pages(pool):
    _check(pool, "pool", torch.bfloat16)
    if pool.dim() != 5 or tuple(pool.shape[1:]) != (2, PAGE_SIZE, NUM_KV_HEADS, HEAD_DIM):
        raise ValueError("pool must be [num_pages][2][16][8][64] bf16")
    return pool.shape[0]


def kv_append(k_new, v_new, pool, block_table, positions, *, rope_theta: float = 500000.0,
              q_in=None, q_out=None, dev_err=None, stream=None) -> None:
    """Append one token per sequence: pool[bt[b][pos/16]][K|V][pos%16] = RoPE(k), v."""
    num_pages = _pool_pages(pool)
    dev = pool.device
    _check(k_new, "k_new", torch.bfloat16, 3, dev)
    _check(v_new, "v_new", torch.bfloat16, 3, dev)
    _check(block_table, "block_table", torch.int32, 2, dev)
    _check(positions, "positions", torch.int32, 1, dev)
    B, Hkv, D = k_new.shape
    if v_new.shape != k_new.shape or positions.shape[0] != B or block_table.shape[0] != B:
        raise ValueError("k_new, v_new, positions and block_table disagree on the batch")
    Hq = 0
    if q_in is not None or q_out is not None:
        _check(q_in, "q_in", torch.bfloat16, 3, dev)
        _check(q_out, "q_out", torch.bfloat16, 3, dev)
        if q_in.shape != q_out.shape or q_in.shape[0] != B:
            raise ValueError("q_in / q_out shape mismatch")
        Hq = q_in.shape[1]
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, None, dev)
    rc = _lib.pkv_kv_append(_ptr(k_new), _ptr(v_new), _ptr(pool), num_pages, _ptr(block_table),
                            block_table.shape[1], _ptr(positions), B, Hkv, D, PAGE_SIZE,
                            float(rope_theta), _ptr(q_in), _ptr(q_out), Hq, _ptr(dev_err),
                            _stream(stream))
    if rc != PKV_OK:
        raise PkvError(rc, "pkv_kv_append")


def paged_decode_attention(q, pool, block_table, seq_lens, out=None, *, scale: float = None,
                           workspace=None, num_splits: int = 0, dev_err=None,
                           stream=None) -> torch.Tensor:
    """out[b][j] = softmax(scale * q[b][j] . K) V over the sequence's pages."""
    num_pages = _pool_pages(pool)
    dev = pool.device
    _check(q, "q", torch.bfloat16, 3, dev)
    _check(block_table, "block_table", torch.int32, 2, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    if seq_lens.shape[0] != B or block_table.shape[0] != B:
        raise ValueError("q, seq_lens and block_table disagree on the batch")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3, dev)
    if scale is None:
        scale = D ** -0.5
    max_blocks = block_table.shape[1]
    need = workspace_bytes(B, max_blocks, num_splits, num_q_heads=Hq, head_dim=D)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the pool's device")
        ws_bytes = workspace.numel() * workspace.element_size()
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, None, dev)
    rc = _lib.pkv_paged_decode_attention(
        _ptr(q), _ptr(pool), num_pages, _ptr(block_table), max_blocks, _ptr(seq_lens), B, Hq,
        NUM_KV_HEADS, D, PAGE_SIZE, float(scale), _ptr(out), _ptr(workspace), ws_bytes,
        int(num_splits), _ptr(dev_err), _stream(stream))
    if rc != PKV_OK:
        raise PkvError(rc, "pkv_paged_decode_attention")
    return out


def decode_step(q, k_new, v_new, pool, block_table, seq_lens, out=None, *,
                rope_theta: float = 500000.0, scale: float = None, workspace=None,
                num_splits: int = 0, dev_err=None, stream=None) -> torch.Tensor:
    """One fused decode step: append (k_new, v_new) at seq_lens - 1, then attend."""
    num_pages = _pool_pages(pool)
    dev = pool.device
    _check(q, "q", torch.bfloat16, 3, dev)
    _check(k_new, "k_new", torch.bfloat16, 3, dev)
    _check(v_new, "v_new", torch.bfloat16, 3, dev)
    _check(block_table, "block_table", torch.int32, 2, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    if (seq_lens.shape[0] != B or block_table.shape[0] != B or k_new.shape[0] != B
            or v_new.shape != k_new.shape):
        raise ValueError("q, k_new, v_new, seq_lens and block_table disagree on the batch")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3, dev)
    if scale is None:
        scale = D ** -0.5
    max_blocks = block_table.shape[1]
    need = workspace_bytes(B, max_blocks, num_splits, num_q_heads=Hq, head_dim=D)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the pool's device")
        ws_bytes = workspace.numel() * workspace.element_size()
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, None, dev)
    rc = _lib.pkv_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(pool), num_pages, _ptr(block_table), max_blocks,
        _ptr(seq_lens), B, Hq, k_new.shape[1], D, PAGE_SIZE, float(rope_theta), float(scale),
        _ptr(out), _ptr(workspace), ws_bytes, int(num_splits), _ptr(dev_err), _stream(stream))
    if rc != PKV_OK:
        raise PkvError(rc, "pkv_decode_step")
    return out


def kv_write_prefill(k, v, token_offsets, start_positions, pool, block_table, *,
                     rope_theta: float = 500000.0, dev_err=None, stream=None) -> None:
    """Write a ragged batch of tokens (k, v: [num_tokens][Hkv][D]) into their pages."""
    num_pages = _pool_pages(pool)
    dev = pool.device
    _check(k, "k", torch.bfloat16, 3, dev)
    _check(v, "v", torch.bfloat16, 3, dev)
    _check(token_offsets, "token_offsets", torch.int32, 1, dev)
    _check(start_positions, "start_positions", torch.int32, 1, dev)
    _check(block_table, "block_table", torch.int32, 2, dev)
    B = start_positions.shape[0]
    if token_offsets.shape[0] != B + 1 or block_table.shape[0] != B or v.shape != k.shape:
        raise ValueError("token_offsets must have batch + 1 entries; k/v shapes must match")
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, None, dev)
    rc = _lib.pkv_kv_write_prefill(_ptr(k), _ptr(v), k.shape[0], _ptr(token_offsets),
                                   _ptr(start_positions), _ptr(pool), num_pages,
                                   _ptr(block_table), block_table.shape[1], B, k.shape[1],
                                   k.shape[2], PAGE_SIZE, float(rope_theta), _ptr(dev_err),
                                   _stream(stream))
    if rc != PKV_OK:
        raise PkvError(rc, "pkv_kv_write_prefill")


def kv_write_prefill_layers(ks, vs, token_offsets, start_positions, pool, block_tables, *,
                            rope_theta: float = 500000.0, dev_err=None, stream=None) -> None:
    """kv_write_prefill for every layer in one native call: ks, vs
    [layers][num_tokens][Hkv][D], block_tables [layers][B][max_blocks]."""
    num_pages = _pool_pages(pool)
    dev = pool.device
    _check(ks, "ks", torch.bfloat16, 4, dev)
    _check(vs, "vs", torch.bfloat16, 4, dev)
    _check(token_offsets, "token_offsets", torch.int32, 1, dev)
    _check(start_positions, "start_positions", torch.int32, 1, dev)
    _check(block_tables, "block_tables", torch.int32, 3, dev)
    layers, B = block_tables.shape[0], start_positions.shape[0]
    if (token_offsets.shape[0] != B + 1 or block_tables.shape[1] != B or vs.shape != ks.shape
            or ks.shape[0] != layers):
        raise ValueError("token_offsets must have batch + 1 entries; ks/vs/block_tables must "
                         "hold the same layers")
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, None, dev)
    rc = _lib.pkv_kv_write_prefill_layers(
        layers, _ptr(ks), _ptr(vs), ks.shape[1], _ptr(token_offsets), _ptr(start_positions),
        _ptr(pool), num_pages, _ptr(block_tables), block_tables.shape[2], B, ks.shape[2],
        ks.shape[3], PAGE_SIZE, float(rope_theta), _ptr(dev_err), _stream(stream))
    if rc != PKV_OK:
        raise PkvError(rc, "pkv_kv_write_prefill_layers")


def attention_kernels(batch: int, max_blocks: int, num_splits: int = 0, plan=None) -> str:
    """The kernels an attention call launches for these sizes ('+'-joined)."""
    r = _lib.pkv_attention_kernels(batch, max_blocks, num_splits,
                                   None if plan is None else plan._host_ptr())
    if r is None:
        raise PkvError(PKV_EINVAL, "pkv_attention_kernels")
    return r.decode()


# ----------------------------------------------------------- host checks --

def check_tables(block_table, seq_lens, num_pages: int, page_size: int = PAGE_SIZE) -> None:
    """Raise PkvError naming the first bad length or live block-table entry
    (pkv_check_tables: host arrays, checked before any launch)."""
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    if bt.ndim != 2 or lens.ndim != 1 or bt.shape[0] != lens.shape[0]:
        raise ValueError("block_table must be [batch][max_blocks] and seq_lens [batch]")
    seq, blk = ctypes.c_int(0), ctypes.c_int(0)
    rc = _lib.pkv_check_tables(bt.ctypes.data_as(ctypes.c_void_p), bt.shape[1],
                               lens.ctypes.data_as(ctypes.c_void_p), lens.shape[0], num_pages,
                               page_size, ctypes.byref(seq), ctypes.byref(blk))
    if rc != PKV_OK:
        where = (f"sequence {seq.value}: length {int(lens[seq.value])}" if blk.value < 0 and
                 seq.value >= 0 else f"sequence {seq.value}, block {blk.value}: page "
                 f"{int(bt[seq.value, blk.value])}" if seq.value >= 0 else "bad sizes")
        raise PkvError(rc, f"pkv_check_tables ({where})")


# ------------------------------------------------------------- work plans --

class Plan:
    """A work plan for one batch, built on the host from host lengths
    (pkv_plan_build in include/pkv.h): ranges of the long sequences first,
    short sequences packed one per warp.  ``to(device)`` uploads it; the
    planned calls take the plan object itself."""

    HEADER = ("magic", "batch", "max_blocks", "num_items", "num_merges", "num_slots",
              "range_pages", "bytes_used", "num_shared", "shared_pages", "num_segs", "layout")

    def __init__(self, seq_lens_host, max_blocks: int, *, num_sms: int = 0, device=None,
                 out=None, block_tables=None, min_shared_pages: int = 16):
        """out: an int32 array of at least plan_bytes(len(seq_lens_host), max_blocks)
        bytes, 16-byte aligned, to build the plan in (e.g. a view of pinned
        staging memory); by default the plan gets a buffer of its own.
        block_tables: the host copy of this layer's tables [B][max_blocks];
        when given, runs of consecutive sequences whose tables start with the
        same min_shared_pages or more pages get them as shared-prefix items
        (pkv_plan_build_shared)."""
        lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
        if lens.ndim != 1:
            raise ValueError("seq_lens_host must be one-dimensional")
        nbytes = _lib.pkv_plan_bytes(lens.shape[0], max_blocks)
        if nbytes == 0:
            raise PkvError(PKV_EINVAL, "pkv_plan_bytes")
        if out is None:
            raw = np.zeros(nbytes // 4 + 4, dtype=np.int32)
            off = (-raw.ctypes.data % 16) // 4      # 16-byte aligned view
            buf = raw[off:off + nbytes // 4]
        else:
            if (out.dtype != np.int32 or out.ndim != 1 or out.shape[0] * 4 < nbytes
                    or out.ctypes.data % 16 or not out.flags.c_contiguous):
                raise ValueError("out must be a contiguous, 16-byte aligned int32 array of at "
                                 "least plan_bytes() bytes")
            raw = out
            buf = out[: nbytes // 4]
        if block_tables is None:
            rc = _lib.pkv_plan_build(lens.ctypes.data_as(ctypes.c_void_p), lens.shape[0],
                                     max_blocks, num_sms, buf.ctypes.data_as(ctypes.c_void_p),
                                     nbytes)
            what = "pkv_plan_build"
        else:
            bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
            if bt.shape != (lens.shape[0], max_blocks):
                raise ValueError("block_tables must be [batch][max_blocks] int32")
            rc = _lib.pkv_plan_build_shared(lens.ctypes.data_as(ctypes.c_void_p),
                                            bt.ctypes.data_as(ctypes.c_void_p), lens.shape[0],
                                            max_blocks, num_sms, int(min_shared_pages),
                                            buf.ctypes.data_as(ctypes.c_void_p), nbytes)
            what = "pkv_plan_build_shared"
        if rc != PKV_OK:
            raise PkvError(rc, what)
        self._raw = raw
        self._buf = buf
        self._args = (lens.shape[0], max_blocks, num_sms, int(min_shared_pages),
                      buf.ctypes.data, nbytes)
        self._read_header()
        self.dev = None
        if device is not None:
            self.to(device)

    def _read_header(self):
        buf = self._buf
        self.host = buf[: int(buf[7]) // 4]
        for i, name in enumerate(self.HEADER):
            setattr(self, name, int(buf[i]))
        self.workspace_bytes = int(_lib.pkv_plan_workspace_bytes(self._args[4]))

    def rebuild(self, seq_lens_host, block_tables=None):
        """Build this step's plan into the same buffer (what a serving loop does
        every step): seq_lens_host and block_tables must be C-contiguous int32
        numpy arrays of this plan's batch ([B], [B][max_blocks]); no copies are
        made.  The device copy (``dev``) is not touched."""
        B, max_blocks, num_sms, min_shared, buf_ptr, nbytes = self._args
        if block_tables is None:
            rc = _lib.pkv_plan_build(seq_lens_host.ctypes.data, B, max_blocks, num_sms, buf_ptr,
                                     nbytes)
        else:
            rc = _lib.pkv_plan_build_shared(seq_lens_host.ctypes.data, block_tables.ctypes.data,
                                            B, max_blocks, num_sms, min_shared, buf_ptr, nbytes)
        if rc != PKV_OK:
            raise PkvError(rc, "pkv_plan_build")
        self._read_header()
        return self

    def items(self) -> np.ndarray:
        """[num_items][16] int32.  Kinds 0 (range) and 1 (packed): kind, slot,
        p_begin, n, seq[4], len[4], 0 x 4.  Kind 2 (segment CTA): 2, first
        segment, segments, pages, 0 x 12."""
        o = PLAN_HEADER_WORDS
        return self.host[o:o + 16 * self.num_items].reshape(self.num_items, 16)

    def merges(self) -> np.ndarray:
        """[num_merges][4] int32: sequence, first slot, ranges, 0."""
        o = PLAN_HEADER_WORDS + 16 * self.num_items
        return self.host[o:o + 4 * self.num_merges].reshape(self.num_merges, 4)

    def shared(self) -> np.ndarray:
        """[num_shared][36] int32: members, p_begin, n, 0, seq[16], slot[16]."""
        o = PLAN_HEADER_WORDS + 16 * self.num_items + 4 * self.num_merges
        return self.host[o:o + 36 * self.num_shared].reshape(self.num_shared, 36)

    def segments(self) -> np.ndarray:
        """[num_segs][8] int32: b, L, p_begin, n, slot (-1: writes the output), fold,
        fold_slot, 0 (fold > 0: the output takes in the partials of slots
        [fold_slot, fold_slot + fold) too);
        item i of kind 2 runs segments [items()[i, 1], items()[i, 1] + items()[i, 2])."""
        o = PLAN_HEADER_WORDS + 16 * self.num_items + 4 * self.num_merges + 36 * self.num_shared
        return self.host[o:o + 8 * self.num_segs].reshape(self.num_segs, 8)

    def to(self, device):
        """Copy the plan to `device`, asynchronously on the current stream (through
        pinned memory, so the host does not wait for the work queued before it)."""
        staged = torch.empty(self.host.shape[0], dtype=torch.int32, pin_memory=True)
        staged.numpy()[:] = self.host
        self.dev = staged.to(device, non_blocking=True)
        return self

    def _host_ptr(self):
        return self.host.ctypes.data_as(ctypes.c_void_p)


def plan_bytes(batch: int, max_blocks: int) -> int:
    """Bytes a plan for this batch and table width can take (pkv_plan_bytes)."""
    return int(_lib.pkv_plan_bytes(batch, max_blocks))


def _plan_workspace(plan, workspace, dev):
    if plan.dev is None or plan.dev.device != dev:
        raise ValueError("upload the plan to the pool's device first (Plan.to)")
    need = plan.workspace_bytes
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the pool's device")
        ws_bytes = workspace.numel() * workspace.element_size()
    return workspace, ws_bytes


def paged_decode_attention_planned(q, pool, block_table, seq_lens, plan, out=None, *,
                                   scale: float = None, workspace=None, dev_err=None,
                                   stream=None) -> torch.Tensor:
    """paged_decode_attention under a work plan built for these lengths."""
    num_pages = _pool_pages(pool)
    dev = pool.device
    _check(q, "q", torch.bfloat16, 3, dev)
    _check(block_table, "block_table", torch.int32, 2, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3, dev)
    if scale is None:
        scale = D ** -0.5
    workspace, ws_bytes = _plan_workspace(plan, workspace, dev)
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, None, dev)
    rc = _lib.pkv_paged_decode_attention_planned(
        _ptr(q), _ptr(pool), num_pages, _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
        Hq, NUM_KV_HEADS, D, PAGE_SIZE, float(scale), _ptr(out), plan._host_ptr(), _ptr(plan.dev),
        _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    if rc != PKV_OK:
        raise PkvError(rc, "pkv_paged_decode_attention_planned")
    return out


def decode_step_planned(q, k_new, v_new, pool, block_table, seq_lens, plan, out=None, *,
                        rope_theta: float = 500000.0, scale: float = None, workspace=None,
                        dev_err=None, stream=None) -> torch.Tensor:
    """decode_step under a work plan built for these lengths."""
    num_pages = _pool_pages(pool)
    dev = pool.device
    _check(q, "q", torch.bfloat16, 3, dev)
    _check(k_new, "k_new", torch.bfloat16, 3, dev)
    _check(v_new, "v_new", torch.bfloat16, 3, dev)
    _check(block_table, "block_table", torch.int32, 2, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3, dev)
    if scale is None:
        scale = D ** -0.5
    workspace, ws_bytes = _plan_workspace(plan, workspace, dev)
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, None, dev)
    rc = _lib.pkv_decode_step_planned(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(pool), num_pages, _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, Hq, k_new.shape[1], D, PAGE_SIZE,
        float(rope_theta), float(scale), _ptr(out), plan._host_ptr(), _ptr(plan.dev),
        _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    if rc != PKV_OK:
        raise PkvError(rc, "pkv_decode_step_planned")
    return out


def decode_steps_planned(qs, k_news, v_news, pool, block_tables, seq_lens, plan, out=None, *,
                         rope_theta: float = 500000.0, scale: float = None, workspace=None,
                         dev_err=None, stream=None) -> torch.Tensor:
    """decode_step_planned for every layer of one step in one native call:
    qs [layers][B][Hq][D], k_news / v_news [layers][B][Hkv][D], block_tables
    [layers][B][max_blocks]; the lengths, plan and workspace are shared."""
    num_pages = _pool_pages(pool)
    dev = pool.device
    _check(qs, "qs", torch.bfloat16, 4, dev)
    _check(k_news, "k_news", torch.bfloat16, 4, dev)
    _check(v_news, "v_news", torch.bfloat16, 4, dev)
    _check(block_tables, "block_tables", torch.int32, 3, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    layers, B, Hq, D = qs.shape
    if k_news.shape[0] != layers or v_news.shape[0] != layers or block_tables.shape[0] != layers:
        raise ValueError("qs, k_news, v_news and block_tables must hold the same layers")
    if tuple(k_news.shape[1:]) != (B, NUM_KV_HEADS, D) or v_news.shape != k_news.shape:
        raise ValueError("k_news and v_news must be [layers][B][8][64]")
    if block_tables.shape[1] != B:
        raise ValueError("block_tables must be [layers][B][max_blocks]")
    if out is None:
        out = torch.empty_like(qs)
    _check(out, "out", torch.bfloat16, 4, dev)
    if out.shape != qs.shape:
        raise ValueError("out must have the shape of qs")
    if scale is None:
        scale = D ** -0.5
    workspace, ws_bytes = _plan_workspace(plan, workspace, dev)
    if dev_err is not None:
        _check(dev_err, "dev_err", torch.int32, None, dev)
    rc = _lib.pkv_decode_steps_planned(
        layers, _ptr(qs), _ptr(k_news), _ptr(v_news), _ptr(pool), num_pages, _ptr(block_tables),
        block_tables.shape[2], _ptr(seq_lens), B, Hq, k_news.shape[2], D, PAGE_SIZE,
        float(rope_theta), float(scale), _ptr(out), plan._host_ptr(), _ptr(plan.dev),
        _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    if rc != PKV_OK:
        raise PkvError(rc, "pkv_decode_steps_planned")
    return out
