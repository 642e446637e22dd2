"""ctypes binding of the host scheduler in libpkv (include/pkv_sched.h).

Marshalling only; the admission, allocation and batching decisions are made
by the C++ scheduler.  Runs without a GPU.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import binding

PKV_EREJECTED = 7
PKV_ENOTFOUND = 8


class SchedStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in (
        "pool_pages", "free_pages", "free_credits", "peak_active", "largest_decode_batch",
        "peak_allocated_pages", "admission_wait_total", "admission_wait_max", "submitted",
        "admitted", "rejected", "finished", "waiting", "active")]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def _lib():
    L = binding.lib()
    if not getattr(L, "_sched_ready", False):
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.pkv_sched_create.argtypes = [i64, i32, i32, i32, i32]
        L.pkv_sched_create.restype = vp
        L.pkv_sched_destroy.argtypes = [vp]
        L.pkv_sched_destroy.restype = None
        L.pkv_sched_budget_pages.argtypes = [vp, i32, i32]
        L.pkv_sched_budget_pages.restype = i64
        L.pkv_sched_submit.argtypes = [vp, i32, i32, ctypes.POINTER(i64)]
        L.pkv_sched_submit.restype = i32
        L.pkv_sched_admit.argtypes = [vp]
        L.pkv_sched_admit.restype = i32
        L.pkv_sched_next_prefill.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_int32),
                                             vp]
        L.pkv_sched_next_prefill.restype = i32
        L.pkv_sched_decode_batch.argtypes = [vp, i32, vp, vp, vp]
        L.pkv_sched_decode_batch.restype = i32
        L.pkv_sched_running.argtypes = [vp]
        L.pkv_sched_running.restype = i32
        L.pkv_sched_finish.argtypes = [vp, i64]
        L.pkv_sched_finish.restype = i32
        L.pkv_sched_seq_len.argtypes = [vp, i64]
        L.pkv_sched_seq_len.restype = ctypes.c_int32
        L.pkv_sched_get_stats.argtypes = [vp, ctypes.POINTER(SchedStats)]
        L.pkv_sched_get_stats.restype = None
        L._sched_ready = True
    return L


class Scheduler:
    """Page-credit admission, lazy page allocation, static or continuous batching."""

    def __init__(self, num_pages: int, layers: int, max_context: int = 2048,
                 page_size: int = 16, static_batching: bool = False):
        self._L = _lib()
        self._h = self._L.pkv_sched_create(num_pages, layers, max_context, page_size,
                                           int(static_batching))
        if not self._h:
            raise ValueError("bad scheduler sizes")
        self.layers = layers
        self.max_blocks = max_context // page_size

    def close(self):
        if self._h:
            self._L.pkv_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def budget_pages(self, prompt: int, max_new: int) -> int:
        return self._L.pkv_sched_budget_pages(self._h, prompt, max_new)

    def submit(self, prompt: int, max_new: int):
        """Request id, or None if rejected (budget larger than the pool)."""
        rid = ctypes.c_int64(-1)
        rc = self._L.pkv_sched_submit(self._h, prompt, max_new, ctypes.byref(rid))
        if rc == PKV_EREJECTED:
            return None
        if rc != 0:
            raise ValueError(binding.strerror(rc))
        return rid.value

    def admit(self) -> int:
        return self._L.pkv_sched_admit(self._h)

    def next_prefill(self):
        """(id, prompt_tokens, block_tables [layers][max_blocks]) or None."""
        rid = ctypes.c_int64(-1)
        plen = ctypes.c_int32(0)
        bt = np.empty((self.layers, self.max_blocks), dtype=np.int32)
        got = self._L.pkv_sched_next_prefill(self._h, ctypes.byref(rid), ctypes.byref(plen),
                                             bt.ctypes.data_as(ctypes.c_void_p))
        return (rid.value, plen.value, bt) if got else None

    def running(self) -> int:
        """Prefilled, unfinished requests: the next decode batch's size before its cap."""
        return self._L.pkv_sched_running(self._h)

    def decode_batch_into(self, ids, seq_lens, block_tables) -> int:
        """decode_batch writing into caller arrays of capacity n = len(ids): ids
        int64 [n], seq_lens int32 [n], block_tables int32 [layers][n][max_blocks]
        (C-contiguous; when the batch is n long, its tables are exactly these)."""
        n = ids.shape[0]
        if (ids.dtype != np.int64 or seq_lens.dtype != np.int32 or block_tables.dtype != np.int32
                or seq_lens.shape != (n,) or block_tables.shape != (self.layers, n, self.max_blocks)
                or not (ids.flags.c_contiguous and seq_lens.flags.c_contiguous
                        and block_tables.flags.c_contiguous)):
            raise ValueError("decode_batch_into: wrong array types or shapes")
        if n == 0:
            return 0
        return self._L.pkv_sched_decode_batch(self._h, n, ids.ctypes.data_as(ctypes.c_void_p),
                                              seq_lens.ctypes.data_as(ctypes.c_void_p),
                                              block_tables.ctypes.data_as(ctypes.c_void_p))

    def decode_batch(self, max_batch: int):
        """(ids [n], seq_lens [n], block_tables [layers][n][max_blocks])."""
        ids = np.empty(max_batch, dtype=np.int64)
        lens = np.empty(max_batch, dtype=np.int32)
        bt = np.empty((self.layers, max_batch, self.max_blocks), dtype=np.int32)
        n = self._L.pkv_sched_decode_batch(self._h, max_batch, ids.ctypes.data_as(ctypes.c_void_p),
                                           lens.ctypes.data_as(ctypes.c_void_p),
                                           bt.ctypes.data_as(ctypes.c_void_p))
        return ids[:n].copy(), lens[:n].copy(), np.ascontiguousarray(bt[:, :n])

    def finish(self, rid: int) -> bool:
        return self._L.pkv_sched_finish(self._h, rid) == 0

    def seq_len(self, rid: int) -> int:
        return self._L.pkv_sched_seq_len(self._h, rid)

    def stats(self) -> dict:
        st = SchedStats()
        self._L.pkv_sched_get_stats(self._h, ctypes.byref(st))
        return st.as_dict()
