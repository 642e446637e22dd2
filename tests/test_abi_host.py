"""The C-ABI library loads, exports what include/pkv.h declares, and rejects bad
arguments on the host before anything touches a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_04_gb300 import build
    path = build.build()
    L = ctypes.CDLL(path)
    from paged_kv_decode_04_gb300 import binding  # sets prototypes on its own handle
    return binding.lib()


def declared_symbols():
    names = []
    for h in HEADERS:
        names += re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", open(h).read())
    return names


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    assert {"pkv_kv_append", "pkv_paged_decode_attention", "pkv_workspace_bytes",
            "pkv_strerror", "pkv_abi_version", "pkv_plan_splits", "pkv_decode_step",
            "pkv_kv_write_prefill", "pkv_sched_create", "pkv_sched_admit",
            "pkv_sched_decode_batch"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_strerror_and_version(lib):
    from paged_kv_decode_04_gb300 import binding
    assert binding.abi_version() == 1
    for s in range(0, 7):
        assert isinstance(binding.strerror(s), str) and binding.strerror(s)
    assert binding.strerror(0) == "ok"


def test_explicit_split_plans(lib):
    from paged_kv_decode_04_gb300 import binding
    assert binding.plan_splits(256, 128, 1) == 1
    assert binding.plan_splits(1, 128, 32) == 32
    assert binding.plan_splits(1, 128, 7) == 7        # ceil(128/7)=19 pages per range -> 7 ranges
    assert binding.plan_splits(1, 128, 500) == 128    # at most one page per range
    assert binding.plan_splits(8, 128, 10) == 10
    assert binding.plan_splits(0, 128, 1) == -1
    assert binding.workspace_bytes(1, 128, 1) == 0
    assert binding.workspace_bytes(2, 128, 4) == 2 * 32 * 4 * (64 + 2) * 4


# Fake, never-dereferenced device addresses: every call below must fail its
# host-side checks before anything is enqueued.
A = ctypes.c_void_p(0x10000)


def attn(lib, **kw):
    args = dict(q=A, pool=A, num_pages=64, bt=A, max_blocks=128, lens=A, batch=1, hq=32, hkv=8,
                d=64, ps=16, scale=0.125, out=A, ws=None, ws_bytes=0, splits=1, err=None,
                stream=None)
    args.update(kw)
    return lib.pkv_paged_decode_attention(*args.values())


def test_attention_argument_errors(lib):
    from paged_kv_decode_04_gb300 import binding as B
    assert attn(lib, q=None) == B.PKV_EINVAL
    assert attn(lib, out=None) == B.PKV_EINVAL
    assert attn(lib, batch=-1) == B.PKV_EINVAL
    assert attn(lib, num_pages=0) == B.PKV_EINVAL
    assert attn(lib, scale=0.0) == B.PKV_EINVAL
    assert attn(lib, scale=float("nan")) == B.PKV_EINVAL
    assert attn(lib, splits=-1) == B.PKV_EINVAL
    assert attn(lib, hq=16) == B.PKV_EUNSUPPORTED
    assert attn(lib, d=128) == B.PKV_EUNSUPPORTED
    assert attn(lib, ps=32) == B.PKV_EUNSUPPORTED
    assert attn(lib, q=ctypes.c_void_p(0x10002)) == B.PKV_EALIGN
    assert attn(lib, pool=ctypes.c_void_p(0x10008)) == B.PKV_EALIGN
    assert attn(lib, splits=4, ws=None) == B.PKV_EWORKSPACE
    assert attn(lib, splits=4, ws=A, ws_bytes=100) == B.PKV_EWORKSPACE
    assert attn(lib, batch=0) == B.PKV_OK      # nothing to do, nothing enqueued


def append(lib, **kw):
    args = dict(k=A, v=A, pool=A, num_pages=64, bt=A, max_blocks=128, pos=A, batch=1, hkv=8,
                d=64, ps=16, theta=500000.0, q_in=None, q_out=None, hq=0, err=None, stream=None)
    args.update(kw)
    return lib.pkv_kv_append(*args.values())


def test_append_argument_errors(lib):
    from paged_kv_decode_04_gb300 import binding as B
    assert append(lib, k=None) == B.PKV_EINVAL
    assert append(lib, pos=None) == B.PKV_EINVAL
    assert append(lib, theta=-1.0) == B.PKV_EINVAL
    assert append(lib, q_in=A) == B.PKV_EINVAL           # q_in without q_out
    assert append(lib, hkv=4) == B.PKV_EUNSUPPORTED
    assert append(lib, q_in=A, q_out=A, hq=8) == B.PKV_EUNSUPPORTED
    assert append(lib, v=ctypes.c_void_p(0x10002)) == B.PKV_EALIGN
    assert append(lib, batch=0) == B.PKV_OK


def test_decode_step_and_prefill_argument_errors(lib):
    from paged_kv_decode_04_gb300 import binding as B
    f = lib.pkv_decode_step

    def step(**kw):
        args = dict(q=A, k=A, v=A, pool=A, num_pages=64, bt=A, max_blocks=128, lens=A, batch=1,
                    hq=32, hkv=8, d=64, ps=16, theta=500000.0, scale=0.125, out=A, ws=None,
                    ws_bytes=0, splits=1, err=None, stream=None)
        args.update(kw)
        return f(*args.values())
    assert step(k=None) == B.PKV_EINVAL
    assert step(theta=0.0) == B.PKV_EINVAL
    assert step(hkv=4) == B.PKV_EUNSUPPORTED
    assert step(v=ctypes.c_void_p(0x10002)) == B.PKV_EALIGN
    assert step(splits=8) == B.PKV_EWORKSPACE
    assert step(batch=0) == B.PKV_OK

    g = lib.pkv_kv_write_prefill

    def pre(**kw):
        args = dict(k=A, v=A, n=10, off=A, st=A, pool=A, num_pages=64, bt=A, max_blocks=128,
                    batch=1, hkv=8, d=64, ps=16, theta=500000.0, err=None, stream=None)
        args.update(kw)
        return g(*args.values())
    assert pre(off=None) == B.PKV_EINVAL
    assert pre(n=-1) == B.PKV_EINVAL
    assert pre(batch=0) == B.PKV_EINVAL
    assert pre(d=128) == B.PKV_EUNSUPPORTED
    assert pre(pool=ctypes.c_void_p(0x10004)) == B.PKV_EALIGN
    assert pre(n=0) == B.PKV_OK


def test_multi_layer_planned_step_argument_errors(lib):
    import numpy as np
    from paged_kv_decode_04_gb300 import binding as B
    plan = B.Plan(np.array([40], np.int32), 128, num_sms=152)
    f = lib.pkv_decode_steps_planned

    def steps(**kw):
        args = dict(layers=2, q=A, k=A, v=A, pool=A, num_pages=64, bt=A, max_blocks=128, lens=A,
                    batch=1, hq=32, hkv=8, d=64, ps=16, theta=500000.0, scale=0.125, out=A,
                    plan_host=plan._host_ptr(), plan_dev=A, ws=None, ws_bytes=0, err=None,
                    stream=None)
        args.update(kw)
        return f(*args.values())
    assert steps(layers=0) == B.PKV_EINVAL
    assert steps(layers=-3) == B.PKV_EINVAL
    assert steps(k=None) == B.PKV_EINVAL
    assert steps(plan_host=None) == B.PKV_EINVAL
    assert steps(batch=2) == B.PKV_EINVAL                # the plan is for one sequence
    assert steps(hkv=4) == B.PKV_EUNSUPPORTED
    assert steps(v=ctypes.c_void_p(0x10002)) == B.PKV_EALIGN


def test_multi_layer_prefill_argument_errors(lib):
    from paged_kv_decode_04_gb300 import binding as B
    f = lib.pkv_kv_write_prefill_layers

    def pre(**kw):
        args = dict(layers=3, k=A, v=A, n=10, off=A, st=A, pool=A, num_pages=64, bt=A,
                    max_blocks=128, batch=1, hkv=8, d=64, ps=16, theta=500000.0, err=None,
                    stream=None)
        args.update(kw)
        return f(*args.values())
    assert pre(layers=0) == B.PKV_EINVAL
    assert pre(off=None) == B.PKV_EINVAL
    assert pre(d=128) == B.PKV_EUNSUPPORTED
    assert pre(v=ctypes.c_void_p(0x10004)) == B.PKV_EALIGN
    assert pre(n=0) == B.PKV_OK
