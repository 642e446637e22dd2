"""The attention entry point that allocates nothing (GPU).

pkv_paged_decode_attention_static_ws serves callers that may not call
cudaMalloc (allocator hooks, host callbacks, processes whose device memory is
owned by another framework's allocator): its split-K partials live in a fixed
device buffer inside libpkv instead of a caller workspace.  This file is named
to be collected last, so a stop-at-first-failure run has already run every
other test when it gets here; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 4 << 20
PKV_ESCRATCH = 6


def _entry(lib):
    f = lib.pkv_paged_decode_attention_static_ws
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [vp, vp, i64, vp, i32, vp, i32, i32, i32, i32, i32, ctypes.c_float, vp, i32,
                  vp, vp]
    f.restype = i32
    return f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_static_scratch_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from paged_kv_decode_04_gb300 import binding, synth
    from _gpu_util import TOL_ABS, TOL_REL

    dev = torch.device("cuda", 0)
    w = synth.make_workload("small", 4)
    d = synth.device_inputs(w, dev)
    bt, lens = d["block_tables"][0], d["seq_lens"]
    binding.kv_append(d["k_new"][0], d["v_new"][0], d["pool"], bt, d["positions"])
    f = _entry(binding.lib())
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for splits in (8, 3):
        need = binding.workspace_bytes(w.batch, w.max_blocks, splits)
        assert 0 < need <= STATIC_SCRATCH_BYTES
        want = binding.paged_decode_attention(d["q"][0], d["pool"], bt, lens, num_splits=splits)
        for call in range(2):   # the second call reuses the buffer the first one left behind
            out = torch.full_like(want, float("nan"))
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            rc = f(_p(d["q"][0]), _p(d["pool"]), w.num_pages, _p(bt), w.max_blocks, _p(lens),
                   w.batch, 32, 8, 64, 16, w.scale, _p(out), splits, _p(err), stream)
            assert rc == 0, binding.strerror(rc)
            torch.cuda.synchronize(dev)
            assert int(err.item()) == 0
            a = out.float().cpu().numpy()
            b = want.float().cpu().numpy()
            assert np.all(np.abs(a - b) <= TOL_ABS + TOL_REL * np.abs(b)), (splits, call)
            # the same plan and kernels as the workspace entry point: the same bits,
            # so a partial left in the buffer by an earlier call cannot hide
            assert torch.equal(out.view(torch.int16), want.view(torch.int16)), (splits, call)


def test_static_scratch_rejects_oversized_plans_before_launch():
    from paged_kv_decode_04_gb300 import binding
    f = _entry(binding.lib())
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: the size check comes first
    batch, splits = 512, 16           # 512 x 32 heads x 16 splits x 66 floats > 4 MiB
    assert binding.workspace_bytes(batch, 128, splits) > STATIC_SCRATCH_BYTES
    rc = f(fake, fake, 64, fake, 128, fake, batch, 32, 8, 64, 16, 0.125, fake, splits, None,
           None)
    assert rc == PKV_ESCRATCH
    assert "static scratch" in binding.strerror(rc)
