"""Thousands of steps in a row raise no device error and keep their bits (GPU).

The warp-specialised kernels hand work between roles through shared-memory
barriers waited on by phase parity; a protocol in which a waiter can fall two
phases behind deadlocks only under rare timings, which the bounded waits then
report as PKV_DEVERR_TIMEOUT.  A few sample launches do not show that; long
runs of the benchmark's configurations do.  Each workload's step (every
layer, the fused step under the host plan the benchmark uses) is captured as
a CUDA graph and replayed back to back; no error bit may appear, and the last
step's outputs must equal the first's bit for bit (the repeated append writes
the same slots with the same values).
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_04_gb300 import synth
from _gpu_util import binding, cuda_or_skip

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,steps,layers,batch", [
    ("prefix", 4000, None, None), ("prefix", 1000, 4, None), ("prefix", 2000, 4, 32),
    ("mix", 600, None, None), ("peak", 1200, None, None), ("small", 4000, None, None)])
def test_many_steps_raise_no_device_error(name, steps, layers, batch):
    # prefix with 4 layers: each layer's shared-prefix grid is launched while
    # the previous layer's segment CTAs (256 sequences) or per-(item, kv head)
    # CTAs (32 sequences) still run beside its own (the plan's beside
    # layout), thousands of times in a row
    dev = cuda_or_skip()
    b = binding()
    kw = {"layers": layers} if layers else {}
    if batch:
        kw.update(batch=batch, num_pages=12000)
    w = synth.make_workload(name, 0, **kw)
    d = synth.device_inputs(w, dev)
    plan = b.Plan(w.seq_lens, w.max_blocks, device=dev, block_tables=w.block_tables[0])
    ws = torch.empty(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
    out = torch.empty((w.layers, w.batch, 32, 64), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        for layer in range(w.layers):
            b.decode_step_planned(d["q"][layer], d["k_new"][layer], d["v_new"][layer], d["pool"],
                                  d["block_tables"][layer], d["seq_lens"], plan, out[layer],
                                  rope_theta=w.rope_theta, scale=w.scale, workspace=ws,
                                  dev_err=err)

    step()
    torch.cuda.synchronize()
    first = synth.bits(out)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(steps):
        g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{name}: device error bits {int(err.item())} in {steps} steps"
    assert np.array_equal(synth.bits(out), first)
