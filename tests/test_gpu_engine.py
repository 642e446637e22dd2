"""The scheduler driving the GPU kernels (GPU): every prefill and every decode
step of a small continuous-batching run is mirrored on the host with the FP64
oracle and compared (appended pages bit-exact at the end, outputs within
tolerance at every step)."""
import numpy as np
import pytest

import oracle
from paged_kv_decode_04_gb300 import synth
from _gpu_util import assert_close, cuda_or_skip

pytestmark = pytest.mark.gpu

POISON = 0xFFFF


@pytest.mark.parametrize("static,use_plan", [(False, True), (True, True), (False, False)])
def test_engine_run_matches_oracle_mirror(static, use_plan):
    dev = cuda_or_skip()
    from paged_kv_decode_04_gb300.engine import Engine
    num_pages, layers = 96, 2
    eng = Engine(num_pages, layers, dev, static_batching=static, max_batch=8, seed=3,
                 host_inputs=True, use_plan=use_plan)
    mirror = np.full((num_pages, 2, 16, 8, 64), POISON, dtype=np.uint16)
    checked = {"prefill": 0, "decode": 0}

    def on_prefill(layer, rid, k, v, bt):
        kb, vb = synth.bits(k), synth.bits(v)
        rc = oracle.kv_write_prefill(kb, vb, np.array([0, kb.shape[0]], np.int32),
                                     np.array([0], np.int32), mirror, bt[None])
        assert rc == 0
        checked["prefill"] += 1

    def on_decode(layer, ids, lens, bt, q, kn, vn, out):
        assert oracle.kv_append(synth.bits(kn), synth.bits(vn), mirror, bt, lens - 1) == 0
        ref = oracle.decode_attention(synth.bits(q), mirror, bt, lens)
        assert_close(synth.bits(out), ref, f"layer {layer} ids {ids.tolist()}")
        checked["decode"] += 1

    rng = np.random.default_rng(11)
    reqs = [(int(rng.integers(1, 60)), int(rng.integers(1, 40))) for _ in range(9)]
    res = eng.run(reqs, on_prefill=on_prefill, on_decode=on_decode)
    st = res["stats"]
    assert st["finished"] == len(reqs) and st["free_pages"] == num_pages
    assert checked["prefill"] == layers * len(reqs) and checked["decode"] > 0
    assert res["decode_tokens"] == sum(n - 1 for _, n in reqs)
    # every page the run wrote holds exactly what the oracle mirror holds
    assert np.array_equal(synth.bits(eng.pool), mirror)
