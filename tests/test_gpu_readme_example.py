"""The README's Python example runs as written and computes the step the
FP64 oracle computes for the same inputs (GPU)."""
import os
import re

import numpy as np
import pytest
import torch

import oracle
from _gpu_util import assert_close, cuda_or_skip

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example():
    cuda_or_skip()
    text = open(os.path.join(ROOT, "README.md"), encoding="utf-8").read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    env = {}
    exec(compile(code, "README.md", "exec"), env)
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    pool = np.zeros((4096, 2, 16, 8, 64), np.uint16)    # the example's pool before the step
    lens = env["lens_host"]
    bt = env["bt"].cpu().numpy()
    assert oracle.kv_append(bits(env["k_new"]), bits(env["v_new"]), pool, bt, lens - 1) == 0
    ref = oracle.decode_attention(bits(env["q"]), pool, bt, lens)
    assert_close(bits(env["out"]), ref, "README example")
    assert np.array_equal(bits(env["pool"]), pool)      # the appended slots, bit for bit
