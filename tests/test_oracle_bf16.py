"""Pins for the oracle's bf16 conversions (CPU only).

The FP64 -> bf16 rounding is checked against hand-derived golden values
(tests/golden/bf16_rne.txt) and, for values that are exactly representable in
binary32, against PyTorch's own binary32 -> bf16 round-to-nearest-even.
"""
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bf16_rne.txt")


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            x, h = line.split()
            cases.append((float.fromhex(x), int(h, 16)))
    return cases


def test_golden_rounding_cases():
    cases = _golden_cases()
    assert len(cases) >= 20
    for x, expected in cases:
        got = int(oracle.f64_to_bf16(np.array([x]))[0])
        assert got == expected, f"{x!r}: got {got:04x}, expected {expected:04x}"


def test_bf16_to_f64_is_exact_for_golden_outputs():
    # Every finite bf16 pattern in the fixture decodes to the value the fixture's
    # derivation names (2^k scalings of small integers), and re-encodes to itself.
    for _, h in _golden_cases():
        v = float(oracle.bf16_to_f64(np.array([h], dtype=np.uint16))[0])
        if np.isfinite(v):
            assert int(oracle.f64_to_bf16(np.array([v]))[0]) == h


def test_matches_torch_float32_rounding_on_float32_values():
    g = torch.Generator().manual_seed(1234)
    x32 = torch.cat([
        torch.randn(20000, generator=g),
        torch.randn(20000, generator=g) * 1e-38,   # binary32 subnormal / bf16 subnormal range
        torch.randn(20000, generator=g) * 3e38,    # near the overflow edge
        (torch.rand(20000, generator=g) * 2 - 1) * 2.0 ** -20,
    ])
    x32 = x32[torch.isfinite(x32)]
    want = x32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16(x32.double().numpy())
    mismatch = np.nonzero(want != got)[0]
    assert mismatch.size == 0, [(float(x32[i]), hex(want[i]), hex(got[i])) for i in mismatch[:5]]


def test_every_bf16_pattern_round_trips():
    pats = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f64(pats)
    finite = np.isfinite(vals)
    back = oracle.f64_to_bf16(vals[finite])
    # +0 and -0 both survive; every finite pattern maps to itself.
    assert np.array_equal(back, pats[finite])
