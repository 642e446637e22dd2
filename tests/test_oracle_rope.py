"""Pins for the oracle's rotate-half RoPE (CPU only).

RoPE enters the decode step through the KV append: the new token's key is
stored at its absolute RoPE position ("Hours of YouTube and 85 handtyped pages
of notes on LLM Inference - Start here", section "これまでの進捗", KV page pool
item; RoPE also appears in the prefill item).  The pages do not state the
variant; the oracle takes rotate-half with inv_freq_i = theta^(-2i/D).  These
tests pin that reading through closed forms and an independent complex-number
formulation rather than by re-typing the oracle's formula.
"""
import math

import numpy as np
import pytest

import oracle

THETA = 500000.0
D = 64


def _rand_bf16(rng, shape):
    import torch
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_inv_freq_closed_forms():
    f = oracle.rope_inv_freq(THETA, D)
    assert f.shape == (32,)
    assert f[0] == 1.0
    assert math.isclose(f[16], 1.0 / math.sqrt(THETA), rel_tol=1e-15)
    assert math.isclose(f[8], THETA ** -0.25, rel_tol=1e-15)
    ratios = f[1:] / f[:-1]
    assert np.allclose(ratios, THETA ** (-1.0 / 32.0), rtol=1e-13, atol=0)
    assert np.all(np.diff(f) < 0)


def test_position_zero_is_identity_bit_exact():
    rng = np.random.default_rng(0)
    x = _rand_bf16(rng, D)
    assert np.array_equal(oracle.rope_rotate(x, 0, THETA), x)


def test_unit_vectors_give_cos_and_sin():
    # e_0 at position 1 rotates by 1 radian within the (0, 32) plane; e_32 likewise.
    one = 0x3F80
    e0 = np.zeros(D, dtype=np.uint16); e0[0] = one
    y = oracle.rope_rotate_f64(e0, 1, THETA)
    assert y[0] == math.cos(1.0) and y[32] == math.sin(1.0)
    assert np.count_nonzero(y) == 2
    e32 = np.zeros(D, dtype=np.uint16); e32[32] = one
    y = oracle.rope_rotate_f64(e32, 1, THETA)
    assert y[0] == -math.sin(1.0) and y[32] == math.cos(1.0)
    # pair 16 at position 7 turns by 7 / sqrt(theta)
    e16 = np.zeros(D, dtype=np.uint16); e16[16] = one
    y = oracle.rope_rotate_f64(e16, 7, THETA)
    a = 7.0 / math.sqrt(THETA)
    assert math.isclose(y[16], math.cos(a), rel_tol=1e-15)
    assert math.isclose(y[48], math.sin(a), rel_tol=1e-12)


@pytest.mark.parametrize("pos", [1, 5, 37, 511, 2047])
def test_matches_complex_multiplication(pos):
    # Independent formulation: z_i = x_i + 1j*x_{i+32} multiplied by exp(1j*pos*theta^(-i/32)).
    rng = np.random.default_rng(pos)
    x = _rand_bf16(rng, D)
    xv = oracle.bf16_to_f64(x)
    z = xv[:32] + 1j * xv[32:]
    i = np.arange(32, dtype=np.float64)
    z = z * np.exp(1j * pos * np.power(THETA, -i / 32.0))
    y = oracle.rope_rotate_f64(x, pos, THETA)
    assert np.allclose(y[:32], z.real, rtol=0, atol=1e-12)
    assert np.allclose(y[32:], z.imag, rtol=0, atol=1e-12)
    # bf16 output is the single rounding of the FP64 rotation
    assert np.array_equal(oracle.rope_rotate(x, pos, THETA), oracle.f64_to_bf16(y))


def test_pair_norms_are_preserved():
    rng = np.random.default_rng(7)
    x = _rand_bf16(rng, D)
    xv = oracle.bf16_to_f64(x)
    y = oracle.rope_rotate_f64(x, 1234, THETA)
    assert np.allclose(y[:32] ** 2 + y[32:] ** 2, xv[:32] ** 2 + xv[32:] ** 2, rtol=1e-13)


def test_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(11)
    q = _rand_bf16(rng, D)
    k = _rand_bf16(rng, D)
    base = np.dot(oracle.rope_rotate_f64(q, 900, THETA), oracle.rope_rotate_f64(k, 880, THETA))
    for shift in (-880, -100, 3, 1000):
        s = np.dot(oracle.rope_rotate_f64(q, 900 + shift, THETA),
                   oracle.rope_rotate_f64(k, 880 + shift, THETA))
        assert math.isclose(s, base, rel_tol=1e-9, abs_tol=1e-9)
    # and it does depend on the offset itself
    other = np.dot(oracle.rope_rotate_f64(q, 900, THETA), oracle.rope_rotate_f64(k, 700, THETA))
    assert abs(other - base) > 1e-3
