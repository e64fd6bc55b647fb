"""Pins for the oracle's MLX affine 4-bit format (``-m "not gpu"``).

``oracle.affine4_*`` follows "qwen CUDA: --prompt-precision int8 ... - #1176"
(TensorFold): 4-bit codes 0..15, one scale and one bias per 64-input group,
w = s * q + b.  It is checked against things other than itself:

* every nibble position and value of a packed word, decoded field by field;
* brute force in exact rationals on tiny layers with distinct scales and
  biases in every 64-group;
* the 4-bit GPTQ frame, itself pinned: with b = -8 s and one scale per 128
  rows the affine weights equal the symmetric GPTQ weights exactly;
* closed forms: all-zero codes leave the biases times the group sums of x.

``test_affine_mutants_are_caught`` plants plausible mistakes and checks that
at least one pin fails for each.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import pq_inputs
from oracle import pq_oracle as O
from test_oracle_pins import bits_value

G64 = 64


def _layer(seed, N, K, fmt):
    r = np.random.default_rng(seed)
    wq = r.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    to_bits = pq_inputs.f32_to_bf16_bits if fmt == "bf16" else pq_inputs.f32_to_f16_bits
    s = to_bits((0.001 + np.abs(r.standard_normal((N, K // G64)) * 0.01)).astype(np.float32))
    b = to_bits((r.standard_normal((N, K // G64)) * 0.05).astype(np.float32))
    return wq, s, b


def pin_every_nibble():
    for i in range(8):
        for v in range(16):
            wq = np.zeros((1, 2), dtype=np.uint32)
            wq[0, 1] = np.uint32(v << (4 * i))
            codes = O.affine4_codes(wq)
            want = np.zeros(16, dtype=np.uint8)
            want[8 + i] = v
            assert np.array_equal(codes[0], want), (i, v)


def pin_brute_force():
    for fmt, seed in (("bf16", 1), ("f16", 2)):
        N, K, M = 3, 128, 2
        wq, s, b = _layer(seed, N, K, fmt)
        x = pq_inputs.activations(seed + 10, M, K, "bf16")
        got = O.affine4_linear(x, "bf16", wq, s, b, fmt)
        for n in range(N):
            for m in range(M):
                acc = Fraction(0)
                mag = Fraction(0)
                for k in range(K):
                    word = int(wq[n, k // 8])
                    q = (word >> (4 * (k % 8))) & 0xF
                    g = k // G64
                    w = bits_value(int(s[n, g]), fmt) * q + bits_value(int(b[n, g]), fmt)
                    t = bits_value(int(x[m, k]), "bf16") * w
                    acc += t
                    mag += abs(t)
                # fp64 products are exact here; the fp64 sum is within K ulps
                assert abs(Fraction(float(got[m, n])) - acc) <= mag * K * Fraction(1, 2 ** 53), (fmt, n, m)


def pin_matches_gptq_frame():
    # b = -8 s and one scale per 128 rows: w = s (q - 8), the symmetric GPTQ weight
    N, K = 24, 512
    r = np.random.default_rng(3)
    wq = r.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    s128 = pq_inputs.f32_to_f16_bits((0.002 + np.abs(r.standard_normal((N, K // 128)) * 0.01)).astype(np.float32))
    s = np.repeat(s128, 2, axis=1)
    b = pq_inputs.f32_to_f16_bits((-8.0 * O.f16_bits_to_f64(s)).astype(np.float32))   # exact: times a power of two
    affine = O.affine4_dequant(wq, s, b, "f16")
    gptq = O.w4_dequant(np.ascontiguousarray(wq.T), np.ascontiguousarray(s128.T))
    assert np.array_equal(affine.T, gptq)


def pin_zero_codes():
    # q = 0: y = sum over groups of b times the group's sum of x (small
    # integers and powers of two keep every sum exact)
    N, K, M = 5, 256, 3
    r = np.random.default_rng(4)
    wq = np.zeros((N, K // 8), dtype=np.uint32)
    s = pq_inputs.f32_to_bf16_bits(np.ones((N, K // G64), dtype=np.float32))
    bv = (2.0 ** r.integers(-4, 4, size=(N, K // G64))).astype(np.float32)
    b = pq_inputs.f32_to_bf16_bits(bv)
    xv = r.integers(-8, 9, size=(M, K)).astype(np.float32)
    x = pq_inputs.f32_to_bf16_bits(xv)
    got = O.affine4_linear(x, "bf16", wq, s, b, "bf16")
    gs = xv.astype(np.float64).reshape(M, K // G64, G64).sum(axis=2)
    want = gs @ bv.astype(np.float64).T
    assert np.array_equal(got, want)


ALL_AFFINE_PINS = [pin_every_nibble, pin_brute_force, pin_matches_gptq_frame, pin_zero_codes]


@pytest.mark.parametrize("pin", ALL_AFFINE_PINS, ids=lambda f: f.__name__)
def test_affine_pin(pin):
    pin()


_orig_codes = O.affine4_codes
_orig_dequant = O.affine4_dequant


def _mutant_msb_first(wq):
    w = np.asarray(wq, dtype=np.uint32)
    codes = np.empty((w.shape[0], w.shape[1] * 8), dtype=np.uint8)
    for i in range(8):
        codes[:, i::8] = (w >> np.uint32(4 * (7 - i))) & np.uint32(0xF)
    return codes


def _mutant_group_128(wq, s, b, fmt):
    s = np.asarray(s)
    b = np.asarray(b)
    return _orig_dequant(wq, np.repeat(s[:, ::2], 2, axis=1), np.repeat(b[:, ::2], 2, axis=1), fmt)


def _mutant_bias_dropped(wq, s, b, fmt):
    return _orig_dequant(wq, s, np.zeros_like(np.asarray(b)), fmt)


def _mutant_bias_negated(wq, s, b, fmt):
    return _orig_dequant(wq, s, np.asarray(b) ^ np.uint16(0x8000), fmt)


def _mutant_centred_codes(wq, s, b, fmt):
    # w = s (q - 8) + b: a GPTQ habit applied to the affine frame
    w = _orig_dequant(wq, s, b, fmt)
    N, K = w.shape
    sv = O.bits_to_f64(np.asarray(s), fmt)[:, np.arange(K) // G64]
    return w - 8.0 * sv


AFFINE_MUTANTS = {
    "nibbles most significant first": ("affine4_codes", _mutant_msb_first),
    "one scale and bias per 128": ("affine4_dequant", _mutant_group_128),
    "bias dropped": ("affine4_dequant", _mutant_bias_dropped),
    "bias negated": ("affine4_dequant", _mutant_bias_negated),
    "codes centred at 8": ("affine4_dequant", _mutant_centred_codes),
}


@pytest.mark.parametrize("name", sorted(AFFINE_MUTANTS))
def test_affine_mutants_are_caught(name, monkeypatch):
    attr, fn = AFFINE_MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failures = 0
    for pin in ALL_AFFINE_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake: {name}"
