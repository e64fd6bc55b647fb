"""Pins for the oracle's fused activation producer (``-m "not gpu"``).

``oracle.norm_quantize`` follows PRISM "E. Keeping preparation data close to
compute", Test 18: RMSNorm (with an optional residual add and a norm weight
stored as an offset from one), a random-sign Hadamard transform, and the
Test 6 group quantiser, all in fp32.  It is checked against things other than
itself:

* a scalar brute force in exact rationals that rounds every fp32 step
  explicitly (lane-sequential sum of squares and the halving lane sum, the
  correctly rounded square root found by exact squaring, a recursive
  Hadamard transform, the quantiser's division and ties-to-even rounding);
* integer inputs, where every fp32 sum is exact, against integer arithmetic
  and the Sylvester Hadamard matrix;
* closed forms (a constant row normalises to the norm weight), the fp64
  formula within the rounding bound, and the orthonormal transform keeping
  the row's 2-norm.

``test_norm_mutants_are_caught`` plants plausible mistakes in the oracle and
checks that at least one pin fails for each.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import pq_inputs
from oracle import pq_oracle as O
from test_oracle_pins import BF16, F16, F32, bits_value, rn

GROUP = 128
LANES = 2048


# --------------------------------------------------------------------------
# exact scalar brute force
# --------------------------------------------------------------------------

def f32(v: Fraction) -> Fraction:
    return rn(v, F32)


def _ulp32(r: Fraction) -> Fraction:
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return Fraction(2) ** (max(e, -126) - 23)


def sqrt_rn32(a: Fraction) -> Fraction:
    """Correctly rounded fp32 square root of a positive rational: the fp32
    value r with (r - ulp/2)^2 <= a < (r + ulp/2)^2 (exact squaring)."""
    r = f32(Fraction(float(np.sqrt(float(a)))))
    for _ in range(8):
        u = _ulp32(r)
        if (r + u / 2) ** 2 <= a:
            r += u
        elif (r - _ulp32(r - u / 2) / 2) ** 2 > a:
            r -= _ulp32(r - u / 2)
        else:
            return r
    raise AssertionError("square root search did not settle")


def _rint_even(v: Fraction) -> int:
    n = v.numerator // v.denominator
    rem = v - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2):
        n += 1
    return n


def _hadamard(x: list) -> list:
    if len(x) == 1:
        return x
    h = len(x) // 2
    a, b = _hadamard(x[:h]), _hadamard(x[h:])
    return [f32(p + q) for p, q in zip(a, b)] + [f32(p - q) for p, q in zip(a, b)]


def brute_norm_quantize(h_bits, r_bits, g_bits, fmt, eps, unit_offset, signs, B, AG):
    spec = BF16 if fmt == "bf16" else F16
    M, K = h_bits.shape
    eps32 = Fraction(float(np.float32(eps)))
    out = {"norm": [], "v": [], "q": [], "xs": [], "r_out": []}
    w = [bits_value(int(b), fmt) for b in g_bits]
    if unit_offset:
        w = [f32(x + 1) for x in w]
    for m in range(M):
        u = [bits_value(int(b), fmt) for b in h_bits[m]]
        if r_bits is not None:
            u = [f32(a + bits_value(int(b), fmt)) for a, b in zip(u, r_bits[m])]
            out["r_out"].append([rn(x, spec) for x in u])
        lanes = [Fraction(0)] * LANES
        for k in range(K):
            lanes[k % LANES] = f32(lanes[k % LANES] + f32(u[k] * u[k]))
        width = LANES
        while width > 1:
            width //= 2
            lanes = [f32(lanes[i] + lanes[i + width]) for i in range(width)]
        inv = f32(1 / sqrt_rn32(f32(f32(lanes[0] / K) + eps32)))
        n = [rn(f32(f32(u[k] * inv) * w[k]), spec) for k in range(K)]
        out["norm"].append(n)
        v = n
        if B:
            scale = f32(Fraction(1.0 / np.sqrt(float(B))))
            s = [(-x if sg < 0 else x) for x, sg in zip(n, signs)]
            v = []
            for b0 in range(0, K, B):
                v += [rn(f32(t * scale), spec) for t in _hadamard(s[b0:b0 + B])]
        out["v"].append(v)
        qrow, xsrow = [], []
        for g0 in range(0, K, AG):
            grp = v[g0:g0 + AG]
            sc = f32(max(abs(t) for t in grp) / 127)
            xsrow.append(sc)
            d = sc if sc > 0 else Fraction(1)
            qrow += [max(-127, min(127, _rint_even(f32(t / d)))) for t in grp]
        out["q"].append(qrow)
        out["xs"].append(xsrow)
    return out


def _values(bits, fmt):
    return [[bits_value(int(b), fmt) for b in row] for row in bits]


def check_brute(seed, fmt, K, residual, unit_offset, B, AG):
    d = pq_inputs.norm_inputs(seed, 2, K, fmt, unit_offset=unit_offset, residual=residual)
    eps = 1e-6
    got = O.norm_quantize(d["h"], d["r"], d["gamma"], fmt, eps, unit_offset, d["signs"], B, AG)
    ref = brute_norm_quantize(d["h"], d["r"], d["gamma"], fmt, eps, unit_offset, d["signs"], B, AG)
    assert _values(got["norm"], fmt) == ref["norm"]
    assert _values(got["v"], fmt) == ref["v"]
    if residual:
        assert _values(got["r_out"], fmt) == ref["r_out"]
    assert got["q"].astype(int).tolist() == ref["q"]
    assert [[Fraction(float(x)) for x in row] for row in got["xs"]] == ref["xs"]
    sq = np.asarray(ref["q"], dtype=np.int64).reshape(2, K // GROUP, GROUP).sum(axis=2)
    assert (got["sq"] == sq).all()


# --------------------------------------------------------------------------
# pins
# --------------------------------------------------------------------------

def pin_brute_small():
    check_brute(11, "bf16", 256, True, True, 128, 128)


def pin_brute_long_row():
    # K > 2048: lanes take more than one element, the last pass partly
    check_brute(12, "bf16", 2304, True, True, 256, 128)


def pin_brute_plain_norm():
    # fp16, no residual, plain weight, no transform, one group per row
    check_brute(13, "f16", 384, False, False, 0, 384)


def pin_sum_squares_integers():
    # |u| <= 64: every square and every partial sum is an exact fp32 integer
    r = np.random.default_rng(5)
    for K in (128, 640, 2048, 4096, 11008):
        u = r.integers(-64, 65, size=(3, K)).astype(np.float32)
        exact = (u.astype(np.int64) ** 2).sum(axis=1)
        assert (O.rms_sum_squares(u).astype(np.int64) == exact).all(), K


def pin_fwht_sylvester():
    sp = pytest.importorskip("scipy.linalg")
    r = np.random.default_rng(6)
    for B in (2, 8, 128, 1024):
        v = r.integers(-8, 9, size=(2, 2 * B)).astype(np.float32)
        H = sp.hadamard(B).astype(np.int64)
        want = np.concatenate([v[:, :B].astype(np.int64) @ H.T, v[:, B:].astype(np.int64) @ H.T], axis=1)
        assert (O.fwht_blocks(v, B).astype(np.int64) == want).all(), B


def pin_constant_row():
    # h = c (a power of two), tiny eps: mean(u^2) = c^2 exactly, inv = 1/|c|,
    # so the normalised row is sign(c) * w, rounded once
    K = 512
    for fmt, c in (("bf16", 0.5), ("bf16", -4.0), ("f16", 2.0)):
        to_bits = pq_inputs.f32_to_bf16_bits if fmt == "bf16" else pq_inputs.f32_to_f16_bits
        h = to_bits(np.full((1, K), c, dtype=np.float32))
        g = to_bits((np.random.default_rng(7).standard_normal(K) * 0.1).astype(np.float32))
        out = O.norm_quantize(h, None, g, fmt, 2.0 ** -40, True, None, 0, GROUP)
        w = [bits_value(int(b), fmt) + 1 for b in g]
        spec = BF16 if fmt == "bf16" else F16
        want = [rn(x if c > 0 else -x, spec) for x in w]
        assert _values(out["norm"], fmt)[0] == want


def pin_fp64_bound():
    # the fp32 chain stays within a few fp32 ulps of the fp64 formula, plus
    # the final rounding to bf16
    K = 4096
    d = pq_inputs.norm_inputs(8, 3, K, "bf16")
    eps = 1e-5
    out = O.norm_quantize(d["h"], d["r"], d["gamma"], "bf16", eps, True, None, 0, GROUP)
    u = O.bf16_bits_to_f64(d["h"]) + O.bf16_bits_to_f64(d["r"])
    w = O.bf16_bits_to_f64(d["gamma"]) + 1.0
    ref = u / np.sqrt((u * u).mean(axis=1, keepdims=True) + eps) * w
    got = O.bf16_bits_to_f64(out["norm"])
    tol = np.abs(ref) * (2.0 ** -8 + 64 * 2.0 ** -24) + 1e-30
    assert (np.abs(got - ref) <= tol).all()


def pin_transform_keeps_norm():
    # the orthonormal transform keeps each block's 2-norm (up to two bf16
    # roundings and the fp32 butterflies)
    K, B = 4096, 1024
    d = pq_inputs.norm_inputs(9, 2, K, "bf16")
    out = O.norm_quantize(d["h"], d["r"], d["gamma"], "bf16", 1e-6, True, d["signs"], B, GROUP)
    n = O.bf16_bits_to_f64(out["norm"]).reshape(2, K // B, B)
    v = O.bf16_bits_to_f64(out["v"]).reshape(2, K // B, B)
    ratio = np.linalg.norm(v, axis=2) / np.linalg.norm(n, axis=2)
    assert np.abs(ratio - 1).max() < 4e-3


ALL_NORM_PINS = [pin_brute_small, pin_brute_long_row, pin_brute_plain_norm, pin_sum_squares_integers,
                 pin_fwht_sylvester, pin_constant_row, pin_fp64_bound, pin_transform_keeps_norm]


@pytest.mark.parametrize("pin", ALL_NORM_PINS, ids=lambda f: f.__name__)
def test_norm_pin(pin):
    pin()


# --------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# --------------------------------------------------------------------------

_orig_sum = O.rms_sum_squares
_orig_inv = O.rms_inverse
_orig_fwht = O.fwht_blocks
_orig_norm = O.norm_quantize


def _mutant_sequential_sum(u):
    u = np.asarray(u, dtype=np.float32)
    acc = np.zeros(u.shape[0], dtype=np.float32)
    for k in range(u.shape[1]):
        acc = (acc + (u[:, k] * u[:, k]).astype(np.float32)).astype(np.float32)
    return acc


def _mutant_lanes_dropped(u):
    u = np.asarray(u, dtype=np.float32)
    return _orig_sum(u[:, :LANES])


def _mutant_mean_k_minus_1(total, K, eps):
    return _orig_inv(total, K - 1, eps)


def _mutant_eps_outside(total, K, eps):
    var = (np.asarray(total, dtype=np.float32) / np.float32(K)).astype(np.float32)
    return (np.float32(1) / (np.sqrt(var) + np.float32(eps))).astype(np.float32)


def _mutant_butterfly_swapped(v, B):
    w = _orig_fwht(v, B)
    M, K = w.shape
    return w.reshape(M, K // B, B)[:, :, ::-1].reshape(M, K)


def _mutant_unit_offset_dropped(h, r, g, fmt, eps, unit_offset, signs, B, AG):
    return _orig_norm(h, r, g, fmt, eps, False, signs, B, AG)


def _mutant_signs_ignored(h, r, g, fmt, eps, unit_offset, signs, B, AG):
    return _orig_norm(h, r, g, fmt, eps, unit_offset, None, B, AG)


def _mutant_residual_not_normalised(h, r, g, fmt, eps, unit_offset, signs, B, AG):
    out = _orig_norm(h, None, g, fmt, eps, unit_offset, signs, B, AG)
    if r is not None:
        out["r_out"] = _orig_norm(h, r, g, fmt, eps, unit_offset, signs, B, AG)["r_out"]
    return out


def _mutant_unnormalised_transform(h, r, g, fmt, eps, unit_offset, signs, B, AG):
    if not B:
        return _orig_norm(h, r, g, fmt, eps, unit_offset, signs, B, AG)
    out = _orig_norm(h, r, g, fmt, eps, unit_offset, signs, 0, AG)
    n = O.bits_to_f64(out["norm"], fmt).astype(np.float32)
    if signs is not None:
        n = np.where(np.asarray(signs)[None, :] < 0, -n, n).astype(np.float32)
    out["v"] = O.f64_to_bits(_orig_fwht(n, B).astype(np.float64), fmt)
    return out


NORM_MUTANTS = {
    "sum of squares in one sequential chain": ("rms_sum_squares", _mutant_sequential_sum),
    "only the first 2048 elements summed": ("rms_sum_squares", _mutant_lanes_dropped),
    "mean over K - 1": ("rms_inverse", _mutant_mean_k_minus_1),
    "eps added outside the square root": ("rms_inverse", _mutant_eps_outside),
    "butterfly outputs reversed": ("fwht_blocks", _mutant_butterfly_swapped),
    "norm weight without its unit offset": ("norm_quantize", _mutant_unit_offset_dropped),
    "random signs ignored": ("norm_quantize", _mutant_signs_ignored),
    "residual not added before the norm": ("norm_quantize", _mutant_residual_not_normalised),
    "transform not scaled by 1/sqrt(B)": ("norm_quantize", _mutant_unnormalised_transform),
}


@pytest.mark.parametrize("name", sorted(NORM_MUTANTS))
def test_norm_mutants_are_caught(name, monkeypatch):
    attr, fn = NORM_MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failures = 0
    for pin in ALL_NORM_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake: {name}"
