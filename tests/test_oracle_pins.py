"""Pins for the CPU oracle (``-m "not gpu"``).

The oracle is checked against things other than itself:

* hand-worked examples from the pages' statements (``tests/golden/*.txt``,
  each with its citation);
* every byte value, decoded through the three closed forms the PRISM page
  prints for PQ2 codes (per-code subtraction, add/XOR spread, byte-permute
  selector) and through every nibble position of a GPTQ word;
* brute force with exact rationals on tiny inputs, including an exact
  emulation of fp32 rounding for the activation quantiser and exact rounding
  of the outputs onto the fp16 / bf16 grids;
* the act-order invariant x[:,perm] @ W[perm] == x @ W (MATE "Act order"),
  the identity-g_idx special case, and the skipped-gather negative test;
* closed forms (zero weights, one-hot activations, constant activations) and
  the minus-one identity of PRISM Test 21.

``test_mutants_are_caught`` plants plausible mistakes in the oracle and
checks that at least one pin fails for each.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest

import pq_inputs
from oracle import pq_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GROUP = 128


# --------------------------------------------------------------------------
# exact helpers (independent of the oracle)
# --------------------------------------------------------------------------

def _exp2(e: int) -> Fraction:
    return Fraction(2) ** e


def round_fraction(v: Fraction, p: int, emin: int, fmax: Fraction | None) -> Fraction | float:
    """Exact round-to-nearest-even of a rational onto a binary grid with p
    significant bits and minimum normal exponent emin."""
    if v == 0:
        return Fraction(0)
    sign = 1 if v > 0 else -1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while _exp2(e) > a:
        e -= 1
    while _exp2(e + 1) <= a:
        e += 1
    e = max(e, emin)
    quantum = _exp2(e - p + 1)
    t = a / quantum
    n = t.numerator // t.denominator
    rem = t - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * quantum
    if fmax is not None and r > fmax:
        return sign * float("inf")
    return sign * r


F32 = (24, -126, None)
F16 = (11, -14, Fraction(65504))
BF16 = (8, -126, Fraction(0x1FE) * _exp2(127 - 8))


def rn(v: Fraction, fmt) -> Fraction:
    return round_fraction(v, *fmt)


def bits_value(bits: int, fmt: str) -> Fraction:
    """Exact value of a 16-bit pattern, decoded field by field."""
    sign = -1 if bits & 0x8000 else 1
    if fmt == "f16":
        e, m, ebits, mbits, bias = (bits >> 10) & 0x1F, bits & 0x3FF, 5, 10, 15
    else:
        e, m, ebits, mbits, bias = (bits >> 7) & 0xFF, bits & 0x7F, 8, 7, 127
    if e == (1 << ebits) - 1:
        raise ValueError("non-finite")
    if e == 0:
        return sign * Fraction(m) * _exp2(1 - bias - mbits)
    return sign * (Fraction(1) + Fraction(m, 1 << mbits)) * _exp2(e - bias)


def load_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                key, val = line.split(":", 1)
                out[key.strip()] = val.split()
            else:
                out.setdefault("_rows", []).append(line.split())
    return out


def expand_spec(tokens):
    """'1x128' -> 128 ones; 'a..b' -> range a..b inclusive."""
    out = []
    for t in tokens:
        if "x" in t:
            v, n = t.split("x")
            out += [int(v)] * int(n)
        elif ".." in t:
            a, b = t.split("..")
            out += list(range(int(a), int(b) + 1))
        else:
            out.append(int(t))
    return out


# --------------------------------------------------------------------------
# independent brute force (exact rationals, scalar loops)
# --------------------------------------------------------------------------

def brute_w4a16(x_bits, fmt, qweight, scales_bits, zeros, g_idx):
    M, K = x_bits.shape
    N = qweight.shape[1]
    xv = [[bits_value(int(x_bits[m, k]), fmt) for k in range(K)] for m in range(M)]
    y = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        for k in range(K):
            word = int(qweight[k // 8, n])
            code = (word >> (4 * (k % 8))) & 0xF
            g = int(g_idx[k]) if g_idx is not None else k // GROUP
            z = 8 if zeros is None else int(zeros[g, n])
            s = bits_value(int(scales_bits[g, n]), "f16")
            w = (code - z) * s
            for m in range(M):
                y[m][n] += xv[m][k] * w
    return y


def brute_quantize(x_bits, fmt, group):
    """fp32 quantiser emulated exactly: every fp32 operation is the exact
    rational result rounded to nearest even on the fp32 grid."""
    M, K = x_bits.shape
    q = [[0] * K for _ in range(M)]
    scales = [[Fraction(0)] * (K // group) for _ in range(M)]
    for m in range(M):
        for gi in range(K // group):
            vals = [bits_value(int(x_bits[m, gi * group + i]), fmt) for i in range(group)]
            amax = max(abs(v) for v in vals)
            scale = rn(amax / 127, F32)
            scales[m][gi] = scale
            div = scale if scale > 0 else Fraction(1)
            for i, v in enumerate(vals):
                t = rn(v / div, F32)
                n = t.numerator // t.denominator
                rem = t - n
                if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
                    n += 1
                q[m][gi * group + i] = max(-127, min(127, n))
    return q, scales


def brute_w2a8(x_bits, fmt, raw, act_group):
    M, K = x_bits.shape
    N = raw.shape[0]
    B = K // GROUP
    q, xs = brute_quantize(x_bits, fmt, act_group)
    S = [[[0] * B for _ in range(N)] for _ in range(M)]
    y = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        for b in range(B):
            blk = raw[n, 34 * b: 34 * b + 34]
            ws = bits_value(int(blk[0]) | (int(blk[1]) << 8), "f16")
            for m in range(M):
                acc = 0
                for i in range(32):
                    byte = int(blk[2 + i])
                    for j in range(4):
                        k = GROUP * b + 4 * i + j
                        acc += (((byte >> (2 * j)) & 3) - 1) * q[m][k]
                S[m][n][b] = acc
                y[m][n] += acc * xs[m][(GROUP * b) // act_group] * ws
    return q, xs, S, y


# --------------------------------------------------------------------------
# pins (plain functions so the mutation test can run them too)
# --------------------------------------------------------------------------

def check_pq2_code_golden():
    table = {int(r[0]): int(r[1]) for r in load_golden("pq2_code_values.txt")["_rows"]}
    # one block: byte i = code (i % 4) repeated in all four fields
    raw = np.zeros((1, 34), dtype=np.uint8)
    for i in range(32):
        c = i % 4
        raw[0, 2 + i] = c | (c << 2) | (c << 4) | (c << 6)
    v = O.pq2_values(raw)[0]
    for k in range(128):
        assert v[k] == table[(k // 4) % 4], (k, v[k])


def check_pq2_block_golden():
    g = load_golden("pq2_block_example.txt")
    raw = np.array([[int(b, 16) for b in g["block"]]], dtype=np.uint8)
    v = O.pq2_values(raw)[0]
    head = [int(t) for t in g["values"]]
    assert list(v[: len(head)]) == head
    assert all(int(t) == int(g["values_rest"][0]) for t in v[len(head):])
    assert O.pq2_scales(raw)[0, 0] == float(g["scale"][0])
    w = O.pq2_dequant(raw)[0]
    assert list(w[:8]) == [-0.5, 0, 0.5, 1, 1, 0.5, 0, -0.5]
    assert all(w[12:] == 0.5)


def _slow_expand(byte):       # PRISM Test 1 SLOW path: subtract one per code
    return [((byte >> (2 * j)) & 3) - 1 for j in range(4)]


def _fast_expand(byte):       # PRISM Test 1 FAST path: spread, +0x7F7F7F7F, ^0x80808080
    spread = (byte & 3) | ((byte << 6) & 0x300) | ((byte << 12) & 0x30000) | ((byte << 18) & 0x3000000)
    word = ((spread + 0x7F7F7F7F) & 0xFFFFFFFF) ^ 0x80808080
    return [((word >> (8 * j)) & 0xFF) - (256 if (word >> (8 * j)) & 0x80 else 0) for j in range(4)]


def _prmt_expand(byte):       # PRISM Test 10: byte_perm(0x020100ff, 0x020100ff, selector)
    src = [0xFF, 0x00, 0x01, 0x02, 0xFF, 0x00, 0x01, 0x02]
    out = []
    for j in range(4):
        b = src[(byte >> (2 * j)) & 3]
        out.append(b - 256 if b & 0x80 else b)
    return out


def check_pq2_all_bytes():
    raw = np.zeros((1, 34 * 8), dtype=np.uint8)
    vals = list(range(256))
    for i, b in enumerate(vals):
        blk, off = divmod(i, 32)
        raw[0, 34 * blk + 2 + off] = b
    v = O.pq2_values(raw)[0]
    for i, b in enumerate(vals):
        got = list(v[4 * i: 4 * i + 4])
        assert got == _slow_expand(b) == _fast_expand(b) == _prmt_expand(b), (b, got)


def check_pq2_scale_bytes():
    # little-endian fp16 at block offset 0, every exponent/mantissa byte pair
    # that is finite: compare with the field-by-field decode
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 0x7C00, size=64).astype(np.uint16)
    raw = np.zeros((1, 34 * 64), dtype=np.uint8)
    for b, s in enumerate(bits):
        raw[0, 34 * b] = int(s) & 0xFF
        raw[0, 34 * b + 1] = int(s) >> 8
    got = O.pq2_scales(raw)[0]
    for b, s in enumerate(bits):
        assert Fraction(float(got[b])) == bits_value(int(s), "f16")


def check_w4_word_golden():
    g = load_golden("w4_word_example.txt")
    words = np.array([[int(w, 16)] for w in g["words"]], dtype=np.uint32)  # [2][1]
    # K must be a multiple of 8 for unpacking; K=16 here
    codes = O.w4_codes(words)[:, 0]
    assert list(codes) == [int(c) for c in g["codes"]]
    qweight = np.zeros((16, 1), dtype=np.uint32)
    qweight[:2] = words
    scales = np.full((1, 1), int(g["scale_bits"][0], 16), dtype=np.uint16)
    w = O.w4_dequant(qweight, scales)[:16, 0]
    assert list(w) == [float(t) for t in g["dequant_sym"]]


def check_w4_every_nibble():
    # every value at every nibble position, and every byte at every byte position
    for pos in range(8):
        for val in range(16):
            word = np.array([[val << (4 * pos)]], dtype=np.uint32)
            codes = O.w4_codes(word)[:, 0]
            expect = [0] * 8
            expect[pos] = val
            assert list(codes) == expect
    for bpos in range(4):
        for b in range(256):
            word = np.array([[b << (8 * bpos)]], dtype=np.uint32)
            codes = O.w4_codes(word)[:, 0]
            expect = [0] * 8
            expect[2 * bpos] = b & 0xF
            expect[2 * bpos + 1] = b >> 4
            assert list(codes) == expect


def check_quantize_golden():
    g = load_golden("quantize_example.txt")
    for case in ("1", "2", "3"):
        x = np.array([float(t) for t in g["x" + case]], dtype=np.float32)[None, :]
        bits = pq_inputs.f32_to_bf16_bits(x)
        q, s = O.quantize_act(bits, "bf16", 8)
        assert list(q[0]) == [int(t) for t in g["q" + case]], (case, q)
        assert float(s[0, 0]) == float(g["scale" + case][0])


def check_act_order_golden():
    g = load_golden("act_order_example.txt")
    g_idx = np.array(expand_spec(g["g_idx"]), dtype=np.int32)
    perm = O.act_order_perm(g_idx, 256)
    assert list(perm) == expand_spec(g["perm"])
    bad = np.array(expand_spec(g["refuse_g_idx"]), dtype=np.int32)
    with pytest.raises(ValueError, match="contiguous run"):
        O.act_order_perm(bad, 256)


def _close_to_exact(y64, exact, M, N, terms_abs):
    for m in range(M):
        for n in range(N):
            err = abs(Fraction(float(y64[m, n])) - exact[m][n])
            assert err <= Fraction(1, 10 ** 12) * (terms_abs[m][n] + Fraction(1, 10 ** 30)), (m, n)


def check_w4_brute(zero_points: bool, act_order, fmt: str, seed: int):
    K, N, M = 256, 5, 3
    fr = pq_inputs.w4_frame(seed, K, N, 0.002, 0.01, zero_points, act_order)
    x = pq_inputs.activations(seed + 100, M, K, fmt)
    exact = brute_w4a16(x, fmt, fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    y64 = O.w4a16_linear(x, fmt, fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    xa = np.abs(O.bits_to_f64(x, fmt))
    Wa = np.abs(O.w4_dequant(fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"]))
    terms = xa @ Wa
    _close_to_exact(y64, exact, M, N, [[Fraction(float(terms[m, n])) for n in range(N)] for m in range(M)])
    out = O.f64_to_bits(y64, fmt)
    fmt_t = F16 if fmt == "f16" else BF16
    for m in range(M):
        for n in range(N):
            assert bits_value(int(out[m, n]), fmt) == rn(exact[m][n], fmt_t), (m, n)


def check_w2a8_brute(act_group: int, fmt: str, seed: int, allow_code3: bool):
    K, N, M = 256, 4, 2
    raw = pq_inputs.pq2_rows(seed, N, K, allow_code3=allow_code3)
    x = pq_inputs.activations(seed + 7, M, K, fmt)
    q_b, xs_b, S_b, y_b = brute_w2a8(x, fmt, raw, act_group)
    q, xs = O.quantize_act(x, fmt, act_group)
    assert q.tolist() == q_b
    for m in range(M):
        for gi in range(K // act_group):
            assert Fraction(float(xs[m, gi])) == xs_b[m][gi]
    S = O.w2a8_group_sums(q, O.pq2_values(raw))
    assert S.tolist() == S_b
    y64 = O.w2a8_linear(x, fmt, raw, act_group)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(float(y64[m, n])) - y_b[m][n]) <= Fraction(1, 10 ** 12) * (abs(y_b[m][n]) + 1)


def check_act_order_invariant(seed: int):
    K, N, M = 256, 3, 2
    fr = pq_inputs.w4_frame(seed, K, N, 0.002, 0.01, True, "scatter")
    x = pq_inputs.activations(seed + 1, M, K, "bf16")
    perm = O.act_order_perm(fr["g_idx"], K)
    W = O.w4_dequant(fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    xv = O.bits_to_f64(x, "bf16")
    # exact: every term is exact in fp64, sum in exact rationals both ways
    for m in range(M):
        for n in range(N):
            a = sum(Fraction(float(xv[m, k])) * Fraction(float(W[k, n])) for k in range(K))
            b = sum(Fraction(float(xv[m, perm[i]])) * Fraction(float(W[perm[i], n])) for i in range(K))
            assert a == b
    # the gather matters: dropping it changes the result by a large margin
    y = xv @ W
    y_skip = xv @ W[perm]
    assert np.abs(y_skip - y).max() > 100 * 1e-12 * np.abs(y).max()
    y_gather = xv[:, perm] @ W[perm]
    assert np.allclose(y_gather, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def check_identity_g_idx(seed: int):
    K, N, M = 512, 8, 2
    fr = pq_inputs.w4_frame(seed, K, N, 0.002, 0.01, True, None)
    x = pq_inputs.activations(seed + 3, M, K, "bf16")
    ident = (np.arange(K) // GROUP).astype(np.int32)
    a = O.w4a16_linear(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], None)
    b = O.w4a16_linear(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], ident)
    assert np.array_equal(a, b)
    assert np.array_equal(O.act_order_perm(ident, K), np.arange(K))


def check_closed_forms():
    K, N = 256, 6
    # symmetric frame with every code 8 dequantises to zero weights
    qweight = np.full((K // 8, N), 0x88888888, dtype=np.uint32)
    fr = pq_inputs.w4_frame(1, K, N, 0.002, 0.01)
    x = pq_inputs.activations(2, 2, K, "f16")
    assert not O.w4a16_linear(x, "f16", qweight, fr["scales"]).any()
    # one-hot activation picks one dequantised row: y = RN(w(k, .))
    for k in (0, 7, 8, 129, 255):
        xb = np.zeros((1, K), dtype=np.uint16)
        xb[0, k] = 0x3C00                       # fp16 1.0
        y = O.f64_to_bits(O.w4a16_linear(xb, "f16", fr["qweight"], fr["scales"]), "f16")
        codes = [(int(fr["qweight"][k // 8, n]) >> (4 * (k % 8))) & 15 for n in range(N)]
        w = [(c - 8) * bits_value(int(fr["scales"][k // GROUP, n]), "f16") for n, c in enumerate(codes)]
        assert [bits_value(int(b), "f16") for b in y[0]] == [rn(v, F16) for v in w]
    # constant activation: every code is 127 and S = 127 * sum(v)
    raw = pq_inputs.pq2_rows(3, 4, K)
    xb = np.full((1, K), 0x3F80, dtype=np.uint16)   # bf16 1.0
    q, xs = O.quantize_act(xb, "bf16", K)
    assert (q == 127).all()
    S = O.w2a8_group_sums(q, O.pq2_values(raw))
    v = O.pq2_values(raw).reshape(4, K // GROUP, GROUP).sum(axis=2)
    assert np.array_equal(S[0], 127 * v)


def check_minus_one_identity(seed: int):
    K, N, M = 384, 5, 3
    raw = pq_inputs.pq2_rows(seed, N, K, allow_code3=True)
    x = pq_inputs.activations(seed, M, K, "bf16")
    q, _ = O.quantize_act(x, "bf16", GROUP)
    S = O.w2a8_group_sums(q, O.pq2_values(raw))
    c = O.pq2_codes(raw).astype(np.int64)
    qb = q.astype(np.int64).reshape(M, K // GROUP, GROUP)
    cq = np.einsum("mbk,nbk->mnb", qb, c.reshape(N, K // GROUP, GROUP))
    sq = qb.sum(axis=2)[:, None, :]
    assert np.array_equal(S, cq - sq)


def check_row_independence(seed: int):
    K, N = 256, 4
    fr = pq_inputs.w4_frame(seed, K, N, 0.002, 0.01, True, "scatter")
    raw = pq_inputs.pq2_rows(seed, N, K)
    x = pq_inputs.activations(seed, 2, K, "bf16")
    x2 = x.copy()
    x2[1] = pq_inputs.activations(seed + 9, 1, K, "bf16")[0]
    a = O.w4a16_linear(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    b = O.w4a16_linear(x2, "bf16", fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    assert np.array_equal(a[0], b[0]) and not np.array_equal(a[1], b[1])
    a = O.w2a8_linear(x, "bf16", raw, GROUP)
    b = O.w2a8_linear(x2, "bf16", raw, GROUP)
    assert np.array_equal(a[0], b[0]) and not np.array_equal(a[1], b[1])


def check_rounding(seed: int):
    rng = np.random.default_rng(seed)
    y = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 6, 4000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]),
    ])
    # fp16: numpy's IEEE double -> half conversion
    with np.errstate(over="ignore"):
        ref16 = y.astype(np.float16).view(np.uint16)
    assert np.array_equal(O.f64_to_bits(y, "f16"), ref16)
    # bf16 on fp32-representable values: the integer round-half-even bit trick
    y32 = y.astype(np.float32)
    u = y32.view(np.uint32).astype(np.uint64)
    trick = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(O.f64_to_bits(y32.astype(np.float64), "bf16"), trick)
    # exact rational rounding on doubles that are not fp32-representable
    for v in rng.standard_normal(300) * 3.0:
        for fmt, t in (("f16", F16), ("bf16", BF16)):
            got = O.round_f64(np.array([v]), fmt)[0]
            assert Fraction(float(got)) == rn(Fraction(float(v)), t)


def check_w4_columns(seed: int):
    """The sampled-column helper against the exact brute force of the whole
    layer, picked column by column (zero points and act order on; columns
    unsorted, not contiguous, one repeated)."""
    K, N, M = 256, 9, 2
    fr = pq_inputs.w4_frame(seed, K, N, 0.002, 0.01, True, "scatter")
    x = pq_inputs.activations(seed + 5, M, K, "bf16")
    cols = np.array([7, 2, 5, 2, 0, 8])
    exact = brute_w4a16(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    got = O.w4a16_linear_columns(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"], cols)
    assert got.shape == (M, len(cols))
    xa = np.abs(O.bits_to_f64(x, "bf16"))
    Wa = np.abs(O.w4_dequant(fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"]))
    terms = xa @ Wa
    _close_to_exact(got, [[exact[m][c] for c in cols] for m in range(M)], M, len(cols),
                    [[Fraction(float(terms[m, c])) for c in cols] for m in range(M)])


def check_w2_rows(seed: int):
    """The sampled-row helper of the ternary layer against the exact brute
    force of the whole layer, picked row by row (rows unsorted, one repeated)."""
    K, N, M = 256, 6, 2
    raw = pq_inputs.pq2_rows(seed, N, K, allow_code3=True)
    x = pq_inputs.activations(seed + 3, M, K, "bf16")
    rows = np.array([4, 1, 5, 1])
    _, _, _, y_b = brute_w2a8(x, "bf16", raw, 128)
    got = O.w2a8_linear_columns(x, "bf16", raw, 128, rows)
    assert got.shape == (M, len(rows))
    for m in range(M):
        for j, n in enumerate(rows):
            assert abs(Fraction(float(got[m, j])) - y_b[m][n]) <= Fraction(1, 10 ** 12) * (abs(y_b[m][n]) + 1)


ALL_PINS = [
    check_pq2_code_golden, check_pq2_block_golden, check_pq2_all_bytes, check_pq2_scale_bytes,
    check_w4_word_golden, check_w4_every_nibble, check_quantize_golden, check_act_order_golden,
    lambda: check_w4_brute(False, None, "f16", 11),
    lambda: check_w4_brute(True, None, "bf16", 12),
    lambda: check_w4_brute(True, "scatter", "bf16", 13),
    lambda: check_w4_brute(False, "blocks", "bf16", 14),
    lambda: check_w2a8_brute(256, "bf16", 21, False),
    lambda: check_w2a8_brute(128, "bf16", 22, True),
    lambda: check_w2a8_brute(128, "f16", 23, False),
    lambda: check_act_order_invariant(31), lambda: check_identity_g_idx(32),
    check_closed_forms, lambda: check_minus_one_identity(41), lambda: check_row_independence(42),
    lambda: check_rounding(51),
    lambda: check_w4_columns(61), lambda: check_w2_rows(62),
]


# --------------------------------------------------------------------------
# tests
# --------------------------------------------------------------------------

def test_pq2_code_golden():
    check_pq2_code_golden()


def test_pq2_block_golden():
    check_pq2_block_golden()


def test_pq2_all_byte_values_three_closed_forms():
    check_pq2_all_bytes()


def test_pq2_scale_bytes():
    check_pq2_scale_bytes()


def test_w4_word_golden():
    check_w4_word_golden()


def test_w4_every_nibble_and_byte():
    check_w4_every_nibble()


def test_quantize_golden():
    check_quantize_golden()


def test_act_order_golden_and_refusal():
    check_act_order_golden()


@pytest.mark.parametrize("zp,act,fmt,seed", [
    (False, None, "f16", 11), (True, None, "bf16", 12),
    (True, "scatter", "bf16", 13), (False, "blocks", "bf16", 14), (True, "scatter", "f16", 15)])
def test_w4a16_brute_force_exact(zp, act, fmt, seed):
    check_w4_brute(zp, act, fmt, seed)


@pytest.mark.parametrize("ag,fmt,seed,code3", [
    (256, "bf16", 21, False), (128, "bf16", 22, True), (128, "f16", 23, False), (256, "f16", 24, True)])
def test_w2a8_brute_force_exact(ag, fmt, seed, code3):
    check_w2a8_brute(ag, fmt, seed, code3)


def test_act_order_invariant_and_skipped_gather():
    check_act_order_invariant(31)


def test_identity_g_idx_matches_plain_groups():
    check_identity_g_idx(32)


def test_closed_forms():
    check_closed_forms()


def test_minus_one_identity():
    check_minus_one_identity(41)


def test_row_independence():
    check_row_independence(42)


def test_output_rounding():
    check_rounding(51)


def test_w4_sampled_columns_match_brute_force():
    check_w4_columns(61)


def test_w2_sampled_rows_match_brute_force():
    check_w2_rows(62)


def test_act_order_refusals():
    K = 256
    with pytest.raises(ValueError, match="must lie in"):
        O.act_order_perm(np.full(K, 2, dtype=np.int32), K)
    with pytest.raises(ValueError, match="K=256 entries"):
        O.act_order_perm(np.zeros(K - 1, dtype=np.int32), K)


def test_act_order_fp64_large():
    # fp64 sums in two orders agree within the fp64 error bound at K=5120
    K, N, M = 5120, 64, 4
    fr = pq_inputs.w4_frame(77, K, N, 0.001, 0.01, True, "scatter")
    x = O.bits_to_f64(pq_inputs.activations(78, M, K, "bf16"), "bf16")
    W = O.w4_dequant(fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    perm = O.act_order_perm(fr["g_idx"], K)
    bound = 4 * K * 2.0 ** -53 * (np.abs(x) @ np.abs(W))
    assert (np.abs(x[:, perm] @ W[perm] - x @ W) <= bound).all()


# --------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# --------------------------------------------------------------------------

def _mutant_nibble_msb_first(qweight):
    qw = np.asarray(qweight, dtype=np.uint32)
    codes = np.empty((qw.shape[0] * 8, qw.shape[1]), dtype=np.uint8)
    for i in range(8):
        codes[i::8, :] = (qw >> np.uint32(4 * (7 - i))) & np.uint32(0xF)
    return codes


def _mutant_zero_seven(G, N, zeros):
    return np.full((G, N), 7, dtype=np.int64) if zeros is None else np.asarray(zeros, np.int64)


def _mutant_zero_plus_one(G, N, zeros):
    return np.full((G, N), 8, dtype=np.int64) if zeros is None else np.asarray(zeros, np.int64) + 1


def _mutant_canonical_groups(K, g_idx):
    return np.arange(K, dtype=np.int64) // GROUP


_orig_codes = O.pq2_codes
_orig_quant = O.quantize_act
_orig_sums = O.w2a8_group_sums
_orig_perm = O.act_order_perm
_orig_scales = O.pq2_scales
_orig_w4_columns = O.w4a16_linear_columns


def _mutant_no_minus_one(raw):
    return _orig_codes(raw).astype(np.int64)


def _mutant_pairs_reversed(raw):
    blocks = O.pq2_blocks(raw)
    N, B, _ = blocks.shape
    cb = blocks[:, :, 2:].astype(np.int64)
    c = np.empty((N, B, 32, 4), dtype=np.int64)
    for j in range(4):
        c[:, :, :, j] = (cb >> (6 - 2 * j)) & 3
    return c.reshape(N, B * GROUP).astype(np.uint8)


def _mutant_scale_big_endian(raw):
    blocks = O.pq2_blocks(raw)
    hi = blocks[:, :, 0].astype(np.uint16)
    lo = blocks[:, :, 1].astype(np.uint16)
    return O.f16_bits_to_f64(lo | (hi << 8))


def _mutant_round_half_up(x_bits, fmt, group):
    x = O.bits_to_f64(x_bits, fmt).astype(np.float32)
    M, K = x.shape
    a = x.reshape(M, K // group, group)
    scale = (np.abs(a).max(axis=2) / np.float32(127)).astype(np.float32)
    d = np.where(scale > 0, scale, np.float32(1)).astype(np.float32)
    q = np.clip(np.floor(a / d[:, :, None] + 0.5), -127, 127).astype(np.int8)
    return q.reshape(M, K), scale


def _mutant_scale_128(x_bits, fmt, group):
    x = O.bits_to_f64(x_bits, fmt).astype(np.float32)
    M, K = x.shape
    a = x.reshape(M, K // group, group)
    scale = (np.abs(a).max(axis=2) / np.float32(128)).astype(np.float32)
    d = np.where(scale > 0, scale, np.float32(1)).astype(np.float32)
    q = np.clip(np.rint(a / d[:, :, None]), -127, 127).astype(np.int8)
    return q.reshape(M, K), scale


def _mutant_blocks_shifted(q, v):
    S = _orig_sums(q, v)
    return np.roll(S, 1, axis=2)


def _mutant_perm_reverse(g_idx, K):
    g = np.asarray(g_idx, dtype=np.int64)
    if g.shape != (K,):
        raise ValueError(f"g_idx must have K={K} entries, got {g.shape}")
    counts = np.bincount(g, minlength=K // GROUP)
    if (counts != GROUP).any():
        raise ValueError("every sorted group must be one contiguous run")
    return np.argsort(-g, kind="stable")


def _mutant_columns_sorted(x_bits, act_fmt, qweight, scales_bits, zeros, g_idx, cols):
    return _orig_w4_columns(x_bits, act_fmt, qweight, scales_bits, zeros, g_idx, np.sort(cols))


def _mutant_columns_zeros_unsliced(x_bits, act_fmt, qweight, scales_bits, zeros, g_idx, cols):
    cols = np.asarray(cols, dtype=np.int64)
    zsel = None if zeros is None else np.asarray(zeros)[:, :len(cols)]
    W = O.w4_dequant(np.asarray(qweight)[:, cols], np.asarray(scales_bits)[:, cols], zsel, g_idx)
    return O.bits_to_f64(x_bits, act_fmt) @ W


def _mutant_rows_ignored(x_bits, act_fmt, raw, act_group, rows):
    return O.w2a8_linear(x_bits, act_fmt, np.asarray(raw)[:len(rows)], act_group)


MUTANTS = {
    "nibble order MSB first": ("w4_codes", _mutant_nibble_msb_first),
    "symmetric zero point 7": ("w4_zero_points", _mutant_zero_seven),
    "explicit zero point +1": ("w4_zero_points", _mutant_zero_plus_one),
    "scale by k//128 under act order": ("w4_groups", _mutant_canonical_groups),
    "ternary value = code": ("pq2_values", _mutant_no_minus_one),
    "2-bit fields reversed": ("pq2_codes", _mutant_pairs_reversed),
    "scale bytes big-endian": ("pq2_scales", _mutant_scale_big_endian),
    "round half up": ("quantize_act", _mutant_round_half_up),
    "scale amax/128": ("quantize_act", _mutant_scale_128),
    "block sums shifted": ("w2a8_group_sums", _mutant_blocks_shifted),
    "act-order perm reversed": ("act_order_perm", _mutant_perm_reverse),
    "sampled columns sorted": ("w4a16_linear_columns", _mutant_columns_sorted),
    "sampled columns' zero points unsliced": ("w4a16_linear_columns", _mutant_columns_zeros_unsliced),
    "sampled rows ignored": ("w2a8_linear_columns", _mutant_rows_ignored),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failures = 0
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake: {name}"
