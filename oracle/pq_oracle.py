"""CPU oracle for the weight-only-quantized linear layer.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain reference the CUDA
library is checked against.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the library never calls it and has
no CPU fallback.  It shares no code, tables or constants with the CUDA path.

Sources (page title, then section):

* [PRISM] "Kernel experiments: recorded evidence" (anthonymorley.com, PRISM
  kernel experiments): ternary PQ2 blocks and their prepared planes (Test 1,
  Diagram 1), byte expansion (Test 1 code), group quantiser (Test 6 code),
  CPU fp64 replay (Test 8), plane order and minus-one correction (Test 21).
* [MATE] "mate: Marlin-class W4A16 GEMM for mp_31 (SQMMA int4 x fp16) - #6":
  GPTQ frame, act order resolution and the invariant x[:,perm]@W[perm]==x@W,
  SCALE[g_idx[k]] dequantisation, explicit zero-point convention (PR
  description, "Act order" and "Two defects" sections).
* [TensorFold] "qwen CUDA: --prompt-precision int8 ... - #1176": amax/127 fp32
  activation scale with nearest-even rounding.

Floating point: dequantised weights and dot products are formed in fp64 (the
PRISM Test 8 replay holds fp64 accumulation fixed).  The activation quantiser
is fp32 because the pages fix it in fp32: scale = max|a| / 127 and a
correctly rounded a / scale, ties to even (PRISM Test 6).

Readings where the pages are silent (also listed in the design notes):

* nibble order inside a GPTQ word: code i of word (k // 8) is bits 4i..4i+3,
  least significant first, for row k = 8 * (k // 8) + i;
* 4-bit dequantisation w = (code - z) * s with z = 8 when symmetric and the
  explicit uint8 zero point otherwise, no +1 offset;
* PQ2 code 3 maps to +2 (value = code - 1 for every code, PRISM Test 1);
* activation scale is the correctly rounded fp32 quotient max|a| / 127;
* an all-zero activation group has scale 0 and all codes 0;
* outputs are the fp64 result rounded once, to nearest even, to fp16 / bf16.

Every function here is pinned by the ``-m "not gpu"`` tests (brute force with
exact rationals, all byte values, closed forms and the act-order invariant).
"""
from __future__ import annotations

import numpy as np

GROUP = 128  # weights per scale group along K (all pages use 128)
PQ2_BLOCK_BYTES = 34  # 2-byte fp16 scale + 32 code bytes per 128 weights [PRISM Test 1]


# --------------------------------------------------------------------------
# fp16 / bf16 <-> fp64
# --------------------------------------------------------------------------

def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of an IEEE binary32; widening is exact."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def bits_to_f64(bits: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == "f16":
        return f16_bits_to_f64(bits)
    if fmt == "bf16":
        return bf16_bits_to_f64(bits)
    raise ValueError(fmt)


_FORMATS = {
    # significand bits (with the hidden bit), minimum normal exponent, max finite
    "f16": (11, -14, 65504.0),
    "bf16": (8, -126, float.fromhex("0x1.fep127")),
}


def round_f64(y: np.ndarray, fmt: str) -> np.ndarray:
    """Round fp64 values once, to nearest even, onto the fp16 / bf16 grid.

    For |y| in [2^e, 2^(e+1)) the grid spacing is 2^(e - p + 1); below the
    smallest normal it is the subnormal spacing.  Values beyond the largest
    finite number that round up become +-inf (IEEE overflow rule).
    """
    p, emin, fmax = _FORMATS[fmt]
    y = np.asarray(y, dtype=np.float64)
    out = np.empty_like(y)
    finite = np.isfinite(y)
    out[~finite] = y[~finite]
    v = y[finite]
    _, e = np.frexp(v)                     # v = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e - 1, emin)            # exponent of the leading bit, clamped
    quantum = np.ldexp(1.0, e - (p - 1))
    r = np.rint(v / quantum) * quantum     # exact scaling by a power of two; rint ties to even
    # a value that rounds past the largest finite number overflows to +-inf
    r = np.where(np.abs(r) > fmax, np.copysign(np.inf, v), r)
    out[finite] = r
    return out


def f64_to_bits(y: np.ndarray, fmt: str) -> np.ndarray:
    """Round (as ``round_f64``) and return the 16-bit pattern."""
    r = round_f64(y, fmt)
    if fmt == "f16":
        return r.astype(np.float16).view(np.uint16)   # exact: r is on the grid
    u = r.astype(np.float32).view(np.uint32)          # exact: bf16 grid is in fp32
    return (u >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# 4-bit GPTQ frame  [MATE PR description; GPTQ words packed 8 per uint32 along K]
# --------------------------------------------------------------------------

def w4_codes(qweight: np.ndarray) -> np.ndarray:
    """Codes [K][N] (0..15) from qweight [K/8][N]: code(k, n) is the 4-bit
    field at bits 4*(k % 8) of word (k // 8, n)."""
    qw = np.asarray(qweight, dtype=np.uint32)
    K = qw.shape[0] * 8
    codes = np.empty((K, qw.shape[1]), dtype=np.uint8)
    for i in range(8):
        codes[i::8, :] = (qw >> np.uint32(4 * i)) & np.uint32(0xF)
    return codes


def w4_zero_points(G: int, N: int, zeros: np.ndarray | None) -> np.ndarray:
    """Zero point z(g, n): 8 for the symmetric frame, else the explicit uint8
    value as given (MATE "Two defects": the caller names the convention)."""
    if zeros is None:
        return np.full((G, N), 8, dtype=np.int64)
    z = np.asarray(zeros, dtype=np.int64)
    if z.shape != (G, N):
        raise ValueError(f"zero points must be [{G}][{N}], got {z.shape}")
    if z.min(initial=0) < 0 or z.max(initial=0) > 15:
        raise ValueError("explicit zero points must lie in 0..15")
    return z


def w4_groups(K: int, g_idx: np.ndarray | None) -> np.ndarray:
    """Group of each row k: g_idx[k] under act order, else k // 128.  The
    act-order reference must use SCALE[g_idx[k]], never SCALE[k // group]
    (MATE "Act order")."""
    if g_idx is None:
        return np.arange(K, dtype=np.int64) // GROUP
    return np.asarray(g_idx, dtype=np.int64)


def w4_dequant(qweight: np.ndarray, scales_bits: np.ndarray,
               zeros: np.ndarray | None = None,
               g_idx: np.ndarray | None = None) -> np.ndarray:
    """Dequantised weights W[K][N] in fp64: w(k,n) = (code - z(g,n)) * s(g,n)
    with g the group of row k.  (code - z) * s is exact in fp64."""
    codes = w4_codes(qweight).astype(np.int64)
    K, N = codes.shape
    G = K // GROUP
    s = f16_bits_to_f64(np.asarray(scales_bits).reshape(G, N))
    z = w4_zero_points(G, N, zeros)
    g = w4_groups(K, g_idx)
    return (codes - z[g, :]).astype(np.float64) * s[g, :]


def act_order_perm(g_idx: np.ndarray, K: int) -> np.ndarray:
    """Resolve act order (MATE "Act order").

    perm = stable argsort of g_idx (ties in ascending k).  Valid only if every
    group 0..K/128-1 is one contiguous run of exactly 128 rows after sorting,
    i.e. g_idx[perm[i]] == i // 128 for all i; otherwise ValueError names the
    violated invariant.
    """
    g = np.asarray(g_idx, dtype=np.int64)
    if g.shape != (K,):
        raise ValueError(f"g_idx must have K={K} entries, got {g.shape}")
    G = K // GROUP
    if g.min(initial=0) < 0 or g.max(initial=0) >= G:
        raise ValueError(f"g_idx values must lie in [0, {G})")
    counts = np.bincount(g, minlength=G)
    bad = np.nonzero(counts != GROUP)[0]
    if bad.size:
        raise ValueError(
            f"g_idx group {int(bad[0])} has {int(counts[bad[0]])} rows; every sorted "
            f"group must be one contiguous run of {GROUP} rows")
    perm = np.argsort(g, kind="stable")
    assert np.array_equal(g[perm], np.arange(K) // GROUP)
    return perm.astype(np.int64)


def w4a16_linear(x_bits: np.ndarray, act_fmt: str, qweight: np.ndarray,
                 scales_bits: np.ndarray, zeros: np.ndarray | None = None,
                 g_idx: np.ndarray | None = None) -> np.ndarray:
    """y[M][N] = x @ W in fp64 (x read exactly from fp16/bf16 bits)."""
    x = bits_to_f64(x_bits, act_fmt)
    W = w4_dequant(qweight, scales_bits, zeros, g_idx)
    return x @ W


def w4a16_linear_columns(x_bits: np.ndarray, act_fmt: str, qweight: np.ndarray,
                         scales_bits: np.ndarray, zeros: np.ndarray | None,
                         g_idx: np.ndarray | None, cols: np.ndarray) -> np.ndarray:
    """The same as ``w4a16_linear`` restricted to output columns ``cols``
    (for sampled checks at sizes where the full product is too slow)."""
    cols = np.asarray(cols, dtype=np.int64)
    zsel = None if zeros is None else np.asarray(zeros)[:, cols]
    W = w4_dequant(np.asarray(qweight)[:, cols], np.asarray(scales_bits)[:, cols], zsel, g_idx)
    return bits_to_f64(x_bits, act_fmt) @ W


# --------------------------------------------------------------------------
# Ternary PQ2  [PRISM Test 1 (block format, byte expansion), Test 8 (replay)]
# --------------------------------------------------------------------------

def pq2_blocks(raw: np.ndarray) -> np.ndarray:
    raw = np.asarray(raw, dtype=np.uint8)
    N, width = raw.shape
    if width % PQ2_BLOCK_BYTES:
        raise ValueError("PQ2 row width must be a multiple of 34 bytes")
    return raw.reshape(N, width // PQ2_BLOCK_BYTES, PQ2_BLOCK_BYTES)


def pq2_codes(raw: np.ndarray) -> np.ndarray:
    """Codes c[N][K] (0..3): weight 4i+j of block b is bits 2j..2j+1 of code
    byte i of that block (the byte follows the 2-byte scale)."""
    blocks = pq2_blocks(raw)
    N, B, _ = blocks.shape
    code_bytes = blocks[:, :, 2:].astype(np.int64)          # [N][B][32]
    c = np.empty((N, B, 32, 4), dtype=np.int64)
    for j in range(4):
        c[:, :, :, j] = (code_bytes >> (2 * j)) & 3
    return c.reshape(N, B * GROUP).astype(np.uint8)


def pq2_values(raw: np.ndarray) -> np.ndarray:
    """Signed weights v = code - 1 in {-1, 0, 1, 2} (PRISM Test 1)."""
    return pq2_codes(raw).astype(np.int64) - 1


def pq2_scales(raw: np.ndarray) -> np.ndarray:
    """Block scales ws[N][K/128]: the little-endian fp16 at block offset 0."""
    blocks = pq2_blocks(raw)
    lo = blocks[:, :, 0].astype(np.uint16)
    hi = blocks[:, :, 1].astype(np.uint16)
    return f16_bits_to_f64(lo | (hi << 8))


def pq2_dequant(raw: np.ndarray) -> np.ndarray:
    """Dense weights Wt[N][K] = v * ws in fp64 (the PRISM Test 8 replay)."""
    v = pq2_values(raw)
    ws = pq2_scales(raw)
    return v.astype(np.float64) * np.repeat(ws, GROUP, axis=1)


def quantize_act(x_bits: np.ndarray, act_fmt: str, group: int):
    """Symmetric int8 activation quantiser (PRISM Test 6 code, TensorFold).

    Per group of ``group`` consecutive values of a row, all in fp32:
        amax  = max |a|
        scale = amax / 127                       (correctly rounded)
        q     = clamp(rint_even(a / scale), -127, 127)   (a / 1 if scale == 0)
    Returns q int8 [M][K] and scale fp32 [M][K/group].
    """
    x = bits_to_f64(x_bits, act_fmt).astype(np.float32)     # exact
    M, K = x.shape
    if group <= 0 or K % group:
        raise ValueError("activation group must divide K")
    a = x.reshape(M, K // group, group)
    amax = np.abs(a).max(axis=2)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    divisor = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    normalized = (a / divisor[:, :, None]).astype(np.float32)
    q = np.clip(np.rint(normalized), -127, 127).astype(np.int8)
    return q.reshape(M, K), scale


def w2a8_group_sums(q: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Exact integer block sums S[m][n][b] = sum over k in block b of
    v[n][k] * q[m][k]."""
    q = np.asarray(q, dtype=np.int64)
    v = np.asarray(v, dtype=np.int64)
    M, K = q.shape
    N = v.shape[0]
    B = K // GROUP
    qb = q.reshape(M, B, GROUP)
    vb = v.reshape(N, B, GROUP)
    return np.einsum("mbk,nbk->mnb", qb, vb)


def w2a8_linear(x_bits: np.ndarray, act_fmt: str, raw: np.ndarray, act_group: int):
    """Ternary W2A8 output in fp64: y[m][n] = sum_b S[m][n][b] * xs[m][b'] *
    ws[n][b], b' the activation group holding block b."""
    q, xs = quantize_act(x_bits, act_fmt, act_group)
    v = pq2_values(raw)
    ws = pq2_scales(raw)
    S = w2a8_group_sums(q, v).astype(np.float64)            # [M][N][B]
    M, K = q.shape
    B = K // GROUP
    blk_group = (np.arange(B) * GROUP) // act_group
    xs_b = xs.astype(np.float64)[:, blk_group]               # [M][B]
    return np.einsum("mnb,mb,nb->mn", S, xs_b, ws)


def w2a8_linear_columns(x_bits: np.ndarray, act_fmt: str, raw: np.ndarray,
                        act_group: int, rows: np.ndarray) -> np.ndarray:
    """``w2a8_linear`` restricted to output features ``rows``."""
    return w2a8_linear(x_bits, act_fmt, np.asarray(raw)[np.asarray(rows)], act_group)


# --------------------------------------------------------------------------
# Fused activation producer  [PRISM "E. Keeping preparation data close to
# compute", Test 18 and Diagram 5: RMSNorm + Hadamard + Q8 in one pass]
#
# Floating point follows the page: every step is fp32 (the normalisation,
# the sign flip and transform, the group quantiser), with the two roundings
# to the activation dtype the page makes (after the norm weight, after the
# transform).  Test 18 states that the reduction order of the sum of squares
# decides codes, so the order is part of the definition here:
#   * 2048 lanes; lane i accumulates u[i]^2, u[i + 2048]^2, ... in turn
#     (fp32 multiply, then fp32 add), as the page's 2048-wide accumulator;
#   * the lanes are then added by halving: lane i += lane i + h for
#     h = 1024, 512, ..., 1 (the page leaves the final lane sum to its
#     compiler; halving is this oracle's reading).
# Further readings: 1/sqrt(var + eps) is taken as the correctly rounded
# square root followed by the correctly rounded reciprocal; the Hadamard
# transform of a block of B values is the orthonormal one, H_B v * RN(1/sqrt(B))
# with H_B the natural-order (Sylvester) matrix, formed by butterflies
# (a, b) -> (a + b, a - b) at strides 1, 2, ..., B/2.
# --------------------------------------------------------------------------

NORM_LANES = 2048


def rms_sum_squares(u: np.ndarray) -> np.ndarray:
    """fp32 sum of u^2 along each row in the order stated above.  u: fp32 [M][K]."""
    u = np.asarray(u, dtype=np.float32)
    M, K = u.shape
    acc = np.zeros((M, NORM_LANES), dtype=np.float32)
    for off in range(0, K, NORM_LANES):
        seg = u[:, off:off + NORM_LANES]
        n = seg.shape[1]
        sq = (seg * seg).astype(np.float32)                   # rounded product
        acc[:, :n] = (acc[:, :n] + sq).astype(np.float32)     # rounded sum
    h = NORM_LANES // 2
    while h >= 1:
        acc = (acc[:, :h] + acc[:, h:2 * h]).astype(np.float32)
        h //= 2
    return acc[:, 0]


def rms_inverse(total: np.ndarray, K: int, eps: float) -> np.ndarray:
    """inv = 1 / sqrt(total / K + eps), each operation a correctly rounded fp32 step."""
    var = (np.asarray(total, dtype=np.float32) / np.float32(K)).astype(np.float32)
    root = np.sqrt((var + np.float32(eps)).astype(np.float32)).astype(np.float32)
    return (np.float32(1.0) / root).astype(np.float32)


def fwht_blocks(v: np.ndarray, B: int) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform of every block of B consecutive
    values of each row (fp32 butterflies, every sum and difference rounded)."""
    v = np.asarray(v, dtype=np.float32)
    M, K = v.shape
    if B < 2 or B & (B - 1) or K % B:
        raise ValueError("Hadamard block must be a power of two dividing K")
    w = v.reshape(M, K // B, B)
    h = 1
    while h < B:
        x = w.reshape(M, K // B, B // (2 * h), 2, h)
        a, b = x[:, :, :, 0, :], x[:, :, :, 1, :]
        w = np.stack([(a + b).astype(np.float32), (a - b).astype(np.float32)], axis=3).reshape(M, K // B, B)
        h *= 2
    return w.reshape(M, K)


def norm_quantize(h_bits: np.ndarray, r_bits: np.ndarray | None, gamma_bits: np.ndarray, act_fmt: str,
                  eps: float, unit_offset: bool, signs: np.ndarray | None, had_block: int, act_group: int):
    """Fused activation producer (PRISM Test 18), all fp32:
        u      = h (+ r)                         residual add; r_out = RN_act(u)
        inv    = 1 / sqrt(sum(u^2) / K + eps)    (order as stated above)
        n      = RN_act((u * inv) * w),  w = gamma (+ 1 when unit_offset)
        v      = RN_act(H_B(n * signs) * RN(1/sqrt(B)))   when had_block = B > 0, else n
        q, xs  = quantize_act(v)                 (Test 6 group quantiser)
        sq     = per-128-block sum of q
    Returns a dict of 16-bit patterns (r_out, norm, v), q int8, xs fp32, sq int64.
    """
    h = bits_to_f64(h_bits, act_fmt).astype(np.float32)       # exact
    M, K = h.shape
    u = h
    r_out = None
    if r_bits is not None:
        u = (h + bits_to_f64(r_bits, act_fmt).astype(np.float32)).astype(np.float32)
        r_out = f64_to_bits(u.astype(np.float64), act_fmt)
    inv = rms_inverse(rms_sum_squares(u), K, eps)
    w = bits_to_f64(gamma_bits, act_fmt).astype(np.float32)
    if unit_offset:
        w = (w + np.float32(1.0)).astype(np.float32)
    t = (u * inv[:, None]).astype(np.float32)
    norm = f64_to_bits((t * w[None, :]).astype(np.float32).astype(np.float64), act_fmt)
    v_bits = norm
    if had_block:
        n = bits_to_f64(norm, act_fmt).astype(np.float32)
        if signs is not None:
            n = np.where(np.asarray(signs)[None, :] < 0, -n, n).astype(np.float32)
        scale = np.float32(1.0 / np.sqrt(float(had_block)))
        v = (fwht_blocks(n, had_block) * scale).astype(np.float32)
        v_bits = f64_to_bits(v.astype(np.float64), act_fmt)
    q, xs = quantize_act(v_bits, act_fmt, act_group)
    sq = q.astype(np.int64).reshape(M, K // GROUP, GROUP).sum(axis=2)
    return {"r_out": r_out, "norm": norm, "v": v_bits, "q": q, "xs": xs, "sq": sq}


# --------------------------------------------------------------------------
# MLX affine 4-bit weights  ["qwen CUDA: --prompt-precision int8 ... - #1176"
# (TensorFold), the affine-4 projections of its prompt pass: 4-bit codes
# 0..15, one scale and one bias per 64-input group, w = s * q + b]
#
# Readings where the page is silent: the weight is stored output-row major,
# [N][K/8] words of eight codes along K, code k of a row in bits 4*(k % 8) of
# word k // 8 (least significant first, as the GPTQ words above); scales and
# biases are [N][K/64] in the model's 16-bit dtype.  The CUDA path checked
# against it repacks these planes for its own decode kernels.
# --------------------------------------------------------------------------

AFFINE_GROUP = 64


def affine4_codes(wq: np.ndarray) -> np.ndarray:
    """Codes [N][K] (0..15) from words [N][K/8]."""
    w = np.asarray(wq, dtype=np.uint32)
    N, KW = w.shape
    codes = np.empty((N, KW * 8), dtype=np.uint8)
    for i in range(8):
        codes[:, i::8] = (w >> np.uint32(4 * i)) & np.uint32(0xF)
    return codes


def affine4_dequant(wq: np.ndarray, scales_bits: np.ndarray, biases_bits: np.ndarray, fmt: str) -> np.ndarray:
    """Dequantised weights W[N][K] in fp64: w(n, k) = s(n, g) * q(n, k) + b(n, g),
    g = k // 64 (each product and sum exact in fp64 for 16-bit s and b)."""
    q = affine4_codes(wq).astype(np.float64)
    N, K = q.shape
    if K % AFFINE_GROUP:
        raise ValueError("K must be a multiple of 64")
    G = K // AFFINE_GROUP
    s = bits_to_f64(np.asarray(scales_bits).reshape(N, G), fmt)
    b = bits_to_f64(np.asarray(biases_bits).reshape(N, G), fmt)
    g = np.arange(K) // AFFINE_GROUP
    return s[:, g] * q + b[:, g]


def affine4_linear(x_bits: np.ndarray, act_fmt: str, wq: np.ndarray, scales_bits: np.ndarray,
                   biases_bits: np.ndarray, wfmt: str) -> np.ndarray:
    """y[M][N] = x . W^T in fp64 (not rounded)."""
    x = bits_to_f64(x_bits, act_fmt)
    return x @ affine4_dequant(wq, scales_bits, biases_bits, wfmt).T
