"""GPU parity of the decode path against the CPU oracle, through the C ABI.

Bit-exact: dequantised weights (pq_debug_unpack), the int8 activation codes
and scales, and the ternary int32 block sums.  Floating outputs: the output
metric of tests/helpers.py within 2e-3, plus a check that nearly every
output equals the correctly rounded oracle value.  Shapes span several
strips / row tiles with ragged tails (N not a multiple of 16) and uneven
K splits.
"""
from __future__ import annotations

import numpy as np
import pytest

import pq_inputs
from oracle import pq_oracle as O
from tests.helpers import TOL, bits_of, exact_fraction, o8_error, rel_rms, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_weight_quantized_pq_gb300 as pq  # noqa: E402

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pq.build()
    return torch.device("cuda:0")


def w4_layer(dev, fr, act, max_m, out=None):
    return pq.QuantizedLinear.from_w4(
        to_dev(fr["qweight"], dev), to_dev(fr["scales"], dev),
        None if fr["zeros"] is None else to_dev(fr["zeros"], dev), fr["g_idx"],
        act_dtype=act, out_dtype=out, max_m=max_m)


def w2_layer(dev, raw, K, act, ag, max_m):
    return pq.QuantizedLinear.from_pq2(to_dev(raw, dev), K, act_dtype=act, act_group=ag, max_m=max_m)


# ---------------------------------------------------------------- W4 ------

@pytest.mark.parametrize("N,K,zp,act", [
    (72, 256, False, None), (200, 640, True, None), (64, 512, True, "scatter"), (48, 384, False, "blocks")])
def test_w4_unpack_bit_exact(dev, N, K, zp, act):
    fr = pq_inputs.w4_frame(3, K, N, 0.002, 0.01, zp, act)
    layer = w4_layer(dev, fr, "bf16", 1)
    w = torch.empty((K, N), dtype=torch.float32, device=dev)
    pq.pq_debug_unpack(layer.handle, w)
    ref = O.w4_dequant(fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    assert np.array_equal(w.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16])
@pytest.mark.parametrize("act_dt", ["f16", "bf16"])
@pytest.mark.parametrize("N,K,zp,act", [
    (200, 640, False, None), (96, 1024, True, None), (136, 768, True, "scatter")])
def test_w4_gemv_parity(dev, M, act_dt, N, K, zp, act):
    fr = pq_inputs.w4_frame(10 + M, K, N, 0.002, 0.01, zp, act)
    x = pq_inputs.activations(20 + M, M, K, act_dt)
    layer = w4_layer(dev, fr, act_dt, 16)
    y = layer(to_dev(x, dev, DT[act_dt]), variant=pq.PQ_VARIANT_W4_GEMV)
    got = bits_of(y)
    ref = O.w4a16_linear(x, act_dt, fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    assert o8_error(got, ref, act_dt) <= TOL
    assert exact_fraction(got, ref, act_dt) >= 0.97, rel_rms(got, ref, act_dt)


@pytest.mark.parametrize("M,N,K", [(20, 72, 896), (1, 40, 82048), (1, 24, 81408), (1, 24, 81536), (2, 24, 128),
                                   (4, 24, 16384), (4, 24, 40960)])
def test_w4_gemv_split_k_edges(dev, M, N, K):
    # M > 16 runs 16-token tiles back to back on one workspace (the 4-token
    # tail on the whole-row kernel); K = 81408 is the longest row the
    # one-token kernel holds beside its ring and static buffer, a longer row
    # takes the split-K kernel with one token; K = 128 is a
    # single slice of one group; four rows of 16384 still fit the whole-row
    # kernel (one CTA per SM), four of 40960 do not (split-K)
    fr = pq_inputs.w4_frame(30 + M, K, N, 0.002, 0.01, True, None)
    x = pq_inputs.activations(31 + M, M, K, "bf16")
    layer = w4_layer(dev, fr, "bf16", M)
    got = [bits_of(layer(to_dev(x, dev, torch.bfloat16), variant=pq.PQ_VARIANT_W4_GEMV)) for _ in range(2)]
    ref = O.w4a16_linear(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], None)
    assert np.array_equal(got[0], got[1])          # fixed-order slice sums: bit-identical
    assert o8_error(got[0], ref, "bf16") <= TOL
    assert exact_fraction(got[0], ref, "bf16") >= 0.97


@pytest.mark.parametrize("M,N,K,zp", [
    (1, 24, 128, False),        # two strips of one group
    (1, 200, 640, True),        # 13 strips, ragged N
    (3, 65536, 128, False),     # 4096 one-group strips: many strips per CTA
    (1, 131088, 128, True),     # 8193 strips
    (2, 4104, 4096, True),      # 257 strips of 32 groups, ragged N
])
def test_w4_decode_strip_counts(dev, M, N, K, zp):
    # Whole-row decode over layers with few or many strips per CTA: matches
    # the oracle and repeats bit for bit.
    fr = pq_inputs.w4_frame(50 + M, K, N, 0.002, 0.01, zp, None)
    x = pq_inputs.activations(51 + M, M, K, "bf16")
    layer = w4_layer(dev, fr, "bf16", M)
    xd = to_dev(x, dev, torch.bfloat16)
    got = [bits_of(layer(xd, variant=pq.PQ_VARIANT_W4_GEMV)) for _ in range(3)]
    assert np.array_equal(got[0], got[1]) and np.array_equal(got[0], got[2])
    ref = O.w4a16_linear(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], None)
    assert o8_error(got[0], ref, "bf16") <= TOL
    assert exact_fraction(got[0], ref, "bf16") >= 0.97


def test_w4_decode_shared_workspace(dev):
    # Three layers of different shapes on one workspace, called in turn (the
    # workspace sized for the largest): every call equals the same layer run
    # alone on a workspace of its own.
    shapes = [(200, 640), (4104, 4096), (24, 128)]
    frames = [pq_inputs.w4_frame(60 + i, K, N, 0.002, 0.01, i == 1, None) for i, (N, K) in enumerate(shapes)]
    alone = []
    for fr in frames:
        L = w4_layer(dev, fr, "bf16", 4)
        xs = to_dev(pq_inputs.activations(70, 4, fr["qweight"].shape[0] * 8, "bf16"), dev, torch.bfloat16)
        alone.append(bits_of(L(xs[:1], variant=pq.PQ_VARIANT_W4_GEMV)))
        L.close()
    descs = [pq.make_desc(pq.PQ_FMT_W4_GPTQ, N, K, zp=pq.PQ_ZP_EXPLICIT_U8 if i == 1 else pq.PQ_ZP_SYMMETRIC_8,
                          act_dtype=pq.PQ_BF16, max_m=4) for i, (N, K) in enumerate(shapes)]
    ws_bytes = max(pq.pq_workspace_bytes(d) for d in descs)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    hs, keep = [], []
    for d, fr in zip(descs, frames):
        prep = torch.empty(pq.pq_prepared_bytes(d), dtype=torch.uint8, device=dev)
        z = None if fr["zeros"] is None else to_dev(fr["zeros"], dev)
        hs.append(pq.pq_prepare_w4(d, to_dev(fr["qweight"], dev), to_dev(fr["scales"], dev), z, None, prep,
                                   prep.numel(), ws, ws_bytes))
        keep.append(prep)
    for rep in range(3):
        for i, (h, (N, K)) in enumerate(zip(hs, shapes)):
            xs = to_dev(pq_inputs.activations(70, 4, K, "bf16"), dev, torch.bfloat16)
            y = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
            pq.pq_linear(xs[:1], h, y, 1)
            assert np.array_equal(bits_of(y), alone[i]), (rep, i)
    for h in hs:
        pq.pq_destroy(h)


def test_split_k_many_strips_mixed_m(dev):
    # Split-K decode over 4097 strips of 16 rows, calls at different M on
    # one handle in turn: each matches the oracle, and a repeated call
    # repeats bit for bit (no state carried from one call to the next).
    N, K = 65552, 256
    fr = pq_inputs.w4_frame(80, K, N, 0.002, 0.01, True, None)
    raw = pq_inputs.pq2_rows(81, N, K)
    L4 = w4_layer(dev, fr, "bf16", 16)
    L2 = w2_layer(dev, raw, K, "bf16", K, 16)
    for rep in range(2):
        for M in (16, 5, 12):
            x = pq_inputs.activations(82 + M, M, K, "bf16")
            xd = to_dev(x, dev, torch.bfloat16)
            got4 = bits_of(L4(xd, variant=pq.PQ_VARIANT_W4_GEMV))
            ref4 = O.w4a16_linear(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], None)
            assert o8_error(got4, ref4, "bf16") <= TOL, (rep, M)
            v = pq.PQ_VARIANT_W2_GEMV_BF if M > 8 else pq.PQ_VARIANT_W2_GEMV_TC
            got2 = bits_of(L2(xd, variant=v))
            ref2 = O.w2a8_linear(x, "bf16", raw, K)
            assert o8_error(got2, ref2, "bf16") <= TOL, (rep, M)
            if rep == 0:
                first = (got4, got2) if M == 16 else first
            elif M == 16:
                assert np.array_equal(got4, first[0]) and np.array_equal(got2, first[1])


@pytest.mark.parametrize("M", [5, 8])
def test_w4_split_k_cluster_three_blocks(dev, M):
    # 11008 x 4096 at M = 5..8: eight K slices run as one cluster per block
    # of 8 strips, and each CTA walks three blocks (the most its shared
    # memory holds the slice sums of): matches the oracle, repeats bit for bit
    N, K = 11008, 4096
    fr = pq_inputs.w4_frame(95 + M, K, N, 0.002, 0.01, True, None)
    x = pq_inputs.activations(96 + M, M, K, "bf16")
    layer = w4_layer(dev, fr, "bf16", 16)
    plan = pq.pq_plan(layer.desc, M, 152)
    assert plan["launches"] == 1 and plan["k_split"] == 8
    xd = to_dev(x, dev, torch.bfloat16)
    got = [bits_of(layer(xd, variant=pq.PQ_VARIANT_W4_GEMV)) for _ in range(2)]
    assert np.array_equal(got[0], got[1])
    rng = np.random.default_rng(3)
    cols = np.sort(rng.choice(N, 512, replace=False))
    ref = O.w4a16_linear_columns(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], None, cols)
    assert o8_error(got[0][:, cols], ref, "bf16") <= TOL
    assert exact_fraction(got[0][:, cols], ref, "bf16") >= 0.97


def test_split_k_shared_workspace(dev):
    # A 4-bit and a ternary layer on one workspace, split-K calls in turn:
    # each equals the same layer on a workspace of its own.
    N4, K4, N2, K2, M = 4104, 1024, 1000, 2048, 9
    fr = pq_inputs.w4_frame(90, K4, N4, 0.002, 0.01, False, None)
    raw = pq_inputs.pq2_rows(91, N2, K2)
    x4 = to_dev(pq_inputs.activations(92, M, K4, "bf16"), dev, torch.bfloat16)
    x2 = to_dev(pq_inputs.activations(93, M, K2, "bf16"), dev, torch.bfloat16)
    a4 = bits_of(w4_layer(dev, fr, "bf16", M)(x4, variant=pq.PQ_VARIANT_W4_GEMV))
    a2 = bits_of(w2_layer(dev, raw, K2, "bf16", 128, M)(x2, variant=pq.PQ_VARIANT_W2_GEMV_BF))
    d4 = pq.make_desc(pq.PQ_FMT_W4_GPTQ, N4, K4, act_dtype=pq.PQ_BF16, max_m=M)
    d2 = pq.make_desc(pq.PQ_FMT_W2_PQ2, N2, K2, act_dtype=pq.PQ_BF16, act_group=128, max_m=M)
    ws_bytes = max(pq.pq_workspace_bytes(d4), pq.pq_workspace_bytes(d2))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    p4 = torch.empty(pq.pq_prepared_bytes(d4), dtype=torch.uint8, device=dev)
    p2 = torch.empty(pq.pq_prepared_bytes(d2), dtype=torch.uint8, device=dev)
    h4 = pq.pq_prepare_w4(d4, to_dev(fr["qweight"], dev), to_dev(fr["scales"], dev), None, None, p4, p4.numel(),
                          ws, ws_bytes)
    r2 = to_dev(raw, dev)
    h2 = pq.pq_prepare_w2(d2, r2, r2.stride(0), p2, p2.numel(), ws, ws_bytes)
    y4 = torch.empty((M, N4), dtype=torch.bfloat16, device=dev)
    y2 = torch.empty((M, N2), dtype=torch.bfloat16, device=dev)
    for rep in range(3):
        pq.pq_linear_variant(x4, h4, y4, M, pq.PQ_VARIANT_W4_GEMV)
        pq.pq_linear_variant(x2, h2, y2, M, pq.PQ_VARIANT_W2_GEMV_BF)
        assert np.array_equal(bits_of(y4), a4) and np.array_equal(bits_of(y2), a2), rep
    pq.pq_destroy(h4)
    pq.pq_destroy(h2)


@pytest.mark.parametrize("M,N,K", [(1, 56, 10240), (3, 40, 9216), (1, 56, 16384), (3, 40, 12288),
                                   (20, 136, 768)])
def test_w4_gemv_act_order_gather(dev, M, N, K):
    # under act order the whole-row kernel permutes x in shared memory itself
    # where the second copy of the rows costs no residency: rows longer than
    # its prefetched permutation chunks (K = 10240 for one token, 9216 for
    # four); one row of 16384 and four of 12288 take a gather launch first;
    # and a 16 + 4 token split runs its 4-token tail on the gathered copy
    fr = pq_inputs.w4_frame(40 + M, K, N, 0.002, 0.01, True, "scatter")
    x = pq_inputs.activations(41 + M, M, K, "bf16")
    layer = w4_layer(dev, fr, "bf16", M)
    got = bits_of(layer(to_dev(x, dev, torch.bfloat16), variant=pq.PQ_VARIANT_W4_GEMV))
    ref = O.w4a16_linear(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    assert o8_error(got, ref, "bf16") <= TOL
    assert exact_fraction(got, ref, "bf16") >= 0.97


def test_w4_mixed_output_dtype(dev):
    K, N, M = 512, 64, 2
    fr = pq_inputs.w4_frame(5, K, N, 0.002, 0.01, True, None)
    x = pq_inputs.activations(6, M, K, "f16")
    layer = w4_layer(dev, fr, "f16", 2, out="bf16")
    got = bits_of(layer(to_dev(x, dev, torch.float16)))
    ref = O.w4a16_linear(x, "f16", fr["qweight"], fr["scales"], fr["zeros"], None)
    assert o8_error(got, ref, "bf16") <= TOL


def test_w4_zero_weights_and_one_hot(dev):
    K, N = 256, 32
    fr = pq_inputs.w4_frame(7, K, N, 0.002, 0.01)
    fr0 = dict(fr, qweight=np.full_like(fr["qweight"], 0x88888888))
    x = pq_inputs.activations(8, 1, K, "bf16")
    y = w4_layer(dev, fr0, "bf16", 1)(to_dev(x, dev, torch.bfloat16))
    assert not bits_of(y).any() or (np.abs(O.bf16_bits_to_f64(bits_of(y))) == 0).all()
    layer = w4_layer(dev, fr, "bf16", 1)
    for k in (0, 9, 130, 255):
        xb = np.zeros((1, K), dtype=np.uint16)
        xb[0, k] = 0x3F80
        got = bits_of(layer(to_dev(xb, dev, torch.bfloat16)))
        ref = O.w4a16_linear(xb, "bf16", fr["qweight"], fr["scales"])
        assert np.array_equal(got, O.f64_to_bits(ref, "bf16"))


def test_w4_act_order_matches_unpermuted(dev):
    # the same weights with identity g_idx and with no g_idx give identical bits
    K, N, M = 512, 80, 4
    fr = pq_inputs.w4_frame(9, K, N, 0.002, 0.01, True, None)
    frg = dict(fr, g_idx=(np.arange(K) // 128).astype(np.int32))
    x = to_dev(pq_inputs.activations(10, M, K, "bf16"), dev, torch.bfloat16)
    a = bits_of(w4_layer(dev, fr, "bf16", M)(x))
    b = bits_of(w4_layer(dev, frg, "bf16", M)(x))
    assert np.array_equal(a, b)


def test_w4_rows_independent_and_deterministic(dev):
    K, N, M = 768, 160, 5
    fr = pq_inputs.w4_frame(11, K, N, 0.002, 0.01, True, "scatter")
    layer = w4_layer(dev, fr, "bf16", M)
    x = pq_inputs.activations(12, M, K, "bf16")
    x2 = x.copy()
    x2[3] = pq_inputs.activations(13, 1, K, "bf16")[0]
    a = bits_of(layer(to_dev(x, dev, torch.bfloat16)))
    a2 = bits_of(layer(to_dev(x, dev, torch.bfloat16)))
    b = bits_of(layer(to_dev(x2, dev, torch.bfloat16)))
    assert np.array_equal(a, a2)
    assert np.array_equal(np.delete(a, 3, 0), np.delete(b, 3, 0)) and not np.array_equal(a[3], b[3])


# ---------------------------------------------------------------- W2 ------

@pytest.mark.parametrize("M,K,ag,act_dt", [
    (1, 4096, 4096, "bf16"), (3, 1024, 128, "bf16"), (2, 640, 640, "f16"), (16, 512, 128, "f16")])
def test_w2_quantize_bit_exact(dev, M, K, ag, act_dt):
    raw = pq_inputs.pq2_rows(1, 16, K)
    x = pq_inputs.activations(30 + M, M, K, act_dt)
    x[0, 5] = 0                                    # exact zeros and a tie-heavy row
    layer = w2_layer(dev, raw, K, act_dt, ag, M)
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    xs = torch.empty((M, K // ag), dtype=torch.float32, device=dev)
    pq.pq_debug_w2a8_quantize(to_dev(x, dev, DT[act_dt]), layer.handle, q, xs, M)
    q_ref, xs_ref = O.quantize_act(x, act_dt, ag)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32))


def test_w2_quantize_zero_row_and_ties(dev):
    K = 256
    raw = pq_inputs.pq2_rows(1, 16, K)
    x = np.zeros((2, K), dtype=np.float32)
    x[1, :8] = [127, -63.5, 0.5, 1.5, 2.5, -0.5, 3, -127]
    xb = pq_inputs.f32_to_bf16_bits(x)
    layer = w2_layer(dev, raw, K, "bf16", 128, 2)
    q = torch.empty((2, K), dtype=torch.int8, device=dev)
    xs = torch.empty((2, 2), dtype=torch.float32, device=dev)
    pq.pq_debug_w2a8_quantize(to_dev(xb, dev, torch.bfloat16), layer.handle, q, xs, 2)
    assert not q[0].any() and float(xs[0, 0]) == 0.0
    assert q[1, :8].tolist() == [127, -64, 0, 2, 2, 0, 3, -127]


def _all_magnitudes(top_bits, K, rng):
    """Every finite non-negative 16-bit pattern up to top_bits (zero, the
    subnormals and all normals), random signs, zero-padded to K."""
    v = np.arange(0, top_bits + 1, dtype=np.uint32)
    v = v[-K:] if v.size > K else v
    v = v | (rng.integers(0, 2, v.size).astype(np.uint32) << 15)
    row = np.zeros(K, dtype=np.uint16)
    row[:v.size] = v.astype(np.uint16)
    return row


@pytest.mark.parametrize("act_dt,K,ag", [("bf16", 32768, 32768), ("bf16", 16384, 16384), ("bf16", 16384, 128),
                                         ("f16", 32768, 32768), ("f16", 16384, 128)])
def test_w2_quantize_every_input_value(dev, act_dt, K, ag):
    # Each row holds every representable magnitude below its maximum, so every
    # quotient a / scale the divider can meet for that scale (exact ties at
    # k + 1/2 included when the scale is a power of two) is checked against the
    # correctly rounded fp32 division of the oracle.
    rng = np.random.default_rng(7)
    if act_dt == "bf16":
        tops = [0x7F7F, 0x42FE, 0x3F80, 0x3B44, 0x0F00]  # max finite, 127, 1, ~3e-3, ~6e-30
    else:
        tops = [0x7BFF, 0x57F0, 0x3C00, 0x1A3D]         # 65504, 127, 1, ~3e-3
    x = np.stack([_all_magnitudes(t, K, rng) for t in tops])
    if ag == 128:
        x = np.stack([rng.permutation(r) for r in x])   # blocks with scattered maxima
    M = x.shape[0]
    layer = w2_layer(dev, pq_inputs.pq2_rows(1, 16, K), K, act_dt, ag, M)
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    xs = torch.empty((M, K // ag), dtype=torch.float32, device=dev)
    pq.pq_debug_w2a8_quantize(to_dev(x, dev, DT[act_dt]), layer.handle, q, xs, M)
    q_ref, xs_ref = O.quantize_act(x, act_dt, ag)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


def _every_scale_groups(act_dt, rng):
    """One 128-value group per positive finite 16-bit magnitude A (every
    value the group maximum can take, so every divisor RN(A / 127) the
    quantiser can meet: all-ones significands, subnormal maxima and, for
    bf16, scales on both sides of 2^-100), plus one all-zero group.  A sits
    at a random position with a random sign; the other 127 values are random
    magnitudes up to A (bit patterns of non-negative floats order like their
    values) with random signs.  Returns [groups][128] uint16 bits."""
    top = 0x7F7F if act_dt == "bf16" else 0x7BFF
    amax = np.arange(0, top + 1, dtype=np.uint32)       # 0 first: the all-zero group
    n = amax.size
    mag = (rng.random((n, 128)) * (amax[:, None] + 1).astype(np.float64)).astype(np.uint32)
    mag = np.minimum(mag, amax[:, None])
    pos = rng.integers(0, 128, n)
    mag[np.arange(n), pos] = amax
    sign = rng.integers(0, 2, (n, 128)).astype(np.uint32) << 15
    return (mag | sign).astype(np.uint16)


@pytest.mark.parametrize("act_dt", ["bf16", "f16"])
def test_w2_quantize_every_group_scale(dev, act_dt):
    # Per-128 activation groups, one per possible group maximum: the divider
    # (reciprocal, one-FMA residual, final correction) must give the
    # correctly rounded fp32 quotient for every scale, on both code layouts
    # (int8 plane order for decode, bf16 tensor-core order for the GEMM).
    rng = np.random.default_rng(101 if act_dt == "bf16" else 102)
    grp = _every_scale_groups(act_dt, rng)
    K = 65536
    per_row = K // 128
    M = -(-grp.shape[0] // per_row)
    pad = np.zeros((M * per_row - grp.shape[0], 128), dtype=np.uint16)
    x = np.concatenate([grp, pad]).reshape(M, K)
    layer = w2_layer(dev, pq_inputs.pq2_rows(1, 16, K), K, act_dt, 128, M)
    xd = to_dev(x, dev, DT[act_dt])
    q_ref, xs_ref = O.quantize_act(x, act_dt, 128)
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    xs = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
    pq.pq_debug_w2a8_quantize(xd, layer.handle, q, xs, M)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    # M > 16: the quantiser writes bf16 codes in tensor-core order
    ab = pq.pq_act_bytes(layer.desc, M)
    act = torch.empty(ab, dtype=torch.uint8, device=dev)
    pq.pq_quantize_act(xd, layer.handle, act, ab, M)
    q2 = torch.empty_like(q)
    xs2 = torch.empty_like(xs)
    sq = torch.empty((M, K // 128), dtype=torch.int32, device=dev)
    pq.pq_debug_act_unpack(act, ab, layer.handle, M, q2, xs2, sq)
    assert np.array_equal(q2.cpu().numpy(), q_ref)
    assert np.array_equal(xs2.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32))
    assert np.array_equal(sq.cpu().numpy().astype(np.int64), q_ref.astype(np.int64).reshape(M, -1, 128).sum(axis=2))


@pytest.mark.parametrize("N,K,code3", [(37, 640, True), (16, 1152, True), (200, 1024, False), (5, 128, True)])
def test_w2_unpack_bit_exact(dev, N, K, code3):
    # Prepared ternary planes against the PQ2 definition: dequantised weights
    # (code - 1) * ws bit for bit, for ragged N, K / 128 not a multiple of 8
    # (padded scale rows) and code 3; and the planes themselves rebuild the
    # caller's 34-byte blocks byte for byte (code plane [Npad][K/4], then the
    # scale plane [Npad][Bp] at the next 256-byte boundary).
    raw = pq_inputs.pq2_rows(9 + N, N, K, allow_code3=code3)
    layer = w2_layer(dev, raw, K, "bf16", 128, 1)
    w = torch.empty((K, N), dtype=torch.float32, device=dev)
    pq.pq_debug_unpack(layer.handle, w)
    ref = O.pq2_dequant(raw).T
    assert np.array_equal(w.cpu().numpy().astype(np.float64), ref)
    planes = layer.prepared.cpu().numpy()
    npad, B = -(-N // 16) * 16, K // 128
    bp = -(-B // 8) * 8
    soff = -(-(npad * K // 4) // 256) * 256
    codes = planes[:npad * K // 4].reshape(npad, B, 32)
    scales = planes[soff:soff + npad * bp * 2].reshape(npad, bp, 2)
    rebuilt = np.concatenate([scales[:N, :B], codes[:N]], axis=2).reshape(N, B * 34)
    assert np.array_equal(rebuilt, raw)
    assert not scales[:, B:].any() and not codes[N:].any() and not scales[N:].any()


@pytest.mark.parametrize("M,N,K,ag,code3", [(1, 48, 4096, 4096, False), (3, 40, 1024, 128, True),
                                             (5, 24, 11008, 128, False)])
def test_w2_group_sums_bit_exact(dev, M, N, K, ag, code3):
    raw = pq_inputs.pq2_rows(2, N, K, allow_code3=code3)
    x = pq_inputs.activations(40, M, K, "bf16")
    layer = w2_layer(dev, raw, K, "bf16", ag, M)
    S = torch.empty((M, N, K // 128), dtype=torch.int32, device=dev)
    pq.pq_debug_w2a8_group_sums(to_dev(x, dev, torch.bfloat16), layer.handle, S, M)
    q, _ = O.quantize_act(x, "bf16", ag)
    S_ref = O.w2a8_group_sums(q, O.pq2_values(raw))
    assert np.array_equal(S.cpu().numpy().astype(np.int64), S_ref)


@pytest.mark.parametrize("M,N,K,ag,act_dt,variant", [
    (1, 200, 4096, 4096, "bf16", pq.PQ_VARIANT_W2_GEMV_FUSED),
    (1, 72, 11008, 11008, "bf16", pq.PQ_VARIANT_W2_GEMV_FUSED),
    (3, 104, 1024, 128, "f16", pq.PQ_VARIANT_W2_GEMV_FUSED),
    (4, 64, 2048, 2048, "bf16", pq.PQ_VARIANT_W2_GEMV),
    (7, 56, 640, 128, "bf16", pq.PQ_VARIANT_W2_GEMV),
    (16, 40, 1280, 1280, "f16", pq.PQ_VARIANT_W2_GEMV),
    (1, 64, 2048, 2048, "bf16", pq.PQ_VARIANT_W2_GEMV_TC),
    (2, 72, 4096, 4096, "bf16", pq.PQ_VARIANT_W2_GEMV_TC),
    (5, 88, 1152, 128, "f16", pq.PQ_VARIANT_W2_GEMV_TC),
    (7, 56, 640, 128, "bf16", pq.PQ_VARIANT_W2_GEMV_TC),
    (9, 40, 11008, 11008, "bf16", pq.PQ_VARIANT_W2_GEMV_TC),
    (16, 200, 1280, 128, "bf16", pq.PQ_VARIANT_W2_GEMV_TC),
    (1, 64, 2048, 2048, "bf16", pq.PQ_VARIANT_W2_GEMV_BF),
    (3, 72, 4096, 4096, "bf16", pq.PQ_VARIANT_W2_GEMV_BF),
    (5, 88, 1152, 128, "f16", pq.PQ_VARIANT_W2_GEMV_BF),
    (7, 56, 640, 128, "bf16", pq.PQ_VARIANT_W2_GEMV_BF),
    (9, 40, 11008, 11008, "bf16", pq.PQ_VARIANT_W2_GEMV_BF),
    (16, 200, 1280, 128, "bf16", pq.PQ_VARIANT_W2_GEMV_BF),
])
def test_w2_gemv_parity(dev, M, N, K, ag, act_dt, variant):
    raw = pq_inputs.pq2_rows(50 + M, N, K, allow_code3=(M == 7))
    x = pq_inputs.activations(60 + M, M, K, act_dt)
    # the split-K variant needs a workspace sized for more than one token
    layer = w2_layer(dev, raw, K, act_dt, ag, max(M, 2))
    got = bits_of(layer(to_dev(x, dev, DT[act_dt]), variant=variant))
    ref = O.w2a8_linear(x, act_dt, raw, ag)
    assert o8_error(got, ref, act_dt) <= TOL
    assert exact_fraction(got, ref, act_dt) >= 0.97, rel_rms(got, ref, act_dt)


@pytest.mark.parametrize("N,K,ag,act_dt", [(5008, 4096, 4096, "bf16"), (5008, 3968, 128, "f16"),
                                         (9760, 2176, 2176, "bf16"), (300, 4096, 128, "bf16")])
def test_w2_gemv_one_token_row_mix(dev, N, K, ag, act_dt):
    # The one-token GEMV gives each warp rows gw, gw + TW, ... (TW = 304 CTAs
    # x 16 warps = 4864 on a 152-SM part): N = 5008 and 9760 put one and two
    # (two and three) rows on different warps of the same launch, so the
    # register-held loop (two rows or more) and the general loop (one row)
    # both write outputs; K = 3968 and 2176 leave lanes without a block.
    # Against the oracle, and bit for bit against the same layer run on the
    # caller-held quantised buffer (the non-fused instance of the kernel).
    raw = pq_inputs.pq2_rows(90 + N % 97, N, K)
    xn = pq_inputs.activations(91 + K % 89, 1, K, act_dt, outlier_rate=0.001)
    layer = w2_layer(dev, raw, K, act_dt, ag, 2)
    assert pq.pq_plan(layer.desc, 1, 152)["variant"] == pq.PQ_VARIANT_W2_GEMV_FUSED
    x = to_dev(xn, dev, DT[act_dt])
    got = bits_of(layer(x))
    ref = O.w2a8_linear(xn, act_dt, raw, ag)
    assert o8_error(got, ref, act_dt) <= TOL
    assert exact_fraction(got, ref, act_dt) >= 0.97, rel_rms(got, ref, act_dt)
    act = layer.quantize_act(x)
    assert np.array_equal(bits_of(layer.run_act(act, 1)), got)
    layer.close()


@pytest.mark.parametrize("M,N,K,ag", [(3, 72, 4096, 4096), (8, 136, 1152, 128), (12, 40, 11008, 11008),
                                      (16, 200, 1280, 128)])
def test_w2_bf16_decode_equals_int8_decode(dev, M, N, K, ag):
    # both tensor-core decodes form the exact block sums, then the same fp32
    # scaling in the same order: identical bits (PQ2 code 3 included)
    raw = pq_inputs.pq2_rows(72 + M, N, K, allow_code3=True)
    x = to_dev(pq_inputs.activations(73 + M, M, K, "bf16"), dev, torch.bfloat16)
    layer = w2_layer(dev, raw, K, "bf16", ag, M)
    a = bits_of(layer(x, variant=pq.PQ_VARIANT_W2_GEMV_TC))
    b = bits_of(layer(x, variant=pq.PQ_VARIANT_W2_GEMV_BF))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("M,N,K,ag,act_dt", [
    (1, 72, 4096, 4096, "bf16"),
    (2, 200, 1280, 128, "bf16"),     # three slices; the last one block short of a full 4
    (5, 88, 1152, 128, "f16"),
    (8, 56, 640, 640, "bf16"),       # two slices of 4 and 1 blocks
    (9, 40, 11008, 11008, "bf16"),   # eight slices of 12 blocks, the last of 2
    (12, 1000, 2048, 2048, "f16"),
    (16, 24, 128, 128, "bf16"),      # one CTA per cluster
    (16, 4104, 4096, 4096, "bf16"),  # 257 strips, 3 per warp
    (16, 24, 24576, 24576, "bf16"),  # the longest row the cluster holds
])
def test_w2_cluster_decode_parity(dev, M, N, K, ag, act_dt):
    raw = pq_inputs.pq2_rows(150 + M, N, K, allow_code3=(M == 5))
    x = pq_inputs.activations(160 + M, M, K, act_dt)
    layer = w2_layer(dev, raw, K, act_dt, ag, 16)
    xd = to_dev(x, dev, DT[act_dt])
    got = [bits_of(layer(xd, variant=pq.PQ_VARIANT_W2_GEMV_CL)) for _ in range(2)]
    assert np.array_equal(got[0], got[1])          # fixed-order slice sums: bit-identical
    ref = O.w2a8_linear(x, act_dt, raw, ag)
    assert o8_error(got[0], ref, act_dt) <= TOL
    assert exact_fraction(got[0], ref, act_dt) >= 0.97, rel_rms(got[0], ref, act_dt)


@pytest.mark.parametrize("M,N,K,ag", [(3, 72, 512, 512), (8, 136, 384, 128), (12, 40, 256, 256),
                                      (16, 200, 512, 128), (1, 24, 128, 128)])
def test_w2_cluster_decode_equals_int8_decode(dev, M, N, K, ag):
    # K <= 512: one K slice in both decodes, so the same exact block sums
    # (the cluster kernel's 1024 + 4^t c operands against the int8 codes),
    # the same fp32 scaling in the same order: identical bits
    raw = pq_inputs.pq2_rows(170 + M, N, K, allow_code3=True)
    x = to_dev(pq_inputs.activations(171 + M, M, K, "bf16"), dev, torch.bfloat16)
    layer = w2_layer(dev, raw, K, "bf16", ag, 16)
    a = bits_of(layer(x, variant=pq.PQ_VARIANT_W2_GEMV_TC))
    b = bits_of(layer(x, variant=pq.PQ_VARIANT_W2_GEMV_CL))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("ag", [512, 128])
def test_w2_cluster_decode_extreme_block_sums(dev, ag):
    # The cluster decode's fp16 operands make every block sum an integer up
    # to 32 * 127 * (1024 + 256 + 64 + 16) + 128 * 3 * 127 = 5575552 in
    # magnitude (all codes 3 against q = +-127), exact only if the tensor
    # cores keep it in fp32 without loss: rows of all-3, all-2, all-0 and
    # mixed codes against full-scale activations of one sign and of
    # alternating signs, bit for bit against the int8 decode (K = 512: one K
    # slice in both, the same scaling order).
    N, K, M = 64, 512, 16
    raw = pq_inputs.pq2_rows(180, N, K, allow_code3=True).reshape(N, K // 128, 34)
    fills = [0xFF, 0xAA, 0x00, 0x55, 0xEE, 0x33]
    for r, f in enumerate(fills):
        raw[r, :, 2:] = f
    raw = np.ascontiguousarray(raw.reshape(N, -1))
    x = np.zeros((M, K), dtype=np.float32)
    x[0] = 1.0
    x[1] = -1.0
    x[2] = np.where(np.arange(K) % 2 == 0, 1.0, -1.0)
    x[3] = np.where((np.arange(K) // 4) % 2 == 0, 1.0, -1.0)
    x[4:] = pq_inputs.rng(181).normal(0.0, 1.0, size=(M - 4, K))
    xd = torch.from_numpy(x).to(dev).to(torch.bfloat16)
    layer = w2_layer(dev, raw, K, "bf16", ag, 16)
    a = bits_of(layer(xd, variant=pq.PQ_VARIANT_W2_GEMV_TC))
    b = bits_of(layer(xd, variant=pq.PQ_VARIANT_W2_GEMV_CL))
    assert np.array_equal(a, b)
    ref = O.w2a8_linear(bits_of(xd), "bf16", raw, ag)
    assert o8_error(b, ref, "bf16") <= TOL


def test_w2_cluster_decode_refuses_long_rows(dev):
    K = 24704                                  # 193 blocks: slices of 28 > 24
    layer = w2_layer(dev, pq_inputs.pq2_rows(5, 16, K), K, "bf16", K, 4)
    x = torch.zeros((2, K), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pq.PQError):
        layer(x, variant=pq.PQ_VARIANT_W2_GEMV_CL)


def test_w2_fused_equals_prepass(dev):
    K, N, M = 2048, 96, 3
    raw = pq_inputs.pq2_rows(70, N, K)
    x = to_dev(pq_inputs.activations(71, M, K, "bf16"), dev, torch.bfloat16)
    layer = w2_layer(dev, raw, K, "bf16", 128, M)
    a = bits_of(layer(x, variant=pq.PQ_VARIANT_W2_GEMV_FUSED))
    b = bits_of(layer(x, variant=pq.PQ_VARIANT_W2_GEMV))
    assert np.array_equal(a, b)


# ------------------------------------------------------------ failures ---

def test_device_status_expiry_and_clear(dev):
    K = 256
    layer = w2_layer(dev, pq_inputs.pq2_rows(1, 16, K), K, "bf16", 128, 1)
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK
    pq.pq_debug_expire_wait(layer.handle, 1000)
    assert pq.pq_device_status(layer.handle) == pq.PQ_ERR_DEVICE_TIMEOUT
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK
    # the context is still usable
    x = to_dev(pq_inputs.activations(1, 1, K, "bf16"), dev, torch.bfloat16)
    layer(x)
    torch.cuda.synchronize()


def test_linear_refusals(dev):
    K, N = 256, 32
    layer = w4_layer(dev, pq_inputs.w4_frame(1, K, N, 0.002, 0.01), "bf16", 2)
    x = torch.zeros((4, K), dtype=torch.bfloat16, device=dev)
    y = torch.empty((4, N), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear(x, layer.handle, y, 3)
    assert e.value.status == pq.PQ_ERR_SHAPE
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear(x.data_ptr() + 2, layer.handle, y, 1)
    assert e.value.status == pq.PQ_ERR_ALIGN
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear_variant(x, layer.handle, y, 1, pq.PQ_VARIANT_W2_GEMV)
    assert e.value.status == pq.PQ_ERR_UNSUPPORTED


def test_graph_replay_reads_new_inputs(dev):
    # a captured call must consume the activations present at replay time
    K, N, M = 1024, 128, 1
    fr = pq_inputs.w4_frame(80, K, N, 0.002, 0.01, True, "scatter")
    layer = w4_layer(dev, fr, "bf16", M)
    raw = pq_inputs.pq2_rows(81, N, K)
    layer2 = w2_layer(dev, raw, K, "bf16", K, M)
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    y2 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer(x, out=y, stream=s)
        layer2(x, out=y2, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer(x, out=y, stream=s)
        layer2(x, out=y2, stream=s)
    for seed in (82, 83):
        xn = pq_inputs.activations(seed, M, K, "bf16")
        x.copy_(to_dev(xn, dev, torch.bfloat16))
        y.fill_(float("nan"))
        y2.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref = O.w4a16_linear(xn, "bf16", fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
        assert o8_error(bits_of(y), ref, "bf16") <= TOL
        assert o8_error(bits_of(y2), O.w2a8_linear(xn, "bf16", raw, K), "bf16") <= TOL
