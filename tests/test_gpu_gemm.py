"""GPU parity of the tensor-core prefill GEMM (TMA + tcgen05/TMEM) against
the CPU oracle, through the C ABI.

Small shapes cover several 128-token and 256-row tiles with ragged tails in
M and N, act order, explicit zero points, fp16 and bf16, and both ternary
activation groupings; the prefill configurations (M in {512, 2048, 3314},
K=4096/N=14336 and K=14336/N=4096, bf16 activations with 0.1% outliers x20)
are checked on sampled rows and columns, the oracle restricted to them.
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


def w4_layer(dev, fr, act, max_m):
    return pq.QuantizedLinear.from_w4(
        to_dev(fr["qweight"], dev), to_dev(fr["scales"], dev),
        None if fr["zeros"] is None else to_dev(fr["zeros"], dev), fr["g_idx"], act_dtype=act, max_m=max_m)


@pytest.mark.parametrize("M", [5, 17, 129, 300])
@pytest.mark.parametrize("N,K,zp,act,act_dt", [
    (200, 640, False, None, "bf16"), (512, 1024, True, None, "f16"), (264, 384, True, "scatter", "bf16")])
def test_w4_gemm_parity(dev, M, N, K, zp, act, act_dt):
    fr = pq_inputs.w4_frame(100 + M, K, N, 0.002, 0.01, zp, act)
    x = pq_inputs.activations(200 + M, M, K, act_dt, outlier_rate=0.001)
    layer = w4_layer(dev, fr, act_dt, 512)
    got = bits_of(layer(to_dev(x, dev, DT[act_dt]), variant=pq.PQ_VARIANT_W4_GEMM))
    ref = O.w4a16_linear(x, act_dt, fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"])
    assert o8_error(got, ref, act_dt) <= TOL, rel_rms(got, ref, act_dt)
    assert exact_fraction(got, ref, act_dt) >= 0.97


@pytest.mark.parametrize("M,N,K,ag,code3", [
    (20, 200, 1024, 128, False), (257, 520, 384, 384, True), (130, 256, 640, 128, False)])
def test_w2_gemm_parity(dev, M, N, K, ag, code3):
    raw = pq_inputs.pq2_rows(300 + M, N, K, allow_code3=code3)
    x = pq_inputs.activations(310 + M, M, K, "bf16")
    layer = pq.QuantizedLinear.from_pq2(to_dev(raw, dev), K, act_dtype="bf16", act_group=ag, max_m=512)
    got = bits_of(layer(to_dev(x, dev, torch.bfloat16), variant=pq.PQ_VARIANT_W2_GEMM))
    ref = O.w2a8_linear(x, "bf16", raw, ag)
    assert o8_error(got, ref, "bf16") <= TOL, rel_rms(got, ref, "bf16")
    assert exact_fraction(got, ref, "bf16") >= 0.97


def test_gemm_deterministic_and_dispatch(dev):
    K, N, M = 512, 300, 100
    fr = pq_inputs.w4_frame(7, K, N, 0.002, 0.01, True, None)
    layer = w4_layer(dev, fr, "bf16", M)
    x = to_dev(pq_inputs.activations(8, M, K, "bf16"), dev, torch.bfloat16)
    a = bits_of(layer(x))                        # dispatcher: M > 16 -> GEMM
    b = bits_of(layer(x, variant=pq.PQ_VARIANT_W4_GEMM))
    assert np.array_equal(a, b)
    assert pq.pq_plan(layer.desc, M, 152)["variant"] == pq.PQ_VARIANT_W4_GEMM
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK


@pytest.mark.parametrize("M,N,K,fmt", [(256, 512, 4096, "w4"), (256, 4096, 4096, "w4"), (300, 520, 2048, "w2"),
                                       (40, 136, 4096, "w4"), (2048, 4096, 4096, "w4"), (2048, 4096, 4096, "w2"),
                                       (300, 520, 2048, "w2g"), (2048, 4096, 4096, "w2g")])
def test_gemm_shared_tiles(dev, M, N, K, fmt):
    """Tiles whose 128-row groups are shared out over several CTAs (many per
    tile at small M: parts added by the fixup launch; two per tile at
    M = 2048: parts added in-kernel by the tile's owner).  Parts are added
    in CTA order, so repeated calls agree bit for bit.  Large cases are
    checked on sampled rows and columns."""
    xn = pq_inputs.activations(40 + M, M, K, "bf16")
    x = to_dev(xn, dev, torch.bfloat16)
    rng = np.random.default_rng(M + N)
    rows = np.arange(M) if M <= 512 else np.sort(rng.choice(M, 256, replace=False))
    cols = np.arange(N) if N <= 1024 else np.sort(rng.choice(N, 256, replace=False))
    if fmt == "w4":
        fr = pq_inputs.w4_frame(41 + M, K, N, 0.002, 0.01, True, None)
        layer = w4_layer(dev, fr, "bf16", 2048)
        variant = pq.PQ_VARIANT_W4_GEMM
        ref = O.w4a16_linear_columns(xn[rows], "bf16", fr["qweight"], fr["scales"], fr["zeros"], None, cols)
    else:
        # ternary, one activation scale per row ("w2") or per 128-input block ("w2g")
        ag = K if fmt == "w2" else 128
        raw = pq_inputs.pq2_rows(42 + M, N, K)
        layer = pq.QuantizedLinear.from_pq2(to_dev(raw, dev), K, act_dtype="bf16", act_group=ag, max_m=2048)
        variant = pq.PQ_VARIANT_W2_GEMM
        ref = O.w2a8_linear(xn[rows], "bf16", raw[cols], ag)
    assert pq.pq_plan(layer.desc, M, torch.cuda.get_device_properties(dev).multi_processor_count)["k_split"] > 1
    a = bits_of(layer(x, variant=variant))
    b = bits_of(layer(x, variant=variant))
    assert np.array_equal(a, b)
    sub = a[rows][:, cols]
    assert o8_error(sub, ref, "bf16") <= TOL, rel_rms(sub, ref, "bf16")
    assert exact_fraction(sub, ref, "bf16") >= 0.97
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK


def test_status_read_clears_shared_tile_flags(dev):
    """A GEMM launch that gives up a bounded wait can leave shared-tile flags
    raised in its workspace.  pq_device_status, when it reports an error,
    clears them.  Here every workspace byte is set to 0xFF (the status word
    then reads as an error, every flag as raised and every partial slot as
    NaN), the status is read once, and a launch whose tiles are shared by two
    CTAs (the owner adds the part after its flag) must match the oracle."""
    M, N, K = 2048, 4096, 4096
    fr = pq_inputs.w4_frame(61, K, N, 0.002, 0.01, False, None)
    layer = w4_layer(dev, fr, "bf16", M)
    plan = pq.pq_plan(layer.desc, M, torch.cuda.get_device_properties(dev).multi_processor_count)
    assert plan["k_split"] > 1 and plan["launches"] == 1      # shared tiles, owners add the parts
    layer.workspace.fill_(0xFF)
    torch.cuda.synchronize()
    assert pq.pq_device_status(layer.handle) != pq.PQ_OK
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK
    xn = pq_inputs.activations(62, M, K, "bf16", outlier_rate=0.001)
    got = bits_of(layer(to_dev(xn, dev, torch.bfloat16), variant=pq.PQ_VARIANT_W4_GEMM))
    rng = np.random.default_rng(63)
    rows = np.sort(rng.choice(M, 128, replace=False))
    cols = np.sort(rng.choice(N, 256, replace=False))
    ref = O.w4a16_linear_columns(xn[rows], "bf16", fr["qweight"], fr["scales"], None, None, cols)
    sub = got[rows][:, cols]
    assert o8_error(sub, ref, "bf16") <= TOL, rel_rms(sub, ref, "bf16")
    assert exact_fraction(sub, ref, "bf16") >= 0.97
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK


def test_gemm_matches_gemv_at_16(dev):
    K, N, M = 1024, 256, 16
    fr = pq_inputs.w4_frame(9, K, N, 0.002, 0.01, False, "scatter")
    layer = w4_layer(dev, fr, "bf16", M)
    xn = pq_inputs.activations(10, M, K, "bf16")
    x = to_dev(xn, dev, torch.bfloat16)
    a = bits_of(layer(x, variant=pq.PQ_VARIANT_W4_GEMM))
    b = bits_of(layer(x, variant=pq.PQ_VARIANT_W4_GEMV))
    ref = O.w4a16_linear(xn, "bf16", fr["qweight"], fr["scales"], None, fr["g_idx"])
    assert o8_error(a, ref, "bf16") <= TOL and o8_error(b, ref, "bf16") <= TOL
    assert (a == b).mean() >= 0.97


@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096)])
@pytest.mark.parametrize("M", [512, 2048, 3314])
def test_prefill_config_sampled(dev, M, K, N):
    fr = pq_inputs.w4_frame(0, K, N, 0.002, 0.01)
    x = pq_inputs.activations(3 + M, M, K, "bf16", outlier_rate=0.001, outlier_scale=20.0)
    layer = w4_layer(dev, fr, "bf16", M)
    got = bits_of(layer(to_dev(x, dev, torch.bfloat16)))
    rng = np.random.default_rng(M + K)
    cols = np.sort(rng.choice(N, 256, replace=False))
    rows = np.sort(rng.choice(M, min(M, 384), replace=False))
    ref = O.w4a16_linear_columns(x[rows], "bf16", fr["qweight"], fr["scales"], None, None, cols)
    sub = got[rows][:, cols]
    assert o8_error(sub, ref, "bf16") <= TOL
    assert exact_fraction(sub, ref, "bf16") >= 0.97
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK


@pytest.mark.parametrize("M", [256, 2048])
def test_ternary_prefill_sampled(dev, M):
    K, N = 4096, 11008
    raw = pq_inputs.pq2_rows(4, N, K)
    x = pq_inputs.activations(5 + M, M, K, "bf16")
    layer = pq.QuantizedLinear.from_pq2(to_dev(raw, dev), K, act_dtype="bf16", act_group=K, max_m=M)
    got = bits_of(layer(to_dev(x, dev, torch.bfloat16)))
    rng = np.random.default_rng(M)
    cols = np.sort(rng.choice(N, 256, replace=False))
    rows = np.sort(rng.choice(M, min(M, 256), replace=False))
    ref = O.w2a8_linear(x[rows], "bf16", raw[cols], K)
    sub = got[rows][:, cols]
    assert o8_error(sub, ref, "bf16") <= TOL
    assert exact_fraction(sub, ref, "bf16") >= 0.97
