"""GPU parity of the MLX affine 4-bit decode (w = s * q + b per 64 inputs;
"qwen CUDA: --prompt-precision int8 ... #1176") against the CPU oracle.

Bit-exact: the prepared planes dequantised by pq_debug_unpack equal the
oracle's exact s * q + b rounded once to fp32.  Outputs: the tests/helpers.py
metric within 2e-3 and nearly all outputs equal to the correctly rounded
oracle value -- decode at M = 1..16 (whole rows, split-K), the tensor-core
GEMM above, on ragged shapes and at prefill sizes on sampled outputs.
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


def affine_layer(dev, L, act, max_m):
    return pq.QuantizedLinear.from_affine4(to_dev(L["wq"], dev), to_dev(L["scales"], dev), to_dev(L["biases"], dev),
                                          act_dtype=act, max_m=max_m)


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(72, 640), (200, 1024)])
def test_affine_unpack_bit_exact(dev, act, N, K):
    L = pq_inputs.affine4_layer(1, N, K, act)
    layer = affine_layer(dev, L, act, 1)
    w = torch.empty((K, N), dtype=torch.float32, device=dev)
    pq.pq_debug_unpack(layer.handle, w)
    torch.cuda.synchronize()
    ref = O.affine4_dequant(L["wq"], L["scales"], L["biases"], act).T.astype(np.float32)
    assert np.array_equal(w.cpu().numpy(), ref)
    layer.close()


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16])
@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(200, 640), (96, 1024), (72, 4096)])
def test_affine_gemv_parity(dev, M, act, N, K):
    """Whole-row kernel for M <= 4, split-K (slices of four 128-input blocks,
    a ragged last slice at K = 640) for M = 5..16, its slices (8 or fewer)
    added inside a thread-block cluster for M <= 8, by a second launch above."""
    L = pq_inputs.affine4_layer(10 + M, N, K, act)
    x = pq_inputs.activations(20 + M, M, K, act)
    layer = affine_layer(dev, L, act, 16)
    plan = pq.pq_plan(layer.desc, M, 152)
    assert plan["variant"] == pq.PQ_VARIANT_W4_GEMV and plan["launches"] == (1 if M <= 8 else 2)
    got = bits_of(layer(to_dev(x, dev, DT[act])))
    ref = O.affine4_linear(x, act, L["wq"], L["scales"], L["biases"], act)
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK
    assert o8_error(got, ref, act) <= TOL
    assert exact_fraction(got, ref, act) >= 0.97, rel_rms(got, ref, act)
    layer.close()


@pytest.mark.parametrize("M,N,K", [(1, 40, 76544), (2, 72, 20480), (16, 1000, 4096)])
def test_affine_split_k_rows(dev, M, N, K):
    """Rows too long for the whole-row kernel's shared memory (one token past
    K = 76416, two tokens of K = 20480) take split-K; and 63 strips of 16
    rows over a few CTAs per slice.  Repeated calls agree bit for bit.  Up to
    8 slices (K <= 4096) at M <= 8 add their sums inside a cluster, else a
    second launch does."""
    L = pq_inputs.affine4_layer(30 + M, N, K, "bf16")
    x = pq_inputs.activations(31 + M, M, K, "bf16")
    layer = affine_layer(dev, L, "bf16", 16)
    assert pq.pq_plan(layer.desc, M, 152)["launches"] == (2 if K > 4096 or M > 8 else 1)
    xd = to_dev(x, dev, torch.bfloat16)
    got = bits_of(layer(xd))
    assert np.array_equal(got, bits_of(layer(xd)))
    ref = O.affine4_linear(x, "bf16", L["wq"], L["scales"], L["biases"], "bf16")
    assert o8_error(got, ref, "bf16") <= TOL
    assert exact_fraction(got, ref, "bf16") >= 0.97, rel_rms(got, ref, "bf16")
    layer.close()


@pytest.mark.parametrize("M", [17, 129, 300])
@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(200, 640), (264, 1024)])
def test_affine_gemm_parity(dev, M, act, N, K):
    """The tensor-core GEMM: one 64-group per k-step, s * dot + b * (sum of
    x) per group in the epilogue; ragged M and N, several 256-token tiles."""
    L = pq_inputs.affine4_layer(40 + M, N, K, act)
    x = pq_inputs.activations(41 + M, M, K, act, outlier_rate=0.001)
    layer = affine_layer(dev, L, act, 512)
    assert pq.pq_plan(layer.desc, M, 152)["variant"] == pq.PQ_VARIANT_W4_GEMM
    got = bits_of(layer(to_dev(x, dev, DT[act])))
    ref = O.affine4_linear(x, act, L["wq"], L["scales"], L["biases"], act)
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK
    assert o8_error(got, ref, act) <= TOL, rel_rms(got, ref, act)
    assert exact_fraction(got, ref, act) >= 0.97
    layer.close()


@pytest.mark.parametrize("M,N,K", [(256, 4096, 4096), (2048, 4096, 4096), (2048, 11008, 4096)])
def test_affine_gemm_shared_tiles(dev, M, N, K):
    """Prefill shapes whose last tiles are shared out by groups (parts added
    by the fixup launch or by the tile's owner), checked on sampled rows and
    columns: the oracle runs on the sampled output rows of the layer."""
    L = pq_inputs.affine4_layer(50 + M, N, K, "bf16")
    xn = pq_inputs.activations(51 + M, M, K, "bf16", outlier_rate=0.001)
    layer = affine_layer(dev, L, "bf16", 2048)
    assert pq.pq_plan(layer.desc, M, torch.cuda.get_device_properties(dev).multi_processor_count)["k_split"] > 1
    x = to_dev(xn, dev, torch.bfloat16)
    a = bits_of(layer(x))
    assert np.array_equal(a, bits_of(layer(x)))
    rng = np.random.default_rng(M + N)
    rows = np.sort(rng.choice(M, 192, replace=False))
    cols = np.sort(rng.choice(N, 256, replace=False))
    ref = O.affine4_linear(xn[rows], "bf16", L["wq"][cols], L["scales"][cols], L["biases"][cols], "bf16")
    sub = a[rows][:, cols]
    assert o8_error(sub, ref, "bf16") <= TOL, rel_rms(sub, ref, "bf16")
    assert exact_fraction(sub, ref, "bf16") >= 0.97
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK
    layer.close()


def test_affine_gemm_matches_gemv_at_16(dev):
    """At M = 16 both variants run; they agree with the oracle and closely
    with each other (different summation orders)."""
    L = pq_inputs.affine4_layer(60, 136, 1024, "bf16")
    x = pq_inputs.activations(61, 16, 1024, "bf16")
    layer = affine_layer(dev, L, "bf16", 64)
    xd = to_dev(x, dev, torch.bfloat16)
    ref = O.affine4_linear(x, "bf16", L["wq"], L["scales"], L["biases"], "bf16")
    for v in (pq.PQ_VARIANT_W4_GEMV, pq.PQ_VARIANT_W4_GEMM):
        got = bits_of(layer(xd, variant=v))
        assert o8_error(got, ref, "bf16") <= TOL, v
        assert exact_fraction(got, ref, "bf16") >= 0.97, v
    layer.close()


def test_affine_refusals(dev):
    """M above max_m, and the GEMM variant on a layer whose workspace holds no
    sums of x (max_m <= 16), are refused before any launch."""
    L = pq_inputs.affine4_layer(3, 64, 512, "bf16")
    layer = affine_layer(dev, L, "bf16", 8)
    x = torch.zeros((9, 512), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pq.PQError) as e:
        layer(x)
    assert e.value.status == pq.PQ_ERR_SHAPE
    with pytest.raises(pq.PQError) as e:
        layer(x[:8], variant=pq.PQ_VARIANT_W4_GEMM)
    assert e.value.status == pq.PQ_ERR_UNSUPPORTED
    layer.close()
