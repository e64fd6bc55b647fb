"""GPU parity of the MLX affine 4-bit decode (w = s * q + b per 64 inputs;
"qwen CUDA: --prompt-precision int8 ... #1176") against the CPU oracle.

Bit-exact: the prepared planes dequantised by pq_debug_unpack equal the
oracle's exact s * q + b rounded once to fp32.  Outputs: the tests/helpers.py
metric within 2e-3 and nearly all outputs equal to the correctly rounded
oracle value, for M = 1..4 on ragged shapes.
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


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(200, 640), (96, 1024), (72, 4096)])
def test_affine_gemv_parity(dev, M, act, N, K):
    L = pq_inputs.affine4_layer(10 + M, N, K, act)
    x = pq_inputs.activations(20 + M, M, K, act)
    layer = affine_layer(dev, L, act, 4)
    got = bits_of(layer(to_dev(x, dev, DT[act])))
    ref = O.affine4_linear(x, act, L["wq"], L["scales"], L["biases"], act)
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK
    assert o8_error(got, ref, act) <= TOL
    assert exact_fraction(got, ref, act) >= 0.97, rel_rms(got, ref, act)
    layer.close()


def test_affine_refuses_larger_m(dev):
    L = pq_inputs.affine4_layer(3, 64, 512, "bf16")
    layer = affine_layer(dev, L, "bf16", 8)
    x = torch.zeros((5, 512), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pq.PQError) as e:
        layer(x)
    assert e.value.status == pq.PQ_ERR_UNSUPPORTED
    layer.close()
