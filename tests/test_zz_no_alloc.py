"""The allocation-free ternary decode entry point, through the C ABI.

pq_linear_w2a8_static serves callers that may not allocate device memory
(a host framework that owns every buffer, or a caller that cannot accept an
allocation's synchronisation): its scratch is a fixed array inside the
library.  It must give the same outputs as the ordinary entry point
(pq_linear with the pre-pass + GEMV variant, which uses the handle's
workspace), call after call, since every call reuses the same array.

This file is collected last on purpose, and it works both alone in a fresh
process and after the other GPU tests.
"""
from __future__ import annotations

import numpy as np
import pytest

import pq_inputs
from tests.helpers import TOL, bits_of, o8_error, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_weight_quantized_pq_gb300 as pq  # noqa: E402
from oracle import pq_oracle as O  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pq.build()
    return torch.device("cuda:0")


# (the K = 32768 case stages a 64 KB activation row: the quantiser's shared
# memory attribute must be set on the device first)
@pytest.mark.parametrize("M,N,K,ag", [(1, 200, 4096, 4096), (4, 136, 2048, 128), (16, 72, 1280, 1280),
                                      (1, 64, 32768, 32768)])
def test_static_matches_workspace_entry_point(dev, M, N, K, ag):
    raw = pq_inputs.pq2_rows(900 + M, N, K)
    layer = pq.QuantizedLinear.from_pq2(to_dev(raw, dev), K, act_dtype="bf16", act_group=ag, max_m=16)
    for call, seed in enumerate((910 + M, 920 + M)):      # two calls in a row, different inputs
        xn = pq_inputs.activations(seed, M, K, "bf16")
        x = to_dev(xn, dev, torch.bfloat16)
        ref = bits_of(layer(x, variant=pq.PQ_VARIANT_W2_GEMV))
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        pq.pq_linear_w2a8_static(x, layer.handle, y, M)
        torch.cuda.synchronize()
        got = bits_of(y)
        assert o8_error(got, O.bf16_bits_to_f64(ref), "bf16") <= TOL, call
        assert o8_error(got, O.w2a8_linear(xn, "bf16", raw, ag), "bf16") <= TOL, call
        assert np.array_equal(got, ref), call


def test_static_rejects_sizes_beyond_its_array(dev):
    # M*K = 131072 needs 139264 bytes of scratch, more than the 131072 the
    # library reserves, although the ordinary entry point runs this size
    K = 8192
    layer = pq.QuantizedLinear.from_pq2(to_dev(pq_inputs.pq2_rows(930, 16, K), dev), K, act_dtype="bf16",
                                        act_group=128, max_m=16)
    x = torch.zeros((16, K), dtype=torch.bfloat16, device=dev)
    y = torch.empty((16, 16), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear_w2a8_static(x, layer.handle, y, 16)
    assert e.value.status == pq.PQ_ERR_BUFFER_TOO_SMALL
    assert "static scratch" in str(e.value)
    layer(x, out=y, variant=pq.PQ_VARIANT_W2_GEMV)      # the workspace entry point accepts it
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear_w2a8_static(x, layer.handle, y, 17)
    assert e.value.status == pq.PQ_ERR_SHAPE
    # M beyond the handle's max_m is refused, as by pq_linear
    small = pq.QuantizedLinear.from_pq2(to_dev(pq_inputs.pq2_rows(931, 16, 1024), dev), 1024, act_dtype="bf16",
                                        act_group=128, max_m=4)
    x = torch.zeros((5, 1024), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear_w2a8_static(x, small.handle, y, 5)
    assert e.value.status == pq.PQ_ERR_SHAPE and "max_m" in str(e.value)
