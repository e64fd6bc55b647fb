"""The benchmark configurations at full size, GPU against the CPU oracle.

* W4A16 GEMV M=1, K=N=4096, fp16, symmetric, seed 0 (full output);
* ternary W2A8 GEMV M=1 at (N,K) = (4096,4096), (11008,4096), (4096,11008),
  bf16, per-row activation scale (full output) plus the exact block sums of
  the first 64 rows;
* W4A16 with explicit zero points and act order, M in {1,4,16}, K=5120,
  N in {5120, 27648}, bf16 (512 sampled output columns, the oracle restricted
  to them).
The launch path is pq_linear's own dispatch, as the benchmark times it.
"""
from __future__ import annotations

import numpy as np
import pytest

import pq_inputs
from oracle import pq_oracle as O
from tests.helpers import TOL, bits_of, exact_fraction, o8_error, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_weight_quantized_pq_gb300 as pq  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pq.build()
    return torch.device("cuda:0")


def test_w4a16_gemv_m1_4096(dev):
    K = N = 4096
    fr = pq_inputs.w4_frame(0, K, N, 0.002, 0.01)
    x = pq_inputs.activations(0, 1, K, "f16")
    layer = pq.QuantizedLinear.from_w4(to_dev(fr["qweight"], dev), to_dev(fr["scales"], dev),
                                       act_dtype="f16", max_m=1)
    got = bits_of(layer(to_dev(x, dev, torch.float16)))
    ref = O.w4a16_linear(x, "f16", fr["qweight"], fr["scales"])
    assert o8_error(got, ref, "f16") <= TOL
    assert exact_fraction(got, ref, "f16") >= 0.97


@pytest.mark.parametrize("N,K", [(4096, 4096), (11008, 4096), (4096, 11008)])
def test_w2a8_gemv_m1(dev, N, K):
    raw = pq_inputs.pq2_rows(1, N, K)
    x = pq_inputs.activations(1, 1, K, "bf16")
    layer = pq.QuantizedLinear.from_pq2(to_dev(raw, dev), K, act_dtype="bf16", act_group=K, max_m=1)
    xd = to_dev(x, dev, torch.bfloat16)
    got = bits_of(layer(xd))
    ref = O.w2a8_linear(x, "bf16", raw, K)
    assert o8_error(got, ref, "bf16") <= TOL
    assert exact_fraction(got, ref, "bf16") >= 0.97
    S = torch.empty((1, N, K // 128), dtype=torch.int32, device=dev)
    pq.pq_debug_w2a8_group_sums(xd, layer.handle, S, 1)
    q, _ = O.quantize_act(x, "bf16", K)
    S_ref = O.w2a8_group_sums(q, O.pq2_values(raw[:64]))
    assert np.array_equal(S.cpu().numpy()[:, :64].astype(np.int64), S_ref)


@pytest.mark.parametrize("N", [5120, 27648])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_w4a16_asym_act_order(dev, M, N):
    K = 5120
    fr = pq_inputs.w4_frame(2, K, N, 0.001, 0.01, zero_points=True, act_order="scatter")
    x = pq_inputs.activations(2 + M, M, K, "bf16")
    layer = pq.QuantizedLinear.from_w4(to_dev(fr["qweight"], dev), to_dev(fr["scales"], dev),
                                       to_dev(fr["zeros"], dev), fr["g_idx"], act_dtype="bf16", max_m=16)
    got = bits_of(layer(to_dev(x, dev, torch.bfloat16)))
    cols = np.sort(np.random.default_rng(N + M).choice(N, 512, replace=False))
    ref = O.w4a16_linear_columns(x, "bf16", fr["qweight"], fr["scales"], fr["zeros"], fr["g_idx"], cols)
    full_rms = None
    err = o8_error(got[:, cols], ref, "bf16")
    assert err <= TOL, (err, full_rms)
    assert exact_fraction(got[:, cols], ref, "bf16") >= 0.97
