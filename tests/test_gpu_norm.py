"""GPU parity of the quantised-activation entry points against the CPU oracle.

The fused producer (pq_norm_quantize: residual add, RMSNorm, random-sign
Hadamard, group quantiser; PRISM "E. Keeping preparation data close to
compute", Test 18) fixes every fp32 operation and the order of its one
reduction, so its results are compared bit for bit with ``oracle.norm_quantize``:
the residual output, the normalised row, the int8 codes, their scales and
block sums.  The layer run on the caller's buffer (pq_linear_act) is checked
against the oracle's ternary output on the transformed row, and bitwise
against pq_linear run on that row where both take the same kernel.
"""
from __future__ import annotations

import numpy as np
import pytest

import pq_inputs
from oracle import pq_oracle as O
from tests.helpers import TOL, bits_of, o8_error, to_dev

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


def w2_layer(dev, raw, K, act, ag, max_m):
    return pq.QuantizedLinear.from_pq2(to_dev(raw, dev), K, act_dtype=act, act_group=ag, max_m=max_m)


def unpack_act(layer, act, M, K, ag, dev):
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    xs = torch.empty((M, K // ag), dtype=torch.float32, device=dev)
    sq = torch.empty((M, K // 128), dtype=torch.int32, device=dev)
    pq.pq_debug_act_unpack(act, act.numel(), layer.handle, M, q, xs, sq)
    torch.cuda.synchronize()
    return q.cpu().numpy(), xs.cpu().numpy(), sq.cpu().numpy()


# (M, K, fmt, residual, unit_offset, had_block, act_group)
CASES = [
    (1, 4096, "bf16", True, True, 1024, 128),
    (1, 11008, "bf16", True, True, 256, 128),       # last 2048-chunk partial
    (2, 2304, "f16", False, False, 0, 2304),         # one group per row, no transform
    (3, 128, "bf16", True, False, 128, 128),         # K below the lane count
    (16, 5120, "bf16", True, True, 1024, 128),
    (17, 4096, "bf16", True, True, 1024, 128),       # first M on the GEMM form
    (40, 2304, "f16", True, True, 256, 2304),
    (300, 4096, "bf16", False, True, 512, 128),
    (1, 65536, "bf16", True, True, 1024, 128),      # the longest row (128 KB in shared memory)
    (4, 256, "bf16", False, True, 2, 128),          # transform in registers only
    (5, 384, "f16", True, True, 64, 384),            # register and shuffle stages
    (20, 1024, "f16", True, False, 128, 128),        # fp16 codes on the GEMM form
]


@pytest.mark.parametrize("M,K,fmt,residual,unit,B,ag", CASES)
def test_norm_quantize_bit_exact(dev, M, K, fmt, residual, unit, B, ag):
    d = pq_inputs.norm_inputs(100 + M, M, K, fmt, unit_offset=unit, residual=residual)
    eps = 1e-6
    ref = O.norm_quantize(d["h"], d["r"], d["gamma"], fmt, eps, unit, d["signs"], B, ag)
    layer = w2_layer(dev, pq_inputs.pq2_rows(5, 48, K), K, fmt, ag, max(M, 2))
    h = to_dev(d["h"], dev, DT[fmt])
    r = to_dev(d["r"], dev, DT[fmt]) if residual else None
    r_out = torch.empty_like(h) if residual else None
    norm_out = torch.empty_like(h)
    act = layer.norm_quantize(h, to_dev(d["gamma"], dev, DT[fmt]), eps, r=r, r_out=r_out, norm_out=norm_out,
                              signs=to_dev(d["signs"], dev) if B else None, unit_offset=unit, had_block=B)
    q, xs, sq = unpack_act(layer, act, M, K, ag, dev)
    assert pq.pq_device_status(layer.handle) == pq.PQ_OK
    if residual:
        assert (bits_of(r_out) == ref["r_out"]).all()
    assert (bits_of(norm_out) == ref["norm"]).all()
    assert (q == ref["q"]).all()
    assert (xs.view(np.uint32) == ref["xs"].view(np.uint32)).all()
    assert (sq == ref["sq"]).all()

    # the layer on the caller's buffer: the oracle's output for the row v
    y = layer.run_act(act, M)
    torch.cuda.synchronize()
    raw = pq_inputs.pq2_rows(5, 48, K)
    y_ref = O.w2a8_linear(ref["v"], fmt, raw, ag)
    assert o8_error(bits_of(y), y_ref, fmt) <= TOL
    layer.close()


def test_residual_in_place(dev):
    # r_out = r: the residual stream updated in place
    M, K = 4, 4096
    d = pq_inputs.norm_inputs(7, M, K, "bf16")
    ref = O.norm_quantize(d["h"], d["r"], d["gamma"], "bf16", 1e-5, True, d["signs"], 1024, 128)
    layer = w2_layer(dev, pq_inputs.pq2_rows(6, 32, K), K, "bf16", 128, M)
    h = to_dev(d["h"], dev, torch.bfloat16)
    r = to_dev(d["r"], dev, torch.bfloat16)
    act = layer.norm_quantize(h, to_dev(d["gamma"], dev, torch.bfloat16), 1e-5, r=r, r_out=r,
                              signs=to_dev(d["signs"], dev), unit_offset=True, had_block=1024)
    q, xs, sq = unpack_act(layer, act, M, K, 128, dev)
    assert (bits_of(r) == ref["r_out"]).all()
    assert (q == ref["q"]).all()
    layer.close()


@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 12, 16, 40])
def test_quantize_act_matches_pq_linear(dev, M):
    # one quantisation, two layers of different N; each equals pq_linear on x
    K = 4096
    x = to_dev(pq_inputs.activations(9, M, K, "bf16", outlier_rate=0.001), dev, torch.bfloat16)
    a = w2_layer(dev, pq_inputs.pq2_rows(7, 200, K), K, "bf16", 128, max(M, 2))
    b = w2_layer(dev, pq_inputs.pq2_rows(8, 72, K), K, "bf16", 128, max(M, 2))
    act = a.quantize_act(x)
    q, xs, sq = unpack_act(a, act, M, K, 128, dev)
    q_ref, xs_ref = O.quantize_act(pq_inputs.activations(9, M, K, "bf16", outlier_rate=0.001), "bf16", 128)
    assert (q == q_ref).all() and (xs.view(np.uint32) == xs_ref.view(np.uint32)).all()
    for layer in (a, b):
        y_act = layer.run_act(act, M)
        y = layer(x)
        torch.cuda.synchronize()
        assert (bits_of(y_act) == bits_of(y)).all()
    a.close()
    b.close()


def test_act_refusals(dev):
    K = 1024
    layer = w2_layer(dev, pq_inputs.pq2_rows(1, 16, K), K, "bf16", 128, 4)
    h = torch.zeros((2, K), dtype=torch.bfloat16, device=dev)
    g = torch.zeros(K, dtype=torch.bfloat16, device=dev)
    act = layer.act_buffer(2)
    with pytest.raises(pq.PQError) as e:
        pq.pq_norm_quantize(h, None, pq.pq_norm(g.data_ptr(), None, 0.0, 0, 0), layer.handle, None, None,
                            act, act.numel(), 2)
    assert e.value.status == pq.PQ_ERR_INVALID_ARG and "eps" in str(e.value)
    with pytest.raises(pq.PQError) as e:
        layer.norm_quantize(h, g, 1e-6, had_block=96, act=act)
    assert e.value.status == pq.PQ_ERR_INVALID_ARG and "had_block" in str(e.value)
    with pytest.raises(pq.PQError) as e:
        layer.norm_quantize(h, g, 1e-6, had_block=2048, act=act)
    assert e.value.status == pq.PQ_ERR_INVALID_ARG
    with pytest.raises(pq.PQError) as e:
        pq.pq_quantize_act(h, layer.handle, act, act.numel() - 1, 2)
    assert e.value.status == pq.PQ_ERR_BUFFER_TOO_SMALL
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear_act(act.data_ptr() + 16, act.numel(), layer.handle, h, 2)
    assert e.value.status == pq.PQ_ERR_ALIGN
    with pytest.raises(pq.PQError) as e:
        pq.pq_quantize_act(h, layer.handle, act, act.numel(), 5)
    assert e.value.status == pq.PQ_ERR_SHAPE
    # the readers check the buffer's size too
    pq.pq_quantize_act(h, layer.handle, act, act.numel(), 2)
    with pytest.raises(pq.PQError) as e:
        pq.pq_linear_act(act, act.numel() - 1, layer.handle, h, 2)
    assert e.value.status == pq.PQ_ERR_BUFFER_TOO_SMALL
    q = torch.empty((2, K), dtype=torch.int8, device=dev)
    xs = torch.empty((2, K // 128), dtype=torch.float32, device=dev)
    sq = torch.empty((2, K // 128), dtype=torch.int32, device=dev)
    with pytest.raises(pq.PQError) as e:
        pq.pq_debug_act_unpack(act, act.numel() - 1, layer.handle, 2, q, xs, sq)
    assert e.value.status == pq.PQ_ERR_BUFFER_TOO_SMALL
    layer.close()
