"""The copy-only read probe (pq_probe_read) reads every 16-byte chunk of its
buffer exactly once: its XOR checksum of the 32-bit words equals the one
computed on the host, for sizes that leave ragged tails against the grid and
the per-thread unroll, in both launch modes and several grid sizes."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_weight_quantized_pq_gb300 as pq  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pq.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, 8650752, 23248896 + 16 * 37])
@pytest.mark.parametrize("ctas,dep", [(0, 0), (2, 1), (8, 0)])
def test_probe_reads_every_chunk_once(dev, nbytes, ctas, dep):
    rng = np.random.default_rng(nbytes % 1000 + ctas)
    host = rng.integers(0, 2 ** 32, nbytes // 4, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).to(dev)
    sink = torch.zeros(64, dtype=torch.int32, device=dev)
    pq.pq_probe_read(buf, nbytes, sink, ctas, dep)
    want = np.bitwise_xor.reduce(host)
    assert int(np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))) == int(want)
    # a second read folds the same checksums in again: zero
    pq.pq_probe_read(buf, nbytes, sink, ctas, dep)
    assert not sink.cpu().numpy().any()
