"""CPU oracle for the weight-only-quantized linear layer.

Test infrastructure: imported only by the tests, the smoke check and the
benchmark's CPU-baseline leg.  The CUDA library never uses it.
"""
from .pq_oracle import *  # noqa: F401,F403
