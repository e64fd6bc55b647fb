"""Shared test helpers: moving seeded inputs to the GPU and the float
comparison metric.

Metric for fp16/bf16 outputs (the 2e-3 bound is stated for the final output,
whose own rounding alone is up to half a unit in the last place, 2^-9 for
bf16, so the rounding of the output is excluded):

    err_i = max(0, |y_i - ref_i| - ulp(y_i)/2) / (|ref_i| + rms(ref row of i))

with ref the oracle's fp64 result; the run passes when max_i err_i <= 2e-3.
"""
from __future__ import annotations

import numpy as np

from oracle import pq_oracle as O

TOL = 2e-3
_P = {"f16": (11, -14), "bf16": (8, -126)}


def ulp(v: np.ndarray, fmt: str) -> np.ndarray:
    p, emin = _P[fmt]
    _, e = np.frexp(np.abs(v))
    e = np.maximum(e - 1, emin)
    return np.ldexp(1.0, e - (p - 1))


def o8_error(got_bits: np.ndarray, ref: np.ndarray, fmt: str) -> float:
    got = O.bits_to_f64(got_bits, fmt)
    ref = np.asarray(ref, dtype=np.float64)
    excess = np.maximum(0.0, np.abs(got - ref) - 0.5 * ulp(got, fmt))
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    denom = np.abs(ref) + rms
    denom = np.where(denom > 0, denom, 1.0)
    return float((excess / denom).max()) if got.size else 0.0


def exact_fraction(got_bits: np.ndarray, ref: np.ndarray, fmt: str) -> float:
    """Fraction of outputs equal to the correctly rounded reference."""
    return float((O.f64_to_bits(ref, fmt) == got_bits).mean()) if got_bits.size else 1.0


def rel_rms(got_bits: np.ndarray, ref: np.ndarray, fmt: str) -> float:
    got = O.bits_to_f64(got_bits, fmt)
    den = np.sqrt((ref * ref).sum())
    return float(np.sqrt(((got - ref) ** 2).sum()) / den) if den > 0 else 0.0


def to_dev(a: np.ndarray, dev, dtype=None):
    import torch
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
        return t.view(dtype) if dtype is not None else t
    if a.dtype == np.uint32:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def bits_of(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)
