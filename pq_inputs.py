"""Seeded synthetic inputs for the weight-only-quantized linear layer.

Every generator draws from numpy's PCG64 with an explicit seed and lays the
draws out in the input formats the layer accepts:

* GPTQ-style 4-bit frames: ``qweight`` uint32 ``[K/8][N]`` (eight 4-bit codes
  per word along K), fp16 ``scales`` ``[K/128][N]``, optional uint8 ``zeros``
  ``[K/128][N]`` and optional int32 ``g_idx`` ``[K]``;
* ternary "PQ2" rows: uint8 ``[N][K/128*34]``, each 34-byte block a
  little-endian fp16 scale followed by 32 code bytes (four 2-bit codes per
  byte);
* fp16 / bf16 activations ``[M][K]`` as raw uint16 bit patterns.

This module holds no dequantisation, quantisation or matmul arithmetic.  It is
shared by the CPU oracle's tests, the CUDA parity tests and the benchmark, so
both sides always see identical bytes.
"""
from __future__ import annotations

import numpy as np

GROUP = 128
PQ2_BLOCK_BYTES = 34


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Store float32 draws as bf16 bit patterns (round to nearest even)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    """Store float32 draws as fp16 bit patterns (numpy's IEEE conversion)."""
    return np.asarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def activations(seed: int, M: int, K: int, dtype: str, outlier_rate: float = 0.0,
                outlier_scale: float = 20.0) -> np.ndarray:
    """N(0,1) activations; an independent Bernoulli(outlier_rate) mask scales
    the selected entries by ``outlier_scale``.  Returns uint16 bits [M][K]."""
    r = rng(seed)
    a = r.standard_normal((M, K), dtype=np.float32)
    if outlier_rate > 0.0:
        mask = r.random((M, K)) < outlier_rate
        a = np.where(mask, a * np.float32(outlier_scale), a).astype(np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(a)
    if dtype == "f16":
        return f32_to_f16_bits(a)
    raise ValueError(dtype)


def affine4_layer(seed: int, N: int, K: int, dtype: str) -> dict:
    """An MLX-style affine 4-bit layer: words uint32 [N][K/8] of uniform codes,
    scales 0.001 + |N(0, 0.01)| and biases N(0, 0.02) per 64-input group
    ([N][K/64], 16-bit patterns of ``dtype``)."""
    r = rng(seed)
    to_bits = f32_to_bf16_bits if dtype == "bf16" else f32_to_f16_bits
    wq = r.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    s = (0.001 + np.abs(r.standard_normal((N, K // 64), dtype=np.float32) * np.float32(0.01))).astype(np.float32)
    b = (r.standard_normal((N, K // 64), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    return {"wq": wq, "scales": to_bits(s), "biases": to_bits(b)}


def norm_inputs(seed: int, M: int, K: int, dtype: str, unit_offset: bool = True,
                residual: bool = True) -> dict:
    """Inputs of the fused activation producer: hidden rows h ~ N(0,1) with
    0.1% outliers x20 (uint16 bits [M][K]), a residual stream r ~ N(0,1) or
    None, a norm weight gamma [K] (N(0, 0.1) when the layer stores it as an
    offset from one, else 1 + N(0, 0.1)) and Rademacher signs int8 [K]."""
    r = rng(seed)
    to_bits = f32_to_bf16_bits if dtype == "bf16" else f32_to_f16_bits
    h = r.standard_normal((M, K), dtype=np.float32)
    h = np.where(r.random((M, K)) < 0.001, h * np.float32(20.0), h).astype(np.float32)
    res = r.standard_normal((M, K), dtype=np.float32) if residual else None
    g = (r.standard_normal(K, dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    if not unit_offset:
        g = (g + np.float32(1.0)).astype(np.float32)
    signs = np.where(r.random(K) < 0.5, -1, 1).astype(np.int8)
    return {"h": to_bits(h), "r": None if res is None else to_bits(res), "gamma": to_bits(g), "signs": signs}


def w4_frame(seed: int, K: int, N: int, scale_floor: float, scale_sigma: float,
             zero_points: bool = False, act_order: str | None = None) -> dict:
    """A GPTQ-style 4-bit frame.

    Codes are uniform on 0..15: uniform random 32-bit words hold eight
    independent uniform 4-bit fields, so the words are drawn directly.
    Scales are fp16(scale_floor + |N(0, scale_sigma)|) per (group, column).
    ``zero_points`` draws explicit uint8 zero points uniform on 0..15.
    ``act_order`` draws ``g_idx``:
      * ``"scatter"``: a random permutation p of 0..K-1 with
        g_idx[p[i]] = i // 128, so every group holds 128 scattered rows;
      * ``"blocks"``: each aligned 128-row block gets a distinct random group;
      * ``None``: no g_idx (group of row k is k // 128).
    """
    if K % GROUP or K % 8:
        raise ValueError("K must be a multiple of 128")
    G = K // GROUP
    r = rng(seed)
    qweight = r.integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
    scales = (scale_floor + np.abs(r.normal(0.0, scale_sigma, size=(G, N)))).astype(np.float32)
    frame = {
        "K": K, "N": N,
        "qweight": qweight,
        "scales": f32_to_f16_bits(scales),
        "zeros": r.integers(0, 16, size=(G, N), dtype=np.uint8) if zero_points else None,
        "g_idx": None,
    }
    if act_order == "scatter":
        p = r.permutation(K)
        g_idx = np.empty(K, dtype=np.int32)
        g_idx[p] = (np.arange(K) // GROUP).astype(np.int32)
        frame["g_idx"] = g_idx
    elif act_order == "blocks":
        blocks = r.permutation(G).astype(np.int32)
        frame["g_idx"] = np.repeat(blocks, GROUP).astype(np.int32)
    elif act_order is not None:
        raise ValueError(act_order)
    return frame


# The 81 byte values whose four 2-bit fields all lie in {0, 1, 2}.  Drawing a
# byte uniformly from this set draws its four codes independently and
# uniformly from {0, 1, 2}; the field order does not matter for the set.
_TERNARY_BYTES = np.array(
    [b for b in range(256) if all(((b >> (2 * j)) & 3) != 3 for j in range(4))],
    dtype=np.uint8)


def device_w4_frame(seed: int, K: int, N: int, scale_floor: float, scale_sigma: float, device):
    """The symmetric ``w4_frame`` distribution drawn on a CUDA device with a
    seeded torch generator (for large benchmark weights): int32 qweight
    [K/8][N] of uniform random words, fp16 scales [K/128][N]."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    qweight = torch.randint(-(1 << 31), (1 << 31) - 1, (K // 8, N), generator=g, dtype=torch.int64,
                            device=device).to(torch.int32)
    s = scale_floor + torch.randn((K // GROUP, N), generator=g, device=device).abs() * scale_sigma
    return qweight, s.to(torch.float16)


def device_pq2_rows(seed: int, N: int, K: int, device, latent_sigma: float = 0.025):
    """The ``pq2_rows`` distribution drawn on a CUDA device: code bytes
    uniform over the 81 bytes with all codes in {0,1,2}; block scale
    fp16(mean |N(0, latent_sigma)|) over 128 latent draws.  uint8 [N][K/128*34]."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B = K // GROUP
    table = torch.from_numpy(_TERNARY_BYTES).to(device)
    idx = torch.randint(0, len(_TERNARY_BYTES), (N, B, 32), generator=g, device=device)
    code_bytes = table[idx]
    absmean = (torch.randn((N, B, GROUP), generator=g, device=device) * latent_sigma).abs().mean(dim=2)
    scale_bytes = absmean.to(torch.float16).view(torch.uint8).reshape(N, B, 2)
    return torch.cat([scale_bytes, code_bytes], dim=2).reshape(N, B * PQ2_BLOCK_BYTES).contiguous()


def pq2_rows(seed: int, N: int, K: int, latent_sigma: float = 0.025,
             allow_code3: bool = False) -> np.ndarray:
    """Ternary PQ2 rows [N][K/128*34].

    Codes are i.i.d. uniform on {0,1,2} (or on all byte values when
    ``allow_code3``); each block's scale is fp16(mean |z|) of 128 latent
    N(0, latent_sigma) draws, about 0.02 for the default sigma.
    """
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    B = K // GROUP
    r = rng(seed)
    if allow_code3:
        code_bytes = r.integers(0, 256, size=(N, B, 32), dtype=np.uint16).astype(np.uint8)
    else:
        code_bytes = _TERNARY_BYTES[r.integers(0, len(_TERNARY_BYTES), size=(N, B, 32))]
    latent = r.normal(0.0, latent_sigma, size=(N, B, GROUP)).astype(np.float32)
    absmean = np.abs(latent).mean(axis=2, dtype=np.float64).astype(np.float32)
    scale_bytes = f32_to_f16_bits(absmean).astype("<u2").view(np.uint8).reshape(N, B, 2)
    raw = np.concatenate([scale_bytes, code_bytes], axis=2)
    return np.ascontiguousarray(raw.reshape(N, B * PQ2_BLOCK_BYTES))
