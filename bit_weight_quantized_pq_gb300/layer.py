"""A PyTorch-facing holder for one prepared layer.

PyTorch supplies the device memory (the prepared planes and the workspace
are uint8 CUDA tensors owned here) and the stream; the computation is the
C library's.
"""
from __future__ import annotations

import torch

from . import (PQ_BF16, PQ_F16, PQ_FMT_W2_PQ2, PQ_FMT_W4_AFFINE, PQ_FMT_W4_GPTQ, PQ_VARIANT_AUTO,
               PQ_ZP_EXPLICIT_U8, PQ_ZP_SYMMETRIC_8, make_desc, pq_act_bytes, pq_destroy, pq_linear_act,
               pq_linear_variant, pq_norm, pq_norm_quantize, pq_prepare_affine4, pq_prepare_w2, pq_prepare_w4,
               pq_prepared_bytes, pq_quantize_act, pq_workspace_bytes)

_DT = {"f16": PQ_F16, "bf16": PQ_BF16, torch.float16: PQ_F16, torch.bfloat16: PQ_BF16}
_TORCH = {PQ_F16: torch.float16, PQ_BF16: torch.bfloat16}


def _alloc(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    t = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
    assert t.data_ptr() % 256 == 0
    return t


class QuantizedLinear:
    def __init__(self, desc, prepared: torch.Tensor, workspace: torch.Tensor, handle: int):
        self.desc = desc
        self.prepared = prepared
        self.workspace = workspace
        self.handle = handle
        self.out_dtype = _TORCH[desc.out_dtype]

    @classmethod
    def from_w4(cls, qweight: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None = None,
                g_idx=None, act_dtype="bf16", out_dtype=None, max_m: int = 16, stream=None):
        """qweight int32 [K/8][N], scales fp16 [K/128][N], zeros uint8 [K/128][N] or None
        (symmetric, z = 8), g_idx host int32 [K] or None; all device tensors on one GPU."""
        K, N = qweight.shape[0] * 8, qweight.shape[1]
        a = _DT[act_dtype]
        desc = make_desc(PQ_FMT_W4_GPTQ, N, K, zp=PQ_ZP_EXPLICIT_U8 if zeros is not None else PQ_ZP_SYMMETRIC_8,
                         has_gidx=1 if g_idx is not None else 0, act_dtype=a,
                         out_dtype=_DT[out_dtype] if out_dtype is not None else a, max_m=max_m)
        pb, wb = pq_prepared_bytes(desc), pq_workspace_bytes(desc)
        prepared, ws = _alloc(pb, qweight.device), _alloc(wb, qweight.device)
        s = stream if stream is not None else torch.cuda.current_stream(qweight.device)
        h = pq_prepare_w4(desc, qweight, scales, zeros, g_idx, prepared, pb, ws, wb, s)
        return cls(desc, prepared, ws, h)

    @classmethod
    def from_pq2(cls, raw: torch.Tensor, K: int, act_dtype="bf16", out_dtype=None, act_group: int = 128,
                 max_m: int = 16, stream=None):
        """raw uint8 [N][K/128*34] PQ2 rows on the GPU."""
        N = raw.shape[0]
        a = _DT[act_dtype]
        desc = make_desc(PQ_FMT_W2_PQ2, N, K, act_dtype=a, out_dtype=_DT[out_dtype] if out_dtype else a,
                         act_group=act_group, max_m=max_m)
        pb, wb = pq_prepared_bytes(desc), pq_workspace_bytes(desc)
        prepared, ws = _alloc(pb, raw.device), _alloc(wb, raw.device)
        s = stream if stream is not None else torch.cuda.current_stream(raw.device)
        h = pq_prepare_w2(desc, raw, raw.stride(0), prepared, pb, ws, wb, s)
        return cls(desc, prepared, ws, h)

    @classmethod
    def from_affine4(cls, wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, act_dtype="bf16",
                     out_dtype=None, max_m: int = 16, stream=None):
        """MLX affine 4-bit: wq int32 [N][K/8], scales and biases [N][K/64]
        in the activation dtype (as int16 bit patterns or fp16/bf16 tensors).
        Decode GEMV up to 16 tokens, the tensor-core GEMM above (max_m > 16)."""
        N, K = wq.shape[0], wq.shape[1] * 8
        a = _DT[act_dtype]
        desc = make_desc(PQ_FMT_W4_AFFINE, N, K, act_dtype=a, out_dtype=_DT[out_dtype] if out_dtype else a,
                         max_m=max_m, group=64)
        pb, wb = pq_prepared_bytes(desc), pq_workspace_bytes(desc)
        prepared, ws = _alloc(pb, wq.device), _alloc(wb, wq.device)
        s = stream if stream is not None else torch.cuda.current_stream(wq.device)
        h = pq_prepare_affine4(desc, wq, scales, biases, prepared, pb, ws, wb, s)
        return cls(desc, prepared, ws, h)

    def __call__(self, x: torch.Tensor, out: torch.Tensor | None = None, variant: int = PQ_VARIANT_AUTO,
                 stream=None) -> torch.Tensor:
        M = x.shape[0]
        if out is None:
            out = torch.empty((M, self.desc.N), dtype=self.out_dtype, device=x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        pq_linear_variant(x, self.handle, out, M, variant, s)
        return out

    # ---- ternary layers: quantised activations held by the caller ----

    def act_buffer(self, M: int, device=None) -> torch.Tensor:
        """A buffer for M tokens of quantised activations (any ternary layer
        with the same K, act_group and act dtype can read it)."""
        return _alloc(pq_act_bytes(self.desc, M), device if device is not None else self.prepared.device)

    def quantize_act(self, x: torch.Tensor, act: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        M = x.shape[0]
        if act is None:
            act = self.act_buffer(M, x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        pq_quantize_act(x, self.handle, act, act.numel(), M, s)
        return act

    def norm_quantize(self, h: torch.Tensor, gamma: torch.Tensor, eps: float, *, r=None, r_out=None,
                      norm_out=None, signs=None, unit_offset: bool = False, had_block: int = 0,
                      act: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Fused residual add + RMSNorm (+ random-sign Hadamard) + quantise of
        h [M][K] into an activation buffer (see pq_norm_quantize)."""
        M = h.shape[0]
        if act is None:
            act = self.act_buffer(M, h.device)
        nrm = pq_norm(gamma.data_ptr(), None if signs is None else signs.data_ptr(), float(eps),
                      1 if unit_offset else 0, int(had_block))
        s = stream if stream is not None else torch.cuda.current_stream(h.device)
        pq_norm_quantize(h, r, nrm, self.handle, r_out, norm_out, act, act.numel(), M, s)
        return act

    def run_act(self, act: torch.Tensor, M: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """y = x . W from quantised activations of M tokens."""
        if out is None:
            out = torch.empty((M, self.desc.N), dtype=self.out_dtype, device=act.device)
        s = stream if stream is not None else torch.cuda.current_stream(act.device)
        pq_linear_act(act, act.numel(), self.handle, out, M, s)
        return out

    def close(self) -> None:
        if self.handle:
            pq_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
