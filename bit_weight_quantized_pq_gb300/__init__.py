"""Python binding of libpq, the GB300 weight-only-quantized linear layer.

Argument marshalling only: every function here forwards to the C entry point
of the same name in ``include/pq.h`` through ctypes.  Device memory and
streams come from PyTorch (or any CUDA allocator); all computation runs in
the library's CUDA kernels.  If ``_lib/libpq.so`` has not been built the first
call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB, build  # noqa: F401  (build() compiles the library)

# ---- constants mirrored from include/pq.h (checked by the tests) ----
PQ_OK = 0
PQ_ERR_INVALID_ARG = -1
PQ_ERR_SHAPE = -2
PQ_ERR_ALIGN = -3
PQ_ERR_GIDX = -4
PQ_ERR_ZP_CONVENTION = -5
PQ_ERR_UNSUPPORTED = -6
PQ_ERR_CUDA = -7
PQ_ERR_DEVICE_TIMEOUT = -8
PQ_ERR_BUFFER_TOO_SMALL = -9

PQ_FMT_W4_GPTQ = 1
PQ_FMT_W2_PQ2 = 2
PQ_FMT_W4_AFFINE = 3
PQ_ZP_SYMMETRIC_8 = 0
PQ_ZP_EXPLICIT_U8 = 1
PQ_F16 = 1
PQ_BF16 = 2

PQ_VARIANT_AUTO = 0
PQ_VARIANT_W4_GEMV = 1
PQ_VARIANT_W4_GEMM = 2
PQ_VARIANT_W2_GEMV_FUSED = 3
PQ_VARIANT_W2_GEMV = 4
PQ_VARIANT_W2_GEMM = 5
PQ_VARIANT_W2_GEMV_TC = 6
PQ_VARIANT_W2_GEMV_BF = 7
PQ_VARIANT_W2_GEMV_CL = 8


class pq_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "fmt", "N", "K", "group", "zp", "has_gidx", "act_dtype", "out_dtype", "act_group", "max_m")]


class pq_plan_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "variant", "grid", "block", "smem_bytes", "launches", "m_tile", "k_split")]


class pq_norm(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_void_p), ("signs", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("unit_offset", ctypes.c_int32), ("had_block", ctypes.c_int32)]


class PQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pq status {status}: {message}")
        self.status = status


_lib = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_DESC = ctypes.POINTER(pq_desc)

_SIGNATURES = {
    "pq_prepared_bytes": (_sz, [_DESC]),
    "pq_workspace_bytes": (_sz, [_DESC]),
    "pq_prepare_w4": (_i32, [_DESC, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "pq_prepare_w2": (_i32, [_DESC, _vp, _sz, _vp, _sz, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "pq_prepare_affine4": (_i32, [_DESC, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "pq_linear": (_i32, [_vp, _vp, _vp, _i32, _vp]),
    "pq_plan": (_i32, [_DESC, _i32, _i32, ctypes.POINTER(pq_plan_info)]),
    "pq_linear_variant": (_i32, [_vp, _vp, _vp, _i32, _i32, _vp]),
    "pq_device_status": (_i32, [_vp, _vp]),
    "pq_destroy": (None, [_vp]),
    "pq_last_error": (ctypes.c_char_p, []),
    "pq_debug_unpack": (_i32, [_vp, _vp, _vp]),
    "pq_debug_w2a8_quantize": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp]),
    "pq_debug_w2a8_group_sums": (_i32, [_vp, _vp, _vp, _i32, _vp]),
    "pq_debug_expire_wait": (_i32, [_vp, _i32, _vp]),
    "pq_linear_w2a8_static": (_i32, [_vp, _vp, _vp, _i32, _vp]),
    "pq_act_bytes": (_sz, [_DESC, _i32]),
    "pq_quantize_act": (_i32, [_vp, _vp, _vp, _sz, _i32, _vp]),
    "pq_norm_quantize": (_i32, [_vp, _vp, ctypes.POINTER(pq_norm), _vp, _vp, _vp, _vp, _sz, _i32, _vp]),
    "pq_linear_act": (_i32, [_vp, _sz, _vp, _vp, _i32, _vp]),
    "pq_debug_act_unpack": (_i32, [_vp, _sz, _vp, _i32, _vp, _vp, _vp, _vp]),
    "pq_probe_read": (_i32, [_vp, _sz, _vp, _i32, _i32, _vp]),
}


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} is missing: build it with __graft_entry__.build() "
                              "(there is no CPU fallback)")
        handle = ctypes.CDLL(LIB)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):           # numpy host array
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int) -> None:
    if rc != PQ_OK:
        raise PQError(rc, pq_last_error())


def make_desc(fmt, N, K, *, zp=PQ_ZP_SYMMETRIC_8, has_gidx=0, act_dtype=PQ_BF16, out_dtype=None,
              act_group=128, max_m=16, group=128) -> pq_desc:
    return pq_desc(fmt, N, K, group, zp, has_gidx, act_dtype,
                   act_dtype if out_dtype is None else out_dtype, act_group, max_m)


def pq_last_error() -> str:
    msg = lib().pq_last_error()
    return msg.decode() if msg else ""


def pq_prepared_bytes(desc: pq_desc) -> int:
    return lib().pq_prepared_bytes(ctypes.byref(desc))


def pq_workspace_bytes(desc: pq_desc) -> int:
    return lib().pq_workspace_bytes(ctypes.byref(desc))


def pq_prepare_w4(desc, qweight, scales, zeros, g_idx, prepared, prepared_bytes, workspace,
                  workspace_bytes, stream=None) -> int:
    """g_idx: host int32 array (numpy) or None.  Returns the handle."""
    out = _vp()
    if g_idx is not None:
        import numpy as np
        g_idx = np.ascontiguousarray(g_idx, dtype=np.int32)
    rc = lib().pq_prepare_w4(ctypes.byref(desc), _ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(g_idx),
                             _ptr(prepared), prepared_bytes, _ptr(workspace), workspace_bytes,
                             _stream(stream), ctypes.byref(out))
    _check(rc)
    return out.value


def pq_prepare_w2(desc, raw, row_stride_bytes, prepared, prepared_bytes, workspace, workspace_bytes,
                  stream=None) -> int:
    out = _vp()
    rc = lib().pq_prepare_w2(ctypes.byref(desc), _ptr(raw), row_stride_bytes, _ptr(prepared),
                             prepared_bytes, _ptr(workspace), workspace_bytes, _stream(stream),
                             ctypes.byref(out))
    _check(rc)
    return out.value


def pq_prepare_affine4(desc, wq, scales, biases, prepared, prepared_bytes, workspace, workspace_bytes,
                       stream=None) -> int:
    out = _vp()
    rc = lib().pq_prepare_affine4(ctypes.byref(desc), _ptr(wq), _ptr(scales), _ptr(biases), _ptr(prepared),
                                  prepared_bytes, _ptr(workspace), workspace_bytes, _stream(stream),
                                  ctypes.byref(out))
    _check(rc)
    return out.value


def pq_linear(x, handle: int, y, M: int, stream=None) -> None:
    _check(lib().pq_linear(_ptr(x), handle, _ptr(y), M, _stream(stream)))


def pq_linear_variant(x, handle: int, y, M: int, variant: int, stream=None) -> None:
    _check(lib().pq_linear_variant(_ptr(x), handle, _ptr(y), M, variant, _stream(stream)))


def pq_plan(desc: pq_desc, M: int, num_sms: int) -> dict:
    info = pq_plan_info()
    _check(lib().pq_plan(ctypes.byref(desc), M, num_sms, ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in pq_plan_info._fields_}


def pq_device_status(handle: int, stream=None) -> int:
    return lib().pq_device_status(handle, _stream(stream))


def pq_destroy(handle: int) -> None:
    lib().pq_destroy(handle)


def pq_debug_unpack(handle: int, w, stream=None) -> None:
    _check(lib().pq_debug_unpack(handle, _ptr(w), _stream(stream)))


def pq_debug_w2a8_quantize(x, handle: int, q, xs, M: int, stream=None) -> None:
    _check(lib().pq_debug_w2a8_quantize(_ptr(x), handle, _ptr(q), _ptr(xs), M, _stream(stream)))


def pq_debug_w2a8_group_sums(x, handle: int, S, M: int, stream=None) -> None:
    _check(lib().pq_debug_w2a8_group_sums(_ptr(x), handle, _ptr(S), M, _stream(stream)))


def pq_linear_w2a8_static(x, handle: int, y, M: int, stream=None) -> None:
    """Ternary decode without any device allocation (scratch in a fixed array
    inside the library); see include/pq.h for its limits."""
    _check(lib().pq_linear_w2a8_static(_ptr(x), handle, _ptr(y), M, _stream(stream)))


def pq_act_bytes(desc: pq_desc, M: int) -> int:
    return lib().pq_act_bytes(ctypes.byref(desc), M)


def pq_quantize_act(x, handle: int, act, act_bytes: int, M: int, stream=None) -> None:
    _check(lib().pq_quantize_act(_ptr(x), handle, _ptr(act), act_bytes, M, _stream(stream)))


def pq_norm_quantize(h, r, norm: pq_norm, handle: int, r_out, norm_out, act, act_bytes: int, M: int,
                     stream=None) -> None:
    _check(lib().pq_norm_quantize(_ptr(h), _ptr(r), ctypes.byref(norm), handle, _ptr(r_out), _ptr(norm_out),
                                  _ptr(act), act_bytes, M, _stream(stream)))


def pq_linear_act(act, act_bytes: int, handle: int, y, M: int, stream=None) -> None:
    _check(lib().pq_linear_act(_ptr(act), act_bytes, handle, _ptr(y), M, _stream(stream)))


def pq_debug_act_unpack(act, act_bytes: int, handle: int, M: int, q, xs, sq, stream=None) -> None:
    _check(lib().pq_debug_act_unpack(_ptr(act), act_bytes, handle, M, _ptr(q), _ptr(xs), _ptr(sq),
                                     _stream(stream)))


def pq_probe_read(src, nbytes: int, sink, ctas_per_sm: int = 0, dependent: int = 0, stream=None) -> None:
    """Copy-only read of nbytes of src (see include/pq.h)."""
    _check(lib().pq_probe_read(_ptr(src), nbytes, _ptr(sink), ctas_per_sm, dependent, _stream(stream)))


def pq_debug_expire_wait(handle: int, spin_limit: int, stream=None) -> None:
    _check(lib().pq_debug_expire_wait(handle, spin_limit, _stream(stream)))


from .layer import QuantizedLinear  # noqa: E402,F401
