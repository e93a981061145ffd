"""Python binding of libqmm_gb300 (group-quantized 4-bit-weight matmul, sm_103a).

The functions carry the names of the C entry points in ``include/qmm.h`` and
only marshal arguments: torch tensors become device pointers, the stream
defaults to torch's current stream, and a status other than ``QMM_OK`` raises
``QmmError``. Every computation happens in the library's CUDA kernels; if the
library is missing this module raises on import (there is no fallback).
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
# QMM_CHECKED_LIBRARY=1 loads the test-only checked variant (same kernels with
# internal range checks recorded in the device error word; see build.py)
LIB_PATH = os.path.join(HERE, "libqmm_gb300_checked.so" if os.environ.get("QMM_CHECKED_LIBRARY") == "1"
                        else "libqmm_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "qmm.h")

QMM_W4A8 = 0
QMM_AFFINE = 1
QMM_CQ4 = 2
QMM_DTYPE_F32, QMM_DTYPE_F16, QMM_DTYPE_BF16 = 0, 1, 2
QMM_PATH_GEMV, QMM_PATH_GEMM = 0, 1
KERNEL_IDS = {0: "none", 1: "pack", 2: "prep_w4a8", 3: "prep_affine", 4: "gemv_w4a8", 5: "gemm_w4a8",
              6: "gemm_affine", 7: "gemv_fused", 8: "gemm_rows", 9: "gemv_fused_siblings", 10: "gemv_cq4",
              11: "gemm_cq4", 12: "prep_rotated", 13: "gemm_narrow",
              14: "gemm_narrow_e4m3"}

STATUS = {0: "QMM_OK", 1: "QMM_ERR_INVALID_ARG", 2: "QMM_ERR_UNSUPPORTED_SHAPE", 3: "QMM_ERR_UNSUPPORTED_DEVICE",
          4: "QMM_ERR_MISALIGNED", 5: "QMM_ERR_CUDA", 6: "QMM_ERR_TIMEOUT", 7: "QMM_ERR_WORKSPACE"}


class QmmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


class qmm_weight_desc(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
                ("group", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{os.path.basename(LIB_PATH)} not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D = ctypes.POINTER(qmm_weight_desc)
    sig = {
        "qmm_packed_size": (SZ, [D]),
        "qmm_pack_weights": (I32, [D, P, P, P, P, P]),
        "qmm_pack_weights_cq4": (I32, [D, P, P, ctypes.c_float, P, P, P]),
        "qmm_pack_weights_interleaved4": (I32, [D, I32, P, P, P, P, ctypes.c_float, P, P]),
        "qmm_prep_act": (I32, [I32, I32, I32, I32, I32, P, I32, P, P, P, P, P, P, P]),
        "qmm_prep_act_rotated": (I32, [I32, I32, I32, P, P, I32, P, P, P, P, P]),
        "qmm_gemv_workspace_size": (SZ, [D]),
        "qmm_gemv": (I32, [D, P, P, P, P, P, SZ, P]),
        "qmm_gemv_static_scratch": (I32, [D, P, P, P, P, P]),
        "qmm_gemv_fused": (I32, [D, P, P, I32, I32, P, P, P, P]),
        "qmm_gemv_fused_siblings": (I32, [I32, D, P, P, I32, I32, P, P, P, P]),
        "qmm_gemm": (I32, [D, P, I32, P, P, P, P]),
        "qmm_debug_partials": (I32, [D, P, I32, I32, P, P, P]),
        "qmm_status_string": (ctypes.c_char_p, [I32]),
        "qmm_last_kernel_id": (I32, []),
        "qmm_device_status": (I32, [P, ctypes.POINTER(I32)]),
        "qmm_set_pdl": (None, [I32]),
        "qmm_set_fault_injection": (None, [I32]),
        "qmm_set_gemm_weight_operand": (None, [I32]),
        "qmm_set_gemm_narrow": (None, [I32]),
        "qmm_set_gemm_rows_max": (None, [I32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


_L = _load()


def declared_symbols(header: str = HEADER) -> list:
    """Names of the functions include/qmm.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_\w+)\s*\(", text)))


def library():
    return _L


# ------------------------------------------------------------------ helpers

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st, what):
    if st != 0:
        raise QmmError(st, what)


def weight_desc(variant: int, N: int, K: int, group: int) -> qmm_weight_desc:
    return qmm_weight_desc(variant, N, K, group)


# ------------------------------------------------------------------ entry points

def status_string(status: int) -> str:
    return _L.qmm_status_string(status).decode()


qmm_status_string = status_string


def qmm_packed_size(desc: qmm_weight_desc) -> int:
    return int(_L.qmm_packed_size(ctypes.byref(desc)))


def qmm_pack_weights(desc, q, scales, biases, packed, stream=None):
    _check(_L.qmm_pack_weights(ctypes.byref(desc), _ptr(q), _ptr(scales), _ptr(biases), _ptr(packed),
                               _stream(stream)), "qmm_pack_weights")


def qmm_pack_weights_cq4(desc, idx, codebook, cb_scale, scales, packed, stream=None):
    """codebook: 16 int8 levels on the host (anything numpy.asarray(..., int8) accepts)."""
    import numpy as np
    levels = np.ascontiguousarray(np.asarray(codebook, dtype=np.int8).reshape(-1))
    if levels.size != 16:
        raise ValueError("a CQ4 codebook has 16 levels")
    _check(_L.qmm_pack_weights_cq4(ctypes.byref(desc), _ptr(idx), levels.ctypes.data_as(ctypes.c_void_p),
                                   float(cb_scale), _ptr(scales), _ptr(packed), _stream(stream)),
           "qmm_pack_weights_cq4")


def qmm_pack_weights_interleaved4(desc, chunk_k, panels, scales, biases, packed, codebook=None, cb_scale=1.0,
                                  stream=None):
    """Weights in 4-row panels; codebook (16 int8 host levels) for QMM_CQ4 only."""
    import numpy as np
    cb = None
    if codebook is not None:
        levels = np.ascontiguousarray(np.asarray(codebook, dtype=np.int8).reshape(-1))
        if levels.size != 16:
            raise ValueError("a CQ4 codebook has 16 levels")
        cb = levels.ctypes.data_as(ctypes.c_void_p)
    _check(_L.qmm_pack_weights_interleaved4(ctypes.byref(desc), int(chunk_k), _ptr(panels), _ptr(scales),
                                            _ptr(biases), cb, float(cb_scale), _ptr(packed), _stream(stream)),
           "qmm_pack_weights_interleaved4")


def qmm_prep_act(variant, M, K, group, hadamard, x, x_dtype, a=None, a16=None, sx=None, asum=None, gsum=None,
                 x16=None, stream=None):
    _check(_L.qmm_prep_act(variant, M, K, group, hadamard, _ptr(x), x_dtype, _ptr(a), _ptr(a16), _ptr(sx),
                           _ptr(asum), _ptr(gsum), _ptr(x16), _stream(stream)), "qmm_prep_act")


def qmm_prep_act_rotated(M, K, group, R, x, x_dtype, a=None, a16=None, sx=None, asum=None, stream=None):
    _check(_L.qmm_prep_act_rotated(M, K, group, _ptr(R), _ptr(x), x_dtype, _ptr(a), _ptr(a16), _ptr(sx),
                                   _ptr(asum), _stream(stream)), "qmm_prep_act_rotated")


def qmm_gemv_workspace_size(desc) -> int:
    return int(_L.qmm_gemv_workspace_size(ctypes.byref(desc)))


def qmm_gemv(desc, packed, a, sx, y, workspace=None, workspace_bytes=0, stream=None):
    if workspace is not None and not workspace_bytes and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(_L.qmm_gemv(ctypes.byref(desc), _ptr(packed), _ptr(a), _ptr(sx), _ptr(y), _ptr(workspace),
                       workspace_bytes, _stream(stream)), "qmm_gemv")


def qmm_gemv_static_scratch(desc, packed, a, sx, y, stream=None):
    """qmm_gemv with the library's own fixed scratch (allocates nothing)."""
    _check(_L.qmm_gemv_static_scratch(ctypes.byref(desc), _ptr(packed), _ptr(a), _ptr(sx), _ptr(y),
                                      _stream(stream)), "qmm_gemv_static_scratch")


def qmm_gemv_fused(desc, packed, x, x_dtype, hadamard, y, a_out=None, sx_out=None, stream=None):
    _check(_L.qmm_gemv_fused(ctypes.byref(desc), _ptr(packed), _ptr(x), x_dtype, hadamard, _ptr(y), _ptr(a_out),
                             _ptr(sx_out), _stream(stream)), "qmm_gemv_fused")


def qmm_gemv_fused_siblings(descs, packed, x, x_dtype, hadamard, ys, a_out=None, sx_out=None, stream=None):
    """descs, packed, ys: sequences of equal length (the sibling matrices)."""
    n = len(descs)
    if len(packed) != n or len(ys) != n:
        raise ValueError("descs, packed and ys must have the same length")
    darr = (qmm_weight_desc * max(n, 1))(*descs)
    parr = (ctypes.c_void_p * max(n, 1))(*[_ptr(p) for p in packed])
    yarr = (ctypes.c_void_p * max(n, 1))(*[_ptr(v) for v in ys])
    _check(_L.qmm_gemv_fused_siblings(n, darr, parr, _ptr(x), x_dtype, hadamard, yarr, _ptr(a_out), _ptr(sx_out),
                                      _stream(stream)), "qmm_gemv_fused_siblings")


def qmm_gemm(desc, packed, M, act16, act_scale, Y, stream=None):
    _check(_L.qmm_gemm(ctypes.byref(desc), _ptr(packed), M, _ptr(act16), _ptr(act_scale), _ptr(Y),
                       _stream(stream)), "qmm_gemm")


def qmm_debug_partials(desc, packed, M, path, act, P, stream=None):
    _check(_L.qmm_debug_partials(ctypes.byref(desc), _ptr(packed), M, path, _ptr(act), _ptr(P), _stream(stream)),
           "qmm_debug_partials")


def qmm_last_kernel_id() -> int:
    return int(_L.qmm_last_kernel_id())


def qmm_device_status(stream=None) -> int:
    """Returns the raw device error word (0 = fine); raises on a CUDA failure."""
    flags = ctypes.c_int32(0)
    st = _L.qmm_device_status(_stream(stream), ctypes.byref(flags))
    if st not in (0, 6):
        raise QmmError(st, "qmm_device_status")
    return int(flags.value)


def qmm_set_pdl(enable: bool):
    _L.qmm_set_pdl(1 if enable else 0)


def qmm_set_fault_injection(point: int):
    """Test-only: 1 makes the rotation prepass's bounded waits run out; 0 = off."""
    _L.qmm_set_fault_injection(int(point))


def qmm_set_gemm_weight_operand(in_shared_memory: bool):
    _L.qmm_set_gemm_weight_operand(1 if in_shared_memory else 0)


NARROW_OFF, NARROW_AUTO, NARROW_ALWAYS, NARROW_F16 = 0, 1, 2, 3


def qmm_set_gemm_narrow(mode: int):
    _L.qmm_set_gemm_narrow(int(mode))


def qmm_set_gemm_rows_max(max_rows: int):
    _L.qmm_set_gemm_rows_max(int(max_rows))
