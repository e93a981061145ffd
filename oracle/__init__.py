"""CPU oracle of the group-quantized 4-bit matmul (ctypes binding).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the CUDA path never does, and the two
share no code. The arithmetic lives in ``qmm_oracle.c`` (plain C, fp32 steps
unfused, fp64 references); this module only builds it with gcc and marshals
numpy arrays.

``Oracle(path)`` binds one compiled copy of the C source (the tests also build
copies with planted mistakes to show the pins catch them); the module-level
functions (``oracle.prep_w4a8(...)`` etc.) use the copy built from
``qmm_oracle.c`` in this directory.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qmm_oracle.c")
HDR = os.path.join(HERE, "qmm_oracle.h")
LIB = os.path.join(HERE, "libqmm_oracle.so")

W4A8 = 0
AFFINE = 1
CQ4 = 2

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]

_lock = threading.Lock()
_default = None


def compile_source(src: str, out: str) -> str:
    """gcc one oracle source file (qmm_oracle.h on the include path) into ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-I", HERE, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (seconds). Returns the library path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC), os.path.getmtime(HDR))):
        return LIB
    return compile_source(SRC, LIB)


def _bind(path: str):
    L = ctypes.CDLL(path)
    c = ctypes
    P = c.c_void_p
    i = c.c_int
    L.oracle_f16_to_f64.restype = c.c_double
    L.oracle_f16_to_f64.argtypes = [c.c_uint16]
    L.oracle_f64_to_f16.restype = c.c_uint16
    L.oracle_f64_to_f16.argtypes = [c.c_double]
    L.oracle_fwht_f32.argtypes = [P, i]
    L.oracle_fwht_f64.argtypes = [P, i]
    L.oracle_unpack_nibbles.argtypes = [i, i, i, P, P]
    L.oracle_packed_size.restype = c.c_size_t
    L.oracle_packed_size.argtypes = [i, i, i, i]
    L.oracle_pack.argtypes = [i, i, i, i, P, P, P, P]
    L.oracle_pack_from_values.argtypes = [i, i, i, i, P, P, P, P]
    L.oracle_unpack_blob.argtypes = [i, i, i, i, P, P, P, P]
    L.oracle_interleaved4_to_rows.argtypes = [i, i, i, i, P, P, P, P, P, P]
    L.oracle_prep_w4a8.argtypes = [i, i, i, i, P, P, P, P]
    L.oracle_prep_rotated.argtypes = [i, i, i, P, P, P, P, P, P]
    L.oracle_partials_w4a8.argtypes = [i, i, i, i, P, P, P]
    L.oracle_gemm_w4a8_rows.argtypes = [i, i, i, i, P, P, P, P, i, P, P, P]
    L.oracle_group_sums_affine.argtypes = [i, i, i, P, P]
    L.oracle_gemm_affine_rows.argtypes = [i, i, i, i, P, P, P, P, i, P, P, P]
    L.oracle_pack_cq4.argtypes = [i, i, i, P, P, c.c_float, P, P]
    L.oracle_partials_cq4.argtypes = [i, i, i, i, P, P, P, P]
    L.oracle_gemm_cq4_rows.argtypes = [i, i, i, i, P, P, c.c_float, P, P, P, i, P, P, P]
    return L


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


class Oracle:
    """The oracle functions bound to one compiled copy of the C source."""

    def __init__(self, path: str):
        self.path = path
        self.L = _bind(path)

    # -------------------------------------------------------------- binary16
    def f16_to_f64(self, bits) -> np.ndarray:
        flat = np.asarray(bits, dtype=np.uint16).ravel()
        f = self.L.oracle_f16_to_f64
        return np.array([f(int(h)) for h in flat], dtype=np.float64).reshape(np.shape(bits))

    def f64_to_f16(self, v) -> np.ndarray:
        flat = np.asarray(v, dtype=np.float64).ravel()
        f = self.L.oracle_f64_to_f16
        return np.array([f(float(x)) for x in flat], dtype=np.uint16).reshape(np.shape(v))

    # -------------------------------------------------------------- Hadamard
    def fwht_f32(self, v) -> np.ndarray:
        out = _c(v, np.float32).copy()
        self.L.oracle_fwht_f32(_p(out), out.size)
        return out

    def fwht_f64(self, v) -> np.ndarray:
        out = _c(v, np.float64).copy()
        self.L.oracle_fwht_f64(_p(out), out.size)
        return out

    # -------------------------------------------------------------- weights
    def unpack_nibbles(self, variant: int, q_bytes, K: int) -> np.ndarray:
        q_bytes = _c(q_bytes, np.uint8)
        N = q_bytes.shape[0]
        out = np.empty((N, K), dtype=np.int8)
        _check(self.L.oracle_unpack_nibbles(variant, N, K, _p(q_bytes), _p(out)), "unpack_nibbles")
        return out

    def packed_size(self, variant: int, N: int, K: int, group: int) -> int:
        return int(self.L.oracle_packed_size(variant, N, K, group))

    def pack(self, variant, N, K, group, q_bytes, scales, biases=None) -> np.ndarray:
        out = np.empty(self.packed_size(variant, N, K, group), dtype=np.uint8)
        _check(self.L.oracle_pack(variant, N, K, group, _p(_c(q_bytes, np.uint8)),
                                  _p(_c(scales, np.uint16)),
                                  _p(None if biases is None else _c(biases, np.uint16)), _p(out)),
               "pack")
        return out

    def pack_from_values(self, variant, N, K, group, q_values, scales, biases=None) -> np.ndarray:
        out = np.empty(self.packed_size(variant, N, K, group), dtype=np.uint8)
        _check(self.L.oracle_pack_from_values(variant, N, K, group, _p(_c(q_values, np.int8)),
                                              _p(_c(scales, np.uint16)),
                                              _p(None if biases is None else _c(biases, np.uint16)),
                                              _p(out)),
               "pack_from_values")
        return out

    def interleaved4_to_rows(self, N, K, group, chunk_k, panels, pscales, pbiases=None):
        """4-row panels -> (q_bytes [N][K/2], scales [N][G], biases [N][G] or None)."""
        G = K // group
        q = np.empty((N, K // 2), dtype=np.uint8)
        s = np.empty((N, G), dtype=np.uint16)
        b = np.empty((N, G), dtype=np.uint16) if pbiases is not None else None
        _check(self.L.oracle_interleaved4_to_rows(N, K, group, chunk_k, _p(_c(panels, np.uint8)),
                                                  _p(_c(pscales, np.uint16)),
                                                  _p(None if pbiases is None else _c(pbiases, np.uint16)),
                                                  _p(q), _p(s), _p(b)), "interleaved4_to_rows")
        return q, s, b

    def unpack_blob(self, variant, N, K, group, blob):
        G = K // group
        q = np.empty((N, K), dtype=np.int8)
        s = np.empty((N, G), dtype=np.uint16)
        b = np.empty((N, G), dtype=np.uint16) if variant == AFFINE else None
        _check(self.L.oracle_unpack_blob(variant, N, K, group, _p(_c(blob, np.uint8)), _p(q), _p(s),
                                         _p(b)), "unpack_blob")
        return q, s, b

    # -------------------------------------------------------------- W4A8
    def prep_w4a8(self, x, group: int, hadamard: int):
        """(a int8 [M][K], sx float32 [M][G], asum int32 [M][G])."""
        x = _c(x, np.float32)
        M, K = x.shape
        G = K // group
        a = np.empty((M, K), dtype=np.int8)
        sx = np.empty((M, G), dtype=np.float32)
        asum = np.empty((M, G), dtype=np.int32)
        _check(self.L.oracle_prep_w4a8(M, K, group, hadamard, _p(x), _p(a), _p(sx), _p(asum)),
               "prep_w4a8")
        return a, sx, asum

    def prep_rotated(self, R, x, group: int):
        """(a int8 [M][K], sx float32 [M][G], asum int32 [M][G], z float32 [M][K])."""
        x = _c(np.atleast_2d(x), np.float32)
        R = _c(R, np.float32)
        M, K = x.shape
        G = K // group
        a = np.empty((M, K), dtype=np.int8)
        sx = np.empty((M, G), dtype=np.float32)
        asum = np.empty((M, G), dtype=np.int32)
        z = np.empty((M, K), dtype=np.float32)
        _check(self.L.oracle_prep_rotated(M, K, group, _p(R), _p(x), _p(a), _p(sx), _p(asum), _p(z)),
               "prep_rotated")
        return a, sx, asum, z

    def partials_w4a8(self, q_bytes, a, group) -> np.ndarray:
        """P int32 [M][N][G]."""
        q_bytes = _c(q_bytes, np.uint8)
        a = _c(a, np.int8)
        M, K = a.shape
        N = q_bytes.shape[0]
        P = np.empty((M, N, K // group), dtype=np.int32)
        _check(self.L.oracle_partials_w4a8(M, N, K, group, _p(q_bytes), _p(a), _p(P)), "partials_w4a8")
        return P

    def gemm_w4a8(self, q_bytes, sw, a, sx, group, rows=None):
        """(Y, Ymag) float64 [M][len(rows)] (all N rows when rows is None)."""
        q_bytes = _c(q_bytes, np.uint8)
        a = _c(a, np.int8)
        M, K = a.shape
        N = q_bytes.shape[0]
        r = None if rows is None else _c(rows, np.int32)
        nr = N if r is None else r.size
        Y = np.empty((M, nr), dtype=np.float64)
        Ym = np.empty((M, nr), dtype=np.float64)
        _check(self.L.oracle_gemm_w4a8_rows(M, N, K, group, _p(q_bytes), _p(_c(sw, np.uint16)), _p(a),
                                            _p(_c(sx, np.float32)), nr, _p(r), _p(Y), _p(Ym)),
               "gemm_w4a8")
        return Y, Ym

    # -------------------------------------------------------------- CQ4
    def pack_cq4(self, N, K, group, idx_bytes, codebook, cb_scale, scales) -> np.ndarray:
        out = np.empty(self.packed_size(CQ4, N, K, group), dtype=np.uint8)
        _check(self.L.oracle_pack_cq4(N, K, group, _p(_c(idx_bytes, np.uint8)), _p(_c(codebook, np.int8)),
                                      float(cb_scale), _p(_c(scales, np.uint16)), _p(out)), "pack_cq4")
        return out

    def partials_cq4(self, idx_bytes, codebook, a, group) -> np.ndarray:
        """P int32 [M][N][G] with P = sum codebook[index] * a."""
        idx_bytes = _c(idx_bytes, np.uint8)
        a = _c(a, np.int8)
        M, K = a.shape
        N = idx_bytes.shape[0]
        P = np.empty((M, N, K // group), dtype=np.int32)
        _check(self.L.oracle_partials_cq4(M, N, K, group, _p(idx_bytes), _p(_c(codebook, np.int8)), _p(a), _p(P)),
               "partials_cq4")
        return P

    def gemm_cq4(self, idx_bytes, codebook, cb_scale, sw, a, sx, group, rows=None):
        """(Y, Ymag) float64 [M][len(rows)] (all N rows when rows is None)."""
        idx_bytes = _c(idx_bytes, np.uint8)
        a = _c(a, np.int8)
        M, K = a.shape
        N = idx_bytes.shape[0]
        r = None if rows is None else _c(rows, np.int32)
        nr = N if r is None else r.size
        Y = np.empty((M, nr), dtype=np.float64)
        Ym = np.empty((M, nr), dtype=np.float64)
        _check(self.L.oracle_gemm_cq4_rows(M, N, K, group, _p(idx_bytes), _p(_c(codebook, np.int8)), float(cb_scale),
                                           _p(_c(sw, np.uint16)), _p(a), _p(_c(sx, np.float32)), nr, _p(r), _p(Y),
                                           _p(Ym)), "gemm_cq4")
        return Y, Ym

    # -------------------------------------------------------------- affine
    def group_sums_affine(self, x_f32, group: int = 64) -> np.ndarray:
        """S float32 [M][G] by the page's tree."""
        x = _c(x_f32, np.float32)
        M, K = x.shape
        S = np.empty((M, K // group), dtype=np.float32)
        _check(self.L.oracle_group_sums_affine(M, K, group, _p(x), _p(S)), "group_sums_affine")
        return S

    def gemm_affine(self, q_bytes, s, b, x16, group=64, rows=None):
        """(Y, Ymag) float64 [M][len(rows)] from fp16 x bits [M][K]."""
        q_bytes = _c(q_bytes, np.uint8)
        x16 = _c(x16, np.uint16)
        M, K = x16.shape
        N = q_bytes.shape[0]
        r = None if rows is None else _c(rows, np.int32)
        nr = N if r is None else r.size
        Y = np.empty((M, nr), dtype=np.float64)
        Ym = np.empty((M, nr), dtype=np.float64)
        _check(self.L.oracle_gemm_affine_rows(M, N, K, group, _p(q_bytes), _p(_c(s, np.uint16)),
                                              _p(_c(b, np.uint16)), _p(x16), nr, _p(r), _p(Y), _p(Ym)),
               "gemm_affine")
        return Y, Ym


def default() -> Oracle:
    """The oracle built from ``qmm_oracle.c`` in this directory."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def __getattr__(name):
    # module-level access to the default oracle: oracle.prep_w4a8(...)
    if name.startswith("__"):
        raise AttributeError(name)
    return getattr(default(), name)
