"""CPU oracle for block-quantized GEMV/GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The product
path (``gemv_mul_mm_gb300``) never does, and this package never imports it.

``qmm_oracle.c`` holds the arithmetic; this module compiles it with the host C
compiler and wraps it with ``ctypes`` + numpy. Formats are named by their GGUF
names; the integer ids below are the oracle's own numbering.

Parity status per format (see ``qmm_oracle.c``): Q5_K, Q2_K and Q3_K byte
layouts are not given by the pages, so their parity against the pages is
unpinned (they are pinned only to the public GGUF reading).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional

import numpy as np

KINDS = ["Q8_0", "Q4_0", "Q5_0", "Q4_K", "Q5_K", "Q6_K",
         "Q2_K", "Q3_K", "IQ4_NL", "IQ4_XS", "MXFP4", "Q4_1", "Q5_1", "Q8_1"]
KIND_ID = {k: i for i, k in enumerate(KINDS)}
PARITY_UNPINNED = ("Q5_K", "Q2_K", "Q3_K")

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_CACHE: dict = {}


def lib_path(sabotage: int = 0) -> str:
    name = "liboracle.so" if sabotage == 0 else f"liboracle_sab{sabotage}.so"
    return os.path.join(_BUILD, name)


def build(sabotage: int = 0, force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (OpenMP when available)."""
    out = lib_path(sabotage)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
            f"-DORACLE_SABOTAGE={int(sabotage)}", _SRC]
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    try:
        r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-o", tmp, "-lm"],
                           capture_output=True, text=True)
        if r.returncode != 0:
            r = subprocess.run(base + ["-o", tmp, "-lm"], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


class Oracle:
    """ctypes view of one oracle build."""

    def __init__(self, sabotage: int = 0):
        self.sabotage = sabotage
        self.lib = ctypes.CDLL(build(sabotage))
        L = self.lib
        L.oracle_f16.restype = ctypes.c_float
        L.oracle_f16.argtypes = [ctypes.c_uint16]
        L.oracle_e8m0.restype = ctypes.c_float
        L.oracle_e8m0.argtypes = [ctypes.c_uint8]
        L.oracle_elem.restype = ctypes.c_float
        L.oracle_elem.argtypes = [ctypes.c_int, _P, _I64]
        L.oracle_block_geometry.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                            ctypes.POINTER(ctypes.c_int)]
        L.oracle_dequant.argtypes = [ctypes.c_int, _P, _I64, _I64, _P]
        L.oracle_gemm.argtypes = [ctypes.c_int, _P, _I64, _I64, _P, ctypes.c_int, _I64,
                                  _P, _P, ctypes.c_int]
        L.oracle_gemm_at.argtypes = [ctypes.c_int, _P, _I64, _I64, _P, ctypes.c_int, _I64,
                                     _P, _P, _P, _P]
        L.oracle_grouped.argtypes = [ctypes.c_int, _P, _I64, ctypes.c_int, _P, ctypes.c_int,
                                     _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P,
                                     ctypes.c_int]
        self.has_openmp = bool(L.oracle_has_openmp())

    # -- scalar decoders ---------------------------------------------------
    def f16(self, h: int) -> float:
        return self.lib.oracle_f16(h)

    def e8m0(self, e: int) -> float:
        return self.lib.oracle_e8m0(e)

    def geometry(self, kind: str):
        bb, be = ctypes.c_int(), ctypes.c_int()
        if self.lib.oracle_block_geometry(KIND_ID[kind], ctypes.byref(bb), ctypes.byref(be)):
            raise ValueError(kind)
        return bb.value, be.value

    def row_bytes(self, kind: str, K: int) -> int:
        bb, be = self.geometry(kind)
        return (K // be) * bb

    # -- arrays ------------------------------------------------------------
    def dequant(self, kind: str, w: np.ndarray, rows: int, cols: int) -> np.ndarray:
        w = np.ascontiguousarray(w, dtype=np.uint8)
        assert w.size >= rows * self.row_bytes(kind, cols)
        out = np.empty((rows, cols), dtype=np.float32)
        rc = self.lib.oracle_dequant(KIND_ID[kind], w.ctypes.data, rows, cols, out.ctypes.data)
        if rc:
            raise ValueError(f"oracle_dequant rc={rc}")
        return out

    @staticmethod
    def _x(x: np.ndarray):
        if x.dtype == np.float16:
            return np.ascontiguousarray(x), 1
        return np.ascontiguousarray(x, dtype=np.float32), 0

    def gemm(self, kind: str, w: np.ndarray, M: int, K: int, x: np.ndarray, N: int,
             nthreads: int = 1):
        """(y, tol), both float64 of shape (N, M): y[n, m] = sum_k W[m,k] x[n,k]."""
        w = np.ascontiguousarray(w, dtype=np.uint8)
        xa, xd = self._x(x)
        assert xa.size >= N * K and w.size >= M * self.row_bytes(kind, K)
        y = np.empty((N, M), dtype=np.float64)
        tol = np.empty((N, M), dtype=np.float64)
        rc = self.lib.oracle_gemm(KIND_ID[kind], w.ctypes.data, M, K, xa.ctypes.data, xd, N,
                                  y.ctypes.data, tol.ctypes.data, nthreads)
        if rc:
            raise ValueError(f"oracle_gemm rc={rc}")
        return y, tol

    def gemm_at(self, kind: str, w: np.ndarray, M: int, K: int, x: np.ndarray,
                n_idx: np.ndarray, m_idx: np.ndarray):
        w = np.ascontiguousarray(w, dtype=np.uint8)
        xa, xd = self._x(x)
        n_idx = np.ascontiguousarray(n_idx, dtype=np.int64)
        m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
        cnt = n_idx.size
        y = np.empty(cnt, dtype=np.float64)
        tol = np.empty(cnt, dtype=np.float64)
        rc = self.lib.oracle_gemm_at(KIND_ID[kind], w.ctypes.data, M, K, xa.ctypes.data, xd,
                                     cnt, n_idx.ctypes.data, m_idx.ctypes.data,
                                     y.ctypes.data, tol.ctypes.data)
        if rc:
            raise ValueError(f"oracle_gemm_at rc={rc}")
        return y, tol

    def grouped(self, kind: str, w: np.ndarray, expert_stride: int, n_experts: int,
                x: np.ndarray, x_row: np.ndarray, expert_id: np.ndarray, M: int, K: int,
                r_idx: Optional[np.ndarray] = None, m_idx: Optional[np.ndarray] = None,
                nthreads: int = 1):
        """All outputs (n_assign, M), or the chosen (r_idx[i], m_idx[i]) outputs."""
        w = np.ascontiguousarray(w, dtype=np.uint8)
        xa, xd = self._x(x)
        x_row = np.ascontiguousarray(x_row, dtype=np.int32)
        expert_id = np.ascontiguousarray(expert_id, dtype=np.int32)
        n_assign = x_row.size
        if r_idx is None:
            y = np.empty((n_assign, M), dtype=np.float64)
            tol = np.empty((n_assign, M), dtype=np.float64)
            cnt, rp, mp = -1, None, None
        else:
            r_idx = np.ascontiguousarray(r_idx, dtype=np.int64)
            m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
            cnt = r_idx.size
            y = np.empty(cnt, dtype=np.float64)
            tol = np.empty(cnt, dtype=np.float64)
            rp, mp = r_idx.ctypes.data, m_idx.ctypes.data
        rc = self.lib.oracle_grouped(KIND_ID[kind], w.ctypes.data, expert_stride, n_experts,
                                     xa.ctypes.data, xd, x_row.ctypes.data,
                                     expert_id.ctypes.data, n_assign, M, K, cnt, rp, mp,
                                     y.ctypes.data, tol.ctypes.data, nthreads)
        if rc:
            raise ValueError(f"oracle_grouped rc={rc}")
        return y, tol


    def moe_ffn(self, *args, **kwargs):
        """The mixture-of-experts layer around the grouped product (oracle/moe.py)."""
        from . import moe
        return moe.moe_ffn(self, *args, **kwargs)


def load(sabotage: int = 0) -> Oracle:
    if sabotage not in _CACHE:
        _CACHE[sabotage] = Oracle(sabotage)
    return _CACHE[sabotage]
