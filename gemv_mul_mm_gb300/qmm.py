"""Thin ctypes binding of libqmm (include/qmm.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libqmm.so``. Tensors are PyTorch CUDA tensors (device memory and
the current stream come from PyTorch). If the library is missing this module
raises; there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqmm.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "qmm.h")

KINDS = ["Q8_0", "Q4_0", "Q5_0", "Q4_K", "Q5_K", "Q6_K",
         "Q2_K", "Q3_K", "IQ4_NL", "IQ4_XS", "MXFP4", "Q4_1", "Q5_1", "Q8_1"]
KIND_ID = {k: i for i, k in enumerate(KINDS)}
F32, F16 = 0, 1

STATUS = {
    0: "QMM_OK", 1: "QMM_ERR_EMPTY_SHAPE", 2: "QMM_ERR_BAD_KIND", 3: "QMM_ERR_BAD_DTYPE",
    4: "QMM_ERR_COLS_NOT_BLOCK_ALIGNED", 5: "QMM_ERR_WEIGHTS_TOO_SMALL",
    6: "QMM_ERR_ACTIVATIONS_TOO_SMALL", 7: "QMM_ERR_NULL_POINTER", 8: "QMM_ERR_MISALIGNED",
    9: "QMM_ERR_BAD_EXPERT_ID", 10: "QMM_ERR_CUDA", 11: "QMM_ERR_DEVICE_TIMEOUT",
    12: "QMM_ERR_UNIMPLEMENTED", 13: "QMM_ERR_BAD_ARGUMENT", 14: "QMM_ERR_OUTPUT_TOO_SMALL",
    15: "QMM_ERR_WORKSPACE_IN_CAPTURE", 16: "QMM_ERR_NOALLOC_LIMIT", 17: "QMM_ERR_WORKSPACE_TOO_SMALL",
}
STATUS_ID = {v: k for k, v in STATUS.items()}

PATH_AUTO, PATH_GENERIC, PATH_GEMV, PATH_TC, PATH_DEQUANT, PATH_GROUPED, PATH_MOE, PATH_REPACKED = range(8)
FLAG_WEIGHTS_CONST = 1
FLAG_Y_F16 = 2
FLAG_Y_BF16 = 4


class QmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name} ({_lib().qmm_status_str(status).decode()})")


_LIB = None
_P, _I64, _SZ, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libqmm.so not built ({LIB_PATH}); run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        L.qmm_kind_info.argtypes = [_I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]
        L.qmm_row_bytes.argtypes = [_I, _I64]
        L.qmm_row_bytes.restype = _SZ
        L.qmm_status_str.argtypes = [_I]
        L.qmm_status_str.restype = ctypes.c_char_p
        L.qmm_kind_name.argtypes = [_I]
        L.qmm_kind_name.restype = ctypes.c_char_p
        L.qdequant.argtypes = [_I, _P, _SZ, _I64, _I64, _P, _SZ, _P]
        L.qgemv.argtypes = [_I, _P, _SZ, _P, _I, _SZ, _P, _SZ, _I64, _I64, _P]
        L.qgemm.argtypes = [_I, _P, _SZ, _P, _I, _SZ, _P, _SZ, _I64, _I64, _I64, _P]
        L.qgemm_ex.argtypes = [_I, _P, _SZ, _P, _I, _SZ, _P, _SZ, _I64, _I64, _I64, ctypes.c_uint32, _P]
        L.qgemm_noalloc.argtypes = [_I, _P, _SZ, _P, _I, _SZ, _P, _SZ, _I64, _I64, _I64, _P]
        L.qgemm_grouped.argtypes = [_I, _P, _SZ, _SZ, _I, _P, _I, _SZ, _I64, _P, _P, _I64,
                                    _P, _SZ, _I64, _I64, _P]
        L.qrepack.argtypes = [_I, _P, _SZ, _I64, _I64, _P, _SZ, _P]
        L.qrepack_bytes.argtypes = [_I, _I64, _I64]
        L.qrepack_bytes.restype = _SZ
        L.qgemm_repacked.argtypes = [_I, _P, _SZ, _P, _I, _SZ, _P, _SZ, _I64, _I64, _I64, _I, ctypes.c_uint32, _P]
        L.qmoe_ffn.argtypes = [_I, _P, _SZ, _SZ, _P, _SZ, _SZ, _I, _P, _SZ, _I64, _I64, _I64, _P, _P, _I,
                               _P, _SZ, _P, _SZ, _P]
        L.qmoe_ffn_workspace_bytes.argtypes = [_I64, _I, _I64, _I64]
        L.qmoe_ffn_workspace_bytes.restype = _SZ
        L.qmm_check_device_error.argtypes = [_P]
        L.qmm_selftest_wait_timeout.argtypes = [_I64, _P]
        L.qmm_set_path.argtypes = [_I]
        L.qmm_launch_count.restype = ctypes.c_uint64
        L.qmm_shutdown.argtypes = []
        _LIB = L
    return _LIB


def lib():
    """The loaded ctypes library (raw C ABI)."""
    return _lib()


def header_symbols():
    """Function names declared in include/qmm.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*QMM_API\s+(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def _kind(kind) -> int:
    return KIND_ID[kind] if isinstance(kind, str) else int(kind)


def _stream(stream) -> int:
    if stream is not None:
        return int(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _check(rc: int, where: str):
    if rc != 0:
        raise QmmError(rc, where)


def kind_info(kind):
    bb, be = _SZ(), _SZ()
    _check(_lib().qmm_kind_info(_kind(kind), ctypes.byref(bb), ctypes.byref(be)), "qmm_kind_info")
    return bb.value, be.value


def row_bytes(kind, K: int) -> int:
    return _lib().qmm_row_bytes(_kind(kind), K)


def set_path(path: int) -> int:
    """Kernel-path override of the calling thread (0 = automatic)."""
    return _lib().qmm_set_path(path)


def last_path() -> int:
    return _lib().qmm_last_path()


def launch_count() -> int:
    return _lib().qmm_launch_count()


def _xdt(X) -> int:
    import torch
    if X.dtype == torch.float32:
        return F32
    if X.dtype == torch.float16:
        return F16
    raise TypeError(f"activations must be float32 or float16, got {X.dtype}")


def qdequant(kind, blocks, rows: int, cols: int, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=blocks.device)
    _check(_lib().qdequant(_kind(kind), _ptr(blocks), blocks.numel() * blocks.element_size(),
                           rows, cols, _ptr(out), out.numel(), _stream(stream)), "qdequant")
    return out


def _yflag(Y) -> int:
    import torch
    if Y.dtype == torch.float32:
        return 0
    if Y.dtype == torch.float16:
        return FLAG_Y_F16
    if Y.dtype == torch.bfloat16:
        return FLAG_Y_BF16
    raise TypeError(f"outputs must be float32, float16 or bfloat16, got {Y.dtype}")


def qgemm(kind, W, X, M: int, K: int, N: int, Y=None, stream=None, weights_const: bool = False,
          out_dtype=None):
    """Y[n, m] = sum_k W[m, k] X[n, k]; returns Y as an (N, M) tensor, fp32
    unless Y (or out_dtype) is float16 / bfloat16 (rounded once at the store).
    weights_const: W is not written by work still in flight on the stream
    (QMM_FLAG_WEIGHTS_CONST: the GEMV may start streaming it early)."""
    import torch
    if Y is None:
        Y = torch.empty((N, M), dtype=out_dtype or torch.float32, device=W.device)
    flags = (FLAG_WEIGHTS_CONST if weights_const else 0) | _yflag(Y)
    _check(_lib().qgemm_ex(_kind(kind), _ptr(W), W.numel() * W.element_size(), _ptr(X), _xdt(X),
                           X.numel(), _ptr(Y), Y.numel(), M, K, N, flags, _stream(stream)), "qgemm")
    return Y


def qgemm_noalloc(kind, W, X, M: int, K: int, N: int, Y=None, stream=None):
    """qgemm on the tensor-core path without any device allocation by the
    library (scratch in a fixed device array); Y must be given by callers that
    cannot allocate either."""
    import torch
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=W.device)
    _check(_lib().qgemm_noalloc(_kind(kind), _ptr(W), W.numel() * W.element_size(), _ptr(X), _xdt(X),
                                X.numel(), _ptr(Y), Y.numel(), M, K, N, _stream(stream)), "qgemm_noalloc")
    return Y


def qgemv(kind, W, x, M: int, K: int, y=None, stream=None, weights_const: bool = False, out_dtype=None):
    """y[m] = sum_k W[m, k] x[k] (qgemm with N = 1)."""
    import torch
    if y is None:
        y = torch.empty((M,), dtype=out_dtype or torch.float32, device=W.device)
    flags = (FLAG_WEIGHTS_CONST if weights_const else 0) | _yflag(y)
    if flags:
        _check(_lib().qgemm_ex(_kind(kind), _ptr(W), W.numel() * W.element_size(), _ptr(x), _xdt(x),
                               x.numel(), _ptr(y), y.numel(), M, K, 1, flags, _stream(stream)), "qgemv")
    else:
        _check(_lib().qgemv(_kind(kind), _ptr(W), W.numel() * W.element_size(), _ptr(x), _xdt(x),
                            x.numel(), _ptr(y), y.numel(), M, K, _stream(stream)), "qgemv")
    return y


def qgemm_grouped(kind, W, expert_stride: int, n_experts: int, X, x_row, expert_id,
                  M: int, K: int, Y=None, stream=None):
    """Y[r, m] = sum_k W_{expert_id[r]}[m, k] X[x_row[r], k]; returns (n_assign, M)."""
    import torch
    n_assign = x_row.numel()
    if Y is None:
        Y = torch.empty((n_assign, M), dtype=torch.float32, device=W.device)
    n_x_rows = X.numel() // K
    _check(_lib().qgemm_grouped(_kind(kind), _ptr(W), W.numel() * W.element_size(), expert_stride,
                                n_experts, _ptr(X), _xdt(X), X.numel(), n_x_rows, _ptr(x_row),
                                _ptr(expert_id), n_assign, _ptr(Y), Y.numel(), M, K,
                                _stream(stream)), "qgemm_grouped")
    return Y


def qrepack_bytes(kind, rows: int, cols: int) -> int:
    return _lib().qrepack_bytes(_kind(kind), rows, cols)


def qrepack(kind, W, rows: int, cols: int, out=None, stream=None):
    """The repacked (structure-of-arrays) copy of Q8_0 / Q4_0 weights, as a
    CUDA uint8 tensor of the same size."""
    import torch
    if out is None:
        out = torch.empty(max(1, qrepack_bytes(kind, rows, cols)), dtype=torch.uint8, device=W.device)
    _check(_lib().qrepack(_kind(kind), _ptr(W), W.numel() * W.element_size(), rows, cols, _ptr(out), out.numel(),
                          _stream(stream)), "qrepack")
    return out


def qgemm_repacked(kind, R, X, M: int, K: int, N: int, Y=None, split: int = 0, stream=None,
                   weights_const: bool = False, out_dtype=None):
    """qgemm (N <= 8) on a repacked tensor, K split `split` ways (0 = automatic)."""
    import torch
    if Y is None:
        Y = torch.empty((N, M), dtype=out_dtype or torch.float32, device=R.device)
    flags = (FLAG_WEIGHTS_CONST if weights_const else 0) | _yflag(Y)
    _check(_lib().qgemm_repacked(_kind(kind), _ptr(R), R.numel(), _ptr(X), _xdt(X), X.numel(), _ptr(Y), Y.numel(),
                                 M, K, N, split, flags, _stream(stream)), "qgemm_repacked")
    return Y


def qmoe_ffn_workspace_bytes(T: int, top_k: int, d_model: int, d_ff: int) -> int:
    return _lib().qmoe_ffn_workspace_bytes(T, top_k, d_model, d_ff)


def qmoe_ffn(kind, W_gu, gu_stride: int, W_down, down_stride: int, n_experts: int, X, topk_ids, topk_w,
             d_model: int, d_ff: int, Y=None, workspace=None, stream=None):
    """One MoE feed-forward layer: Y[t] = sum_j w[t, j] W_down_e (silu(g) * u),
    (g, u) = W_gu_e x_t, e = topk_ids[t, j]; returns Y as (T, d_model) fp32.
    The scratch comes from `workspace` (a CUDA uint8 tensor of at least
    qmoe_ffn_workspace_bytes(...) bytes), allocated here with torch if None."""
    import torch
    T, top_k = topk_ids.shape
    if Y is None:
        Y = torch.empty((T, d_model), dtype=torch.float32, device=W_gu.device)
    need = qmoe_ffn_workspace_bytes(T, top_k, d_model, d_ff)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=W_gu.device)
    _check(_lib().qmoe_ffn(_kind(kind), _ptr(W_gu), W_gu.numel() * W_gu.element_size(), gu_stride,
                           _ptr(W_down), W_down.numel() * W_down.element_size(), down_stride, n_experts,
                           _ptr(X), X.numel(), T, d_model, d_ff, _ptr(topk_ids), _ptr(topk_w), top_k,
                           _ptr(Y), Y.numel(), _ptr(workspace), workspace.numel(), _stream(stream)), "qmoe_ffn")
    return Y


def selftest_wait_timeout(cycles: int, stream=None):
    """Queue the failure-path self-test kernel (a bounded wait that runs out)."""
    _check(_lib().qmm_selftest_wait_timeout(int(cycles), _stream(stream)), "qmm_selftest_wait_timeout")


def shutdown():
    """Free the library's grown per-device workspaces (later calls regrow them)."""
    _check(_lib().qmm_shutdown(), "qmm_shutdown")


def check_device_error(stream=None) -> int:
    """Synchronize and return (and clear) the device error latch status."""
    return _lib().qmm_check_device_error(_stream(stream))
