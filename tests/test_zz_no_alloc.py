"""qgemm_noalloc, called through the C ABI, against the oracle and against qgemm.

qgemm_noalloc is the entry point for callers that cannot let the library
allocate device memory: serving runtimes that reserve all of the GPU's memory
at start-up and hand out only their own pools, and hot paths where an
allocation's implicit device synchronisation is not allowed. It keeps its
scratch in a fixed device array instead of a grown workspace. Every output
must match the oracle within the suite's tolerance, and the existing entry
point (qgemm) within the same tolerance, also on the second of two calls in a
row (the array still holds the first call's contents). This file is collected
last, so a run that stops at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest

from gemv_mul_mm_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    import torch  # noqa: F401
    from gemv_mul_mm_gb300 import build as qbuild
    from gemv_mul_mm_gb300 import qmm
    qbuild.build()
    qmm.set_path(0)
    return qmm


def _noalloc(Q, kind, W, X, Y, M, K, N):
    import torch
    L = Q.lib()
    return L.qgemm_noalloc(Q.KIND_ID[kind], ctypes.c_void_p(W.data_ptr()), W.numel(),
                           ctypes.c_void_p(X.data_ptr()), Q.F16, X.numel(),
                           ctypes.c_void_p(Y.data_ptr()), Y.numel(), M, K, N,
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("kind", ["Q4_K", "Q2_K", "Q5_K", "IQ4_NL", "Q4_1"])
def test_noalloc_matches_oracle_and_qgemm_on_two_calls_in_a_row(Q, orc, kind):
    import torch
    problems = [(384, 2048, 160, 11), (256, 4096, 96, 12)]   # (M, K, N, seed)
    outs = []
    for M, K, N, seed in problems:
        w = synth.quant_weights(kind, M, K, seed)
        x = synth.activations(N, K, seed + 1, "f16")
        Wd, Xd = torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda()
        Yn = torch.full((N, M), -1e30, dtype=torch.float32, device="cuda")
        assert _noalloc(Q, kind, Wd, Xd, Yn, M, K, N) == 0
        outs.append((w, x, Wd, Xd, Yn, M, K, N))
    torch.cuda.synchronize()
    assert Q.check_device_error() == 0
    for w, x, Wd, Xd, Yn, M, K, N in outs:
        Yq = Q.qgemm(kind, Wd, Xd, M, K, N)
        got, other = Yn.cpu().numpy().astype(np.float64), Yq.cpu().numpy().astype(np.float64)
        assert not np.any(got == -1e30), "output not fully written"
        y, tol = orc.gemm(kind, w, M, K, x, N)
        bad = ~(np.abs(got - y) <= tol)
        assert not bad.any(), f"{int(bad.sum())} outputs outside the oracle's tolerance"
        bad = ~(np.abs(got - other) <= tol)
        assert not bad.any(), f"{int(bad.sum())} outputs differ from qgemm's by more than the tolerance"


def test_noalloc_refuses_oversize_and_unsupported(Q):
    import torch
    M, K = 128, 4096
    w = torch.zeros(M * synth.row_bytes("Q2_K", K), dtype=torch.uint8, device="cuda")
    # Q2_K needs N * (K / 256) * 64 bytes of scratch: 4097 tokens exceed 4 MiB
    N = 4097
    x = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    y = torch.zeros((N, M), dtype=torch.float32, device="cuda")
    assert _noalloc(Q, "Q2_K", w, x, y, M, K, N) == Q.STATUS_ID["QMM_ERR_NOALLOC_LIMIT"]
    # fp32 activations are not on the tensor-core path
    x32 = torch.zeros((8, K), dtype=torch.float32, device="cuda")
    L = Q.lib()
    rc = L.qgemm_noalloc(Q.KIND_ID["Q2_K"], ctypes.c_void_p(w.data_ptr()), w.numel(),
                         ctypes.c_void_p(x32.data_ptr()), Q.F32, x32.numel(),
                         ctypes.c_void_p(y.data_ptr()), y.numel(), M, K, 8,
                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == Q.STATUS_ID["QMM_ERR_UNIMPLEMENTED"]
