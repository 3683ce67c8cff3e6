"""qrepack and qgemm_repacked (split-K streaming GEMV) against the CPU layout
and the oracle, through the C ABI."""
import numpy as np
import pytest

from gemv_mul_mm_gb300 import synth
from tests.gpu_util import assert_within, dev, sentinel
from tests.test_repack_layout import repack_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    import torch  # noqa: F401
    from gemv_mul_mm_gb300 import build as qbuild
    from gemv_mul_mm_gb300 import qmm
    qbuild.build()
    qmm.set_path(0)
    return qmm


@pytest.mark.parametrize("kind", ["Q8_0", "Q4_0"])
def test_repack_bytes_match_the_layout(Q, kind):
    import torch
    rows, cols = 130, 2048
    w = synth.quant_weights(kind, rows, cols, 50)
    buf = torch.zeros(w.size + 1, dtype=torch.uint8, device="cuda")
    buf[1:] = dev(w)                                           # unaligned source
    out = Q.qrepack(kind, buf[1:], rows, cols)
    assert np.array_equal(out.cpu().numpy(), repack_np(kind, w, rows, cols))


@pytest.mark.parametrize("kind", ["Q8_0", "Q4_0"])
@pytest.mark.parametrize("M,K,N,split,xdt", [(130, 1024, 1, 0, "f32"), (130, 1024, 3, 2, "f32"),
                                             (2048, 4096, 1, 0, "f32"), (2048, 4096, 8, 4, "f16"),
                                             (256, 4096, 1, 16, "f32"), (1000, 2048, 2, 1, "f32"),
                                             (14336, 4096, 1, 0, "f32"), (2048, 14336, 1, 0, "f32"),
                                             (2048, 14336, 5, 0, "f32")])
def test_repacked_gemv_matches_oracle(Q, orc, kind, M, K, N, split, xdt):
    w = synth.quant_weights(kind, M, K, 51 + M + N)
    x = synth.activations(N, K, 52 + N, xdt)
    R = Q.qrepack(kind, dev(w), M, K)
    Y = sentinel((N, M))
    Q.qgemm_repacked(kind, R, dev(x), M, K, N, Y=Y, split=split)
    assert Q.last_path() == Q.PATH_REPACKED
    assert Q.check_device_error() == 0
    y, tol = orc.gemm(kind, w, M, K, x, N, nthreads=8)
    assert_within(Y.cpu().numpy(), y, tol, f"{kind} repacked M={M} K={K} N={N} split={split}")


def test_repacked_refusals(Q):
    import torch
    M, K = 64, 1024
    R = torch.zeros(M * synth.row_bytes("Q4_0", K), dtype=torch.uint8, device="cuda")
    x = torch.zeros(K, dtype=torch.float32, device="cuda")
    for split, name in ((3, "QMM_ERR_BAD_ARGUMENT"), (-1, "QMM_ERR_BAD_ARGUMENT")):
        with pytest.raises(Q.QmmError) as e:
            Q.qgemm_repacked("Q4_0", R, x, M, K, 1, split=split)
        assert e.value.name == name
    with pytest.raises(Q.QmmError) as e:
        Q.qgemm_repacked("Q6_K", R, x, M, K, 1)
    assert e.value.name == "QMM_ERR_UNIMPLEMENTED"
    with pytest.raises(Q.QmmError) as e:
        Q.qrepack("Q4_0", R, M, 800)
    assert e.value.name == "QMM_ERR_COLS_NOT_BLOCK_ALIGNED"
