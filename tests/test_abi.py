"""The C-ABI library builds, loads and exports every symbol include/qmm.h
declares; host-side validation refuses bad arguments by name before any CUDA
call (no GPU needed: none of these calls reaches a launch)."""
import ctypes

import pytest

from gemv_mul_mm_gb300 import build as qbuild
from gemv_mul_mm_gb300 import qmm


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return qmm.lib()


def test_exports_every_declared_symbol(L):
    syms = qmm.header_symbols()
    assert {"qdequant", "qgemv", "qgemm", "qgemm_grouped", "qmm_check_device_error"} <= set(syms)
    for s in syms:
        assert hasattr(L, s), f"{s} declared in qmm.h but not exported"


def test_kind_table(L):
    want = {"Q8_0": (34, 32), "Q4_0": (18, 32), "Q5_0": (22, 32), "Q4_K": (144, 256),
            "Q5_K": (176, 256), "Q6_K": (210, 256), "Q2_K": (84, 256), "Q3_K": (110, 256),
            "IQ4_NL": (18, 32), "IQ4_XS": (136, 256), "MXFP4": (17, 32),
            "Q4_1": (20, 32), "Q5_1": (24, 32), "Q8_1": (36, 32)}
    assert set(want) == set(qmm.KINDS)
    for k, g in want.items():
        assert qmm.kind_info(k) == g
        assert L.qmm_kind_name(qmm.KIND_ID[k]).decode() == k
        assert qmm.row_bytes(k, 4096) == 4096 // g[1] * g[0]
        assert qmm.row_bytes(k, g[1] + 16) == 0       # not a whole number of blocks
    assert L.qmm_kind_name(14) is None and L.qmm_kind_name(-1) is None
    # absent formats are not silently mapped (ferrox-cuda mul_mm.rs kind_by_name):
    # the grid-codebook kinds have no id at all
    assert L.qmm_row_bytes(14, 256) == 0
    assert not {"IQ1_S", "IQ2_XXS", "IQ3_S"} & set(qmm.KINDS)
    bb, be = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.qmm_kind_info(42, ctypes.byref(bb), ctypes.byref(be)) == qmm.STATUS_ID["QMM_ERR_BAD_KIND"]


def test_status_strings(L):
    for code in range(18):
        assert L.qmm_status_str(code)
    assert L.qmm_status_str(999) == b"unknown status"


FAKE = 0x10000  # never dereferenced: every call below is refused before a launch


def _gemm(L, kind=1, W=FAKE, wb=1 << 30, X=FAKE, xdt=0, xe=1 << 30, Y=FAKE, ye=1 << 30,
          M=64, K=256, N=1):
    return L.qgemm(kind, W, wb, X, xdt, xe, Y, ye, M, K, N, None)


@pytest.mark.parametrize("args,status", [
    (dict(kind=14), "QMM_ERR_BAD_KIND"),
    (dict(kind=-1), "QMM_ERR_BAD_KIND"),
    (dict(M=0), "QMM_ERR_EMPTY_SHAPE"),
    (dict(N=0), "QMM_ERR_EMPTY_SHAPE"),
    (dict(K=0), "QMM_ERR_EMPTY_SHAPE"),
    (dict(M=-3), "QMM_ERR_BAD_ARGUMENT"),
    (dict(W=0), "QMM_ERR_NULL_POINTER"),
    (dict(Y=0), "QMM_ERR_NULL_POINTER"),
    (dict(xdt=7), "QMM_ERR_BAD_DTYPE"),
    (dict(X=FAKE + 2), "QMM_ERR_MISALIGNED"),
    (dict(Y=FAKE + 1), "QMM_ERR_MISALIGNED"),
    (dict(K=48), "QMM_ERR_COLS_NOT_BLOCK_ALIGNED"),
    (dict(kind=3, K=288), "QMM_ERR_COLS_NOT_BLOCK_ALIGNED"),
    (dict(wb=64 * 144 - 1), "QMM_ERR_WEIGHTS_TOO_SMALL"),
    (dict(xe=255), "QMM_ERR_ACTIVATIONS_TOO_SMALL"),
    (dict(N=4, xe=3 * 256), "QMM_ERR_ACTIVATIONS_TOO_SMALL"),
    (dict(N=2, ye=127), "QMM_ERR_OUTPUT_TOO_SMALL"),
])
def test_qgemm_refusals(L, args, status):
    assert _gemm(L, **args) == qmm.STATUS_ID[status]


def test_qgemv_and_dequant_refusals(L):
    S = qmm.STATUS_ID
    assert L.qgemv(1, FAKE, 1 << 30, FAKE, 0, 255, FAKE, 64, 64, 256, None) == S["QMM_ERR_ACTIVATIONS_TOO_SMALL"]
    assert L.qgemv(1, FAKE, 1 << 30, FAKE, 1, 256, FAKE, 64, 64, 0, None) == S["QMM_ERR_EMPTY_SHAPE"]
    assert L.qdequant(1, FAKE, 18 * 7, 2, 128, FAKE, 256, None) == S["QMM_ERR_WEIGHTS_TOO_SMALL"]
    assert L.qdequant(1, FAKE, 18 * 8, 2, 128, FAKE, 255, None) == S["QMM_ERR_OUTPUT_TOO_SMALL"]
    assert L.qdequant(3, FAKE, 1 << 20, 2, 100, FAKE, 1 << 20, None) == S["QMM_ERR_COLS_NOT_BLOCK_ALIGNED"]
    assert L.qdequant(1, 0, 1 << 20, 2, 128, FAKE, 1 << 20, None) == S["QMM_ERR_NULL_POINTER"]
    assert L.qdequant(1, FAKE, 1 << 20, 0, 128, FAKE, 1 << 20, None) == S["QMM_ERR_EMPTY_SHAPE"]


def test_grouped_refusals(L):
    S = qmm.STATUS_ID
    rb = 8 * 18

    def g(**kw):
        a = dict(kind=1, W=FAKE, wb=1 << 30, stride=64 * rb, ne=4, X=FAKE, xdt=0, xe=1 << 20,
                 nx=2, xr=FAKE, eid=FAKE, na=3, Y=FAKE, ye=1 << 20, M=64, K=256)
        a.update(kw)
        return L.qgemm_grouped(a["kind"], a["W"], a["wb"], a["stride"], a["ne"], a["X"], a["xdt"],
                               a["xe"], a["nx"], a["xr"], a["eid"], a["na"], a["Y"], a["ye"],
                               a["M"], a["K"], None)
    assert g(na=0) == S["QMM_ERR_EMPTY_SHAPE"]
    assert g(xr=0) == S["QMM_ERR_NULL_POINTER"]
    assert g(eid=FAKE + 2) == S["QMM_ERR_MISALIGNED"]
    assert g(stride=64 * rb - 1) == S["QMM_ERR_BAD_EXPERT_ID"]
    assert g(ne=0) == S["QMM_ERR_BAD_EXPERT_ID"]
    assert g(wb=3 * 64 * rb + 64 * rb - 1) == S["QMM_ERR_WEIGHTS_TOO_SMALL"]
    assert g(xe=2 * 256 - 1) == S["QMM_ERR_ACTIVATIONS_TOO_SMALL"]
    assert g(ye=3 * 64 - 1) == S["QMM_ERR_OUTPUT_TOO_SMALL"]


def test_path_override_is_per_thread(L):
    import threading
    assert qmm.set_path(1) == 0
    seen = []
    t = threading.Thread(target=lambda: seen.append(qmm.set_path(2)))
    t.start()
    t.join()
    assert seen == [0]                 # another thread starts from the default
    assert qmm.set_path(0) == 1        # and did not change this thread's setting
    assert qmm.set_path(9) == -1
    assert qmm.set_path(0) == 0


def test_qgemm_ex_flags(L):
    S = qmm.STATUS_ID
    args = (1, FAKE, 1 << 30, FAKE, 0, 1 << 30, FAKE, 1 << 30, 64, 256)
    # unknown flag bits, and both 16-bit output types at once, are refused
    # before anything else is looked at
    assert L.qgemm_ex(*args, 1, 8, None) == S["QMM_ERR_BAD_ARGUMENT"]
    assert L.qgemm_ex(*args, 1, 0x80000000, None) == S["QMM_ERR_BAD_ARGUMENT"]
    assert L.qgemm_ex(*args, 1, qmm.FLAG_Y_F16 | qmm.FLAG_Y_BF16, None) == S["QMM_ERR_BAD_ARGUMENT"]
    # a 16-bit output needs 2-byte alignment, an fp32 one 4-byte
    for flag, y, want in ((qmm.FLAG_Y_F16, FAKE + 1, "QMM_ERR_MISALIGNED"),
                          (qmm.FLAG_Y_BF16, FAKE + 1, "QMM_ERR_MISALIGNED"),
                          (0, FAKE + 2, "QMM_ERR_MISALIGNED"),
                          (qmm.FLAG_Y_F16, FAKE + 2, "QMM_ERR_COLS_NOT_BLOCK_ALIGNED")):
        assert L.qgemm_ex(1, FAKE, 1 << 30, FAKE, 0, 1 << 30, y, 1 << 30, 64, 48 if flag else 256, 1, flag,
                          None) == S[want], (flag, y)
    # the known flag passes validation like qgemm (refused later for the shape)
    assert L.qgemm_ex(1, FAKE, 1 << 30, FAKE, 0, 1 << 30, FAKE, 1 << 30, 64, 48, 1,
                      qmm.FLAG_WEIGHTS_CONST, None) == S["QMM_ERR_COLS_NOT_BLOCK_ALIGNED"]


def test_selftest_refuses_bad_cycle_counts(L):
    import ctypes
    for bad in (0, -5, (1 << 32) + 1):
        assert L.qmm_selftest_wait_timeout(ctypes.c_int64(bad), None) == 13   # QMM_ERR_BAD_ARGUMENT


def test_moe_layer_refusals(L):
    S = qmm.STATUS_ID
    rb_gu, rb_dn = 8 * 18, 24 * 18      # Q4_0, d_model 256, d_ff 768

    def m(**kw):
        a = dict(kind=1, gu=FAKE, gub=1 << 30, gus=2 * 768 * rb_gu, dn=FAKE, dnb=1 << 30, dns=256 * rb_dn,
                 ne=4, x=FAKE, xe=1 << 20, T=2, dm=256, dff=768, ids=FAKE, w=FAKE, k=2, y=FAKE, ye=1 << 20,
                 ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return L.qmoe_ffn(a["kind"], a["gu"], a["gub"], a["gus"], a["dn"], a["dnb"], a["dns"], a["ne"], a["x"],
                          a["xe"], a["T"], a["dm"], a["dff"], a["ids"], a["w"], a["k"], a["y"], a["ye"], a["ws"],
                          a["wsb"], None)
    assert m(kind=14) == S["QMM_ERR_BAD_KIND"]
    assert m(T=0) == S["QMM_ERR_EMPTY_SHAPE"]
    assert m(k=-1) == S["QMM_ERR_BAD_ARGUMENT"]
    assert m(ids=0) == S["QMM_ERR_NULL_POINTER"]
    assert m(ws=FAKE + 16) == S["QMM_ERR_MISALIGNED"]
    assert m(x=FAKE + 4) == S["QMM_ERR_MISALIGNED"]
    assert m(dff=760) == S["QMM_ERR_COLS_NOT_BLOCK_ALIGNED"]
    assert m(gus=2 * 768 * rb_gu - 1) == S["QMM_ERR_BAD_EXPERT_ID"]
    assert m(dnb=3 * 256 * rb_dn + 256 * rb_dn - 1) == S["QMM_ERR_WEIGHTS_TOO_SMALL"]
    assert m(xe=2 * 256 - 1) == S["QMM_ERR_ACTIVATIONS_TOO_SMALL"]
    assert m(ye=2 * 256 - 1) == S["QMM_ERR_OUTPUT_TOO_SMALL"]
    need = qmm.qmoe_ffn_workspace_bytes(2, 2, 256, 768)
    assert need > 4 * 2 * (2 * 768 + 256)
    assert m(wsb=need - 1) == S["QMM_ERR_WORKSPACE_TOO_SMALL"]
    assert qmm.qmoe_ffn_workspace_bytes(0, 2, 256, 768) == 0
