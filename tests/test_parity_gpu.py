"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Dequant: bit-exact (NaN matches NaN). GEMV/GEMM: |y - y_ref| <= 1e-3 *
sum_k |w x| + 1e-6 per element, with every sentinel-prefilled output
overwritten. Small shapes span several row groups / chunks and a ragged tail;
the pages' full workloads are checked on all outputs where the oracle is fast
and on sampled outputs otherwise.
"""
import numpy as np
import pytest

import oracle
from gemv_mul_mm_gb300 import synth
from tests.gpu_util import SENTINEL, assert_bits, assert_within, dev, sentinel

pytestmark = pytest.mark.gpu

KINDS = oracle.KINDS
ELEMS = {k: synth.block_geometry(k)[1] for k in KINDS}


@pytest.fixture(scope="module")
def Q():
    import torch  # noqa: F401
    from gemv_mul_mm_gb300 import build as qbuild
    from gemv_mul_mm_gb300 import qmm
    qbuild.build()
    qmm.set_path(0)
    yield qmm
    qmm.set_path(0)


def raw_random_blocks(kind, rows, K, seed):
    """Random bytes everywhere, scale fields included (NaN/Inf/subnormal scales)."""
    n = rows * synth.row_bytes(kind, K)
    return synth.Stream(seed).bytes(n)


# ---------------------------------------------------------------------------
# dequant
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("variant", ["scaled", "raw", "unaligned"])
def test_dequant_bit_exact(Q, orc, kind, variant):
    import torch
    rows, cols = 131, 4 * ELEMS[kind]
    seed = 1000 + oracle.KIND_ID[kind]
    if variant == "raw":
        w = raw_random_blocks(kind, rows, cols, seed)
    else:
        w = synth.quant_weights(kind, rows, cols, seed)
    want = orc.dequant(kind, w, rows, cols)
    if variant == "unaligned":
        buf = torch.zeros(w.size + 1, dtype=torch.uint8, device="cuda")
        buf[1:] = dev(w)
        wd = buf[1:]
        out = sentinel((rows, cols), offset_elems=1)
    else:
        wd = dev(w)
        out = sentinel((rows, cols))
    Q.qdequant(kind, wd, rows, cols, out=out)
    got = out.cpu().numpy()
    assert not np.any(got == SENTINEL)
    assert_bits(got, want, f"{kind} {variant}")


@pytest.mark.parametrize("kind", KINDS)
def test_dequant_workload_size(Q, orc, kind):
    """The pages' workload tensors (decode GEMV, K-quant and codebook GEMMs)."""
    cfg = {"Q8_0": synth.DECODE, "Q4_0": synth.DECODE, "Q5_0": synth.DECODE,
           "IQ4_NL": synth.CODEBOOK, "IQ4_XS": synth.CODEBOOK, "MXFP4": synth.CODEBOOK}.get(kind, synth.KQUANT)
    M, K = cfg["M"], cfg["K"]
    if kind == "Q5_0":
        w = synth.quant_weights(kind, M, K, synth.config_seed(1, kind))
    else:
        w = synth.workload_weights(cfg, kind)
    out = sentinel((M, K))
    Q.qdequant(kind, dev(w), M, K, out=out)
    got = out.cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(8), np.arange(M - 8, M),
                                     np.random.default_rng(3).integers(0, M, 256)]))
    rb = synth.row_bytes(kind, K)
    for r in rows:
        want = orc.dequant(kind, w[r * rb:(r + 1) * rb], 1, K)
        assert_bits(got[r:r + 1], want, f"{kind} row {r}")
    assert not np.any(got == SENTINEL)


# ---------------------------------------------------------------------------
# GEMV / GEMM, small shapes, every path
# ---------------------------------------------------------------------------
def k_values(kind):
    be = ELEMS[kind]
    return sorted({be * 3, 2048, 4096 + 512 if be == 32 else 4096 + 2048})


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("N", [1, 3, 8, 33])
@pytest.mark.parametrize("xdt", ["f32", "f16"])
def test_gemm_small(Q, orc, kind, N, xdt):
    M = 130
    for K in k_values(kind):
        seed = 77 + 31 * oracle.KIND_ID[kind] + K
        w = synth.quant_weights(kind, M, K, seed)
        x = synth.activations(N, K, seed + 1, xdt)
        y, tol = orc.gemm(kind, w, M, K, x, N)
        for path in (Q.PATH_AUTO, Q.PATH_GENERIC, Q.PATH_GEMV):
            Q.set_path(path)
            Y = sentinel((N, M))
            try:
                Q.qgemm(kind, dev(w), dev(x), M, K, N, Y=Y)
            except Q.QmmError as e:
                assert path == Q.PATH_GEMV and e.name == "QMM_ERR_UNIMPLEMENTED"
                continue
            finally:
                Q.set_path(0)
            assert_within(Y.cpu().numpy(), y, tol, f"{kind} M={M} K={K} N={N} {xdt} path={path}")


@pytest.mark.parametrize("kind", ["Q4_0", "Q8_0", "Q4_K", "MXFP4"])
def test_unaligned_weights_take_generic_path(Q, orc, kind):
    import torch
    M, K, N = 70, 2048, 3
    w = synth.quant_weights(kind, M, K, 5)
    x = synth.activations(N, K, 6)
    y, tol = orc.gemm(kind, w, M, K, x, N)
    buf = torch.zeros(w.size + 3, dtype=torch.uint8, device="cuda")
    buf[3:] = dev(w)
    Y = sentinel((N, M))
    Q.qgemm(kind, buf[3:], dev(x), M, K, N, Y=Y)
    assert Q.last_path() == Q.PATH_GENERIC
    assert_within(Y.cpu().numpy(), y, tol, kind)


def test_qgemv_is_qgemm_column(Q):
    M, K = 300, 4096
    for kind in ("Q4_0", "Q8_0", "Q6_K"):
        w = dev(synth.quant_weights(kind, M, K, 9))
        x = dev(synth.activations(1, K, 10))
        y1 = Q.qgemv(kind, w, x, M, K).cpu().numpy()
        y2 = Q.qgemm(kind, w, x, M, K, 1).cpu().numpy()[0]
        np.testing.assert_array_equal(y1, y2)


# ---------------------------------------------------------------------------
# the pages' workloads
# ---------------------------------------------------------------------------
def test_tiny_q4_0_qgemm(Q, orc):
    c = synth.TINY
    w = synth.workload_weights(c, "Q4_0")
    x = synth.workload_x(c, "Q4_0")
    y, tol = orc.gemm("Q4_0", w, c["M"], c["K"], x, c["N"])
    Y = sentinel((c["N"], c["M"]))
    Q.qgemm("Q4_0", dev(w), dev(x), c["M"], c["K"], c["N"], Y=Y)
    assert_within(Y.cpu().numpy(), y, tol, "tiny Q4_0")


@pytest.mark.parametrize("kind", ["Q8_0", "Q4_0"])
def test_decode_gemv_full(Q, orc, kind):
    """The decode workload as configured: every output against the oracle's
    own element-indexed product."""
    c = synth.DECODE
    M, K = c["M"], c["K"]
    w = synth.workload_weights(c, kind)
    x = synth.workload_x(c, kind)
    y, tol = orc.gemm(kind, w, M, K, x, 1, nthreads=8)
    Y = sentinel((1, M))
    Q.qgemv(kind, dev(w), dev(x), M, K, y=Y.view(-1))
    assert Q.last_path() == Q.PATH_GEMV
    assert_within(Y.cpu().numpy(), y, tol, f"decode {kind}")


@pytest.mark.parametrize("kind", [k for k in KINDS if k not in ("Q8_0", "Q4_0")])
def test_decode_shape_gemv_every_kind(Q, orc, kind):
    """Every other kind at the decode shape (M 14336, K 4096, one fp32
    column, the per-kind table of the bench): all outputs against the oracle's
    dequant + fp64 product."""
    c = synth.DECODE
    M, K = c["M"], c["K"]
    w = synth.quant_weights(kind, M, K, synth.config_seed(1, kind))
    x = synth.workload_x(c, "Q4_0")
    y, tol = oracle_full_product(orc, kind, w, M, K, x)
    Y = sentinel((1, M))
    Q.qgemv(kind, dev(w), dev(x), M, K, y=Y.view(-1), weights_const=True)
    assert Q.last_path() == Q.PATH_GEMV
    assert_within(Y.cpu().numpy(), y, tol, f"decode shape {kind}")


@pytest.mark.parametrize("kind", ["Q4_0", "Q8_0", "IQ4_NL"])
@pytest.mark.parametrize("M", [4100, 14336])
def test_gemv_back_to_back_with_weight_prefetch(Q, orc, kind, M):
    """Consecutive GEMVs on one stream, weights streamed early (programmatic
    dependent launch): each call must still see the previous call's output as
    its input (y of call i is x of call i+1) and write every output."""
    import torch
    K = 4096
    w = [synth.quant_weights(kind, M, K, 40 + i) for i in range(3)]
    x0 = synth.activations(1, K, 41)
    wd = [dev(wi) for wi in w]
    xs, ys = [dev(x0)], []
    for i in range(3):
        y = sentinel((M,))
        Q.qgemv(kind, wd[i], xs[-1], M, K, y=y, weights_const=True)
        ys.append(y)
        xs.append((y[:K] * 0.05).contiguous())      # next input depends on this output
    torch.cuda.synchronize()
    for i in range(3):
        # step i's input is what the GPU produced at step i-1; its whole
        # output (unscaled) is compared at the bare tolerance
        xin = xs[i].cpu().numpy().reshape(1, -1)
        yref, tol = orc.gemm(kind, w[i], M, K, xin, 1)
        assert_within(ys[i].cpu().numpy().reshape(1, -1), yref, tol, f"{kind} chain step {i}")


def sample_positions(N, M, count, seed):
    rng = np.random.default_rng(seed)
    n = np.concatenate([[0, 0, N - 1, N - 1], rng.integers(0, N, count)])
    m = np.concatenate([[0, M - 1, 0, M - 1], rng.integers(0, M, count)])
    return n, m


def oracle_full_product(orc, kind, w, M, K, x):
    """Every output of a workload-sized product: the oracle's bit-exact fp32
    dequant followed by an fp64 matmul (the form that the oracle's own GEMM
    reduces to, pinned by tests/test_oracle.py), with the same per-element
    tolerance 1e-3 * sum_k |w x| + 1e-6."""
    deq = orc.dequant(kind, w, M, K).astype(np.float64)
    x64 = np.asarray(x, dtype=np.float64).reshape(-1, K)
    y = x64 @ deq.T
    tol = 1e-3 * (np.abs(x64) @ np.abs(deq).T) + 1e-6
    return y, tol


@pytest.mark.parametrize("cfg,kind", [(synth.KQUANT, k) for k in synth.KQUANT["kinds"]] +
                         [(synth.CODEBOOK, k) for k in synth.CODEBOOK["kinds"]] +
                         [(synth.LEGACY1, k) for k in synth.LEGACY1["kinds"]])
def test_prefill_gemm_workload(Q, orc, cfg, kind):
    """The prefill workloads as configured, in the launch configuration the
    bench times: every output against the oracle's dequant + fp64 matmul, and
    a sample of outputs against the oracle's own element-indexed GEMM."""
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    w = synth.workload_weights(cfg, kind)
    x = synth.workload_x(cfg, kind)
    Y = sentinel((N, M))
    Q.qgemm(kind, dev(w), dev(x), M, K, N, Y=Y)
    path = Q.last_path()
    got = Y.cpu().numpy()
    assert not np.any(got == SENTINEL)
    n, m = sample_positions(N, M, 400, 11)
    y, tol = orc.gemm_at(kind, w, M, K, x, n, m)
    assert_within(got[n, m], y, tol, f"{kind} prefill sampled (path {path})")
    y, tol = oracle_full_product(orc, kind, w, M, K, x)
    assert_within(got, y, tol, f"{kind} prefill, all {N * M} outputs (path {path})")


# Tile schedules of the tensor-core GEMM. When the 128 x 128 output tiles do
# not fill the SMs evenly, consecutive CTAs share a tile's K range and a second
# kernel adds their partial tiles; otherwise each CTA owns one tile.
#   many_partials: 6 tiles (ragged in M and N), 32 super-steps each, on every
#                  SM -- each tile's sum is split over about 25 CTAs;
#   whole_inside:  190 tiles (ragged in M) of 8 super-steps over the SMs --
#                  CTAs take one or two partial tiles and whole tiles between;
#   one_per_cta:   152 tiles of one super-step -- one wave, no sharing.
SCHEDULES = {"many_partials": (300, 8192, 150), "whole_inside": (24300, 2048, 128),
             "one_per_cta": (19456, 256, 128)}


@pytest.mark.parametrize("case,kind", [("many_partials", "Q4_K"), ("many_partials", "IQ4_NL"),
                                       ("many_partials", "Q6_K"), ("whole_inside", "Q4_K"),
                                       ("whole_inside", "MXFP4"), ("one_per_cta", "Q5_K"),
                                       ("one_per_cta", "IQ4_NL"), ("many_partials", "Q5_1"),
                                       ("whole_inside", "Q4_1"), ("one_per_cta", "Q8_1")])
def test_gemm_tile_schedules(Q, orc, case, kind):
    M, K, N = SCHEDULES[case]
    seed = sum(map(ord, case + kind))
    w = synth.quant_weights(kind, M, K, seed)
    x = synth.activations(N, K, seed + 1, "f16")
    Y = sentinel((N, M))
    Q.qgemm(kind, dev(w), dev(x), M, K, N, Y=Y)
    assert Q.last_path() == Q.PATH_TC
    assert Q.check_device_error() == 0
    got = Y.cpu().numpy()
    assert not np.any(got == SENTINEL)
    # whole token columns (every tile along M) and whole weight rows (every
    # tile along N): first, middle and last of each
    cols = np.array([0, N // 2 + 1, N - 1]) if case != "whole_inside" else np.array([0, N - 1])
    rows = np.array([0, M // 2, M - 1])
    n = np.concatenate([np.repeat(cols, M), np.tile(np.arange(N), rows.size)])
    m = np.concatenate([np.tile(np.arange(M), cols.size), np.repeat(rows, N)])
    y, tol = orc.gemm_at(kind, w, M, K, x, n, m)
    assert_within(got[n, m], y, tol, f"{kind} {case}")


def test_gemm_graph_replay_is_bit_identical_to_eager(Q, orc):
    # 16 tiles of 16 super-steps: the K ranges are shared over all SMs and
    # the partial tiles are added in a fixed order, so a replayed graph gives
    # the eager call's bits exactly
    import torch
    kind, (M, K, N) = "IQ4_NL", (1000, 4096, 130)
    w = synth.quant_weights(kind, M, K, 91)
    x = synth.activations(N, K, 92, "f16")
    Wd, Xd = dev(w), dev(x)
    Ye = Q.qgemm(kind, Wd, Xd, M, K, N)          # eager: the workspace grows here
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    Yg = sentinel((N, M))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        Q.qgemm(kind, Wd, Xd, M, K, N, Y=Yg, stream=s.cuda_stream)
    for _ in range(2):
        Yg.fill_(SENTINEL)
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(Ye, Yg)
    assert Q.check_device_error() == 0
    n, m = sample_positions(N, M, 300, 93)
    y, tol = orc.gemm_at(kind, w, M, K, x, n, m)
    assert_within(Ye.cpu().numpy()[n, m], y, tol, "eager")


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_workspace_growth_during_capture_is_refused(Q, orc):
    # activation sums of 16384 tokens x 64 super-blocks (33.5 MB) plus the
    # partial tiles: more workspace than any other test needs, so the
    # library must grow it -- which it refuses inside a capture, before
    # launching anything; the capture ends cleanly and the next eager call
    # grows the workspace and computes
    import torch
    kind, (M, K, N) = "Q4_K", (256, 16384, 16384)
    w = synth.quant_weights(kind, M, K, 95)
    Wd = dev(w)
    Xd = torch.empty((N, K), dtype=torch.float16, device="cuda")
    Y = torch.empty((N, M), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(Q.QmmError) as ei:
        with torch.cuda.graph(g, stream=s):
            Q.qgemm(kind, Wd, Xd, M, K, N, Y=Y, stream=s.cuda_stream)
    assert ei.value.name == "QMM_ERR_WORKSPACE_IN_CAPTURE"
    torch.cuda.synchronize()
    x = synth.activations(64, K, 96, "f16")
    Xd[:64].copy_(dev(x).view(64, K))
    Q.qgemm(kind, Wd, Xd, M, K, N, Y=Y)
    torch.cuda.synchronize()
    assert Q.check_device_error() == 0
    n, m = sample_positions(64, M, 200, 97)
    y, tol = orc.gemm_at(kind, w, M, K, x, n, m)
    assert_within(Y.cpu().numpy()[n, m], y, tol, "after the refused capture")


def test_shutdown_frees_workspaces_and_calls_regrow_them(Q, orc):
    import torch
    kind, (M, K, N) = "Q4_K", (300, 4096, 150)     # activation sums + shared tiles
    w = synth.quant_weights(kind, M, K, 98)
    x = synth.activations(N, K, 99, "f16")
    Wd, Xd = dev(w), dev(x)
    Y1 = Q.qgemm(kind, Wd, Xd, M, K, N)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    Q.shutdown()
    Q.shutdown()                                    # nothing left to free: still fine
    assert torch.cuda.mem_get_info()[0] > free0     # the workspace went back to the device
    Y2 = Q.qgemm(kind, Wd, Xd, M, K, N)              # grows it again
    torch.cuda.synchronize()
    assert Q.check_device_error() == 0
    assert torch.equal(Y1, Y2)


@pytest.mark.parametrize("T", synth.MOE["tokens"])
@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_moe_grouped(Q, orc, T, which):
    p = synth.moe_problem(T, which)
    M, K = p["M"], p["K"]
    Y = sentinel((p["x_row"].size, M))
    Q.qgemm_grouped(p["kind"], dev(p["w"]), p["stride"], p["n_experts"], dev(p["x"]),
                    dev(p["x_row"]), dev(p["expert_id"]), M, K, Y=Y)
    got = Y.cpu().numpy()
    assert not np.any(got == SENTINEL)
    assert Q.check_device_error() == 0
    nr = p["x_row"].size
    rng = np.random.default_rng(T)
    r_idx = np.concatenate([[0, nr - 1], rng.integers(0, nr, 300)])
    m_idx = np.concatenate([[0, M - 1], rng.integers(0, M, 300)])
    y, tol = orc.grouped(p["kind"], p["w"], p["stride"], p["n_experts"], p["x"], p["x_row"],
                         p["expert_id"], M, K, r_idx=r_idx, m_idx=m_idx)
    assert_within(got[r_idx, m_idx], y, tol, f"moe {which} T={T}")


def test_grouped_is_per_assignment_gemv(Q, orc):
    E, M, K = 6, 96, 512
    rb = synth.row_bytes("Q4_0", K)
    w = synth.quant_weights("Q4_0", E * M, K, 3)
    x = synth.activations(5, K, 4)
    x_row = np.array([4, 0, 0, 2, 3, 1, 4], dtype=np.int32)
    eid = np.array([5, 0, 3, 3, 1, 2, 0], dtype=np.int32)
    Y = Q.qgemm_grouped("Q4_0", dev(w), M * rb, E, dev(x), dev(x_row), dev(eid), M, K).cpu().numpy()
    _, tol = orc.grouped("Q4_0", w, M * rb, E, x, x_row, eid, M, K)
    for r in range(x_row.size):
        we = dev(w[eid[r] * M * rb:(eid[r] + 1) * M * rb])
        yr = Q.qgemv("Q4_0", we, dev(x[x_row[r]]), M, K).cpu().numpy()
        # two different kernels, each within tol of the exact value
        assert np.all(np.abs(Y[r] - yr) <= 2 * tol[r]), r


def test_grouped_bad_expert_is_flagged(Q):
    E, M, K = 2, 64, 256
    rb = synth.row_bytes("Q4_0", K)
    w = synth.quant_weights("Q4_0", E * M, K, 3)
    x = synth.activations(2, K, 4)
    x_row = np.array([0, 1, 1], dtype=np.int32)
    eid = np.array([1, 7, 0], dtype=np.int32)      # 7 is out of range
    Y = Q.qgemm_grouped("Q4_0", dev(w), M * rb, E, dev(x), dev(x_row), dev(eid), M, K)
    assert Q.check_device_error() == Q.STATUS_ID["QMM_ERR_BAD_EXPERT_ID"]
    got = Y.cpu().numpy()
    assert np.all(np.isnan(got[1])) and np.all(np.isfinite(got[[0, 2]]))
    assert Q.check_device_error() == 0               # the latch was cleared


def test_empty_and_refused_shapes(Q):
    import torch
    w = torch.zeros(18 * 8, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, dtype=torch.float32, device="cuda")
    with pytest.raises(Q.QmmError) as e:
        Q.qgemm("Q4_0", w, x, 1, 256, 0, Y=torch.zeros(1, device="cuda"))
    assert e.value.name == "QMM_ERR_EMPTY_SHAPE"
    with pytest.raises(Q.QmmError) as e:
        Q.qgemm("Q4_0", w, x, 2, 256, 1)
    assert e.value.name == "QMM_ERR_WEIGHTS_TOO_SMALL"


# ---------------------------------------------------------------------------
# degenerate blocks: nonzero scales, every code decoding to a zero weight
# ---------------------------------------------------------------------------
def zero_valued_block(kind: str) -> np.ndarray:
    """One block whose scales are nonzero but whose every element decodes to
    exactly 0 (the oracle confirms it), so the exact product is 0 and the
    tolerance is the bare 1e-6: a kernel that cancels a fixed code offset in
    fp32 (sum (q + c) x - c sum x) would miss it."""
    bb, _ = synth.block_geometry(kind)
    b = np.zeros(bb, dtype=np.uint8)
    d = np.frombuffer(np.float16(3.0e-3).tobytes(), dtype=np.uint8)
    if kind == "Q8_0":
        b[0:2] = d                                   # codes 0
    elif kind == "Q4_0":
        b[0:2] = d
        b[2:18] = 0x88                               # q = 8 -> q - 8 = 0
    elif kind == "Q5_0":
        b[0:2] = d
        b[2:6] = 0xFF                                # 5th bit set, low nibbles 0 -> q = 16
    elif kind in ("Q4_K", "Q5_K"):
        b[0:2] = d
        b[2:4] = d                                   # dmin nonzero
        b[4:8] = 0x05                                # sub-scales 5 (j < 4)
        b[12:16] = 0x05                              # sub-scales 5 (j >= 4), mins 0
    elif kind == "Q6_K":
        b[128:192] = 0xAA                            # high bits 2, low 0 -> q = 32
        b[192:208] = 3
        b[208:210] = d
    elif kind == "Q2_K":
        b[0:16] = 0x05                               # scale 5, min 0; codes 0
        b[80:82] = d
        b[82:84] = d
    elif kind == "Q3_K":
        b[0:32] = 0xFF                               # no -4 bias; codes 0
        b[96:108] = 0x11
        b[108:110] = d
    elif kind == "IQ4_XS":
        b[0:2] = d
        b[2:4] = 0xAA                                # ls = 32 -> group scale 0
        b[8:136] = (np.arange(128) * 37 % 256).astype(np.uint8)
    elif kind == "MXFP4":
        b[0] = 127
        b[1:17] = np.tile(np.array([0x00, 0x08, 0x80, 0x88], dtype=np.uint8), 4)  # +0 and -0
    elif kind in ("Q4_1", "Q5_1"):
        b[0:2] = d                                   # codes 0, min 0 (a nonzero min with
                                                     # nonzero codes cancels only to rounding)
    elif kind == "Q8_1":
        b[0:2] = d
        b[2:4] = d                                   # the unread field, nonzero; codes 0
    else:
        raise ValueError(kind)
    return b


@pytest.mark.parametrize("kind", [k for k in KINDS if k != "IQ4_NL"])
@pytest.mark.parametrize("N,xdt", [(1, "f32"), (4, "f32"), (33, "f16")])
def test_zero_valued_codes_with_nonzero_scales(Q, orc, kind, N, xdt):
    M, K = 96, 4096
    nb = M * (K // ELEMS[kind])
    w = np.tile(zero_valued_block(kind), nb)
    assert not np.any(orc.dequant(kind, w, M, K)), "the hand-built block must decode to zeros"
    x = synth.activations(N, K, 5 + N, xdt)
    y, tol = orc.gemm(kind, w, M, K, x, N)
    Y = sentinel((N, M))
    Q.qgemm(kind, dev(w), dev(x), M, K, N, Y=Y)
    assert_within(Y.cpu().numpy(), y, tol, f"{kind} zero codes N={N} path={Q.last_path()}")


# ---------------------------------------------------------------------------
# largest shapes: activations the streaming kernel stages, and past them
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kind", ["Q4_0", "Q8_0"])
@pytest.mark.parametrize("K,path", [(32768, "gemv"), (65536, "generic")])
def test_long_rows_stream_or_fall_back(Q, orc, kind, K, path):
    """A 32768-element row still has its activations staged in shared memory
    by the streaming GEMV; a 65536-element row does not fit and must take the
    generic kernel. Both must match the oracle."""
    M = 64
    w = synth.quant_weights(kind, M, K, 31)
    x = synth.activations(1, K, 32)
    y, tol = orc.gemm(kind, w, M, K, x, 1)
    Y = sentinel((1, M))
    Q.qgemv(kind, dev(w), dev(x), M, K, y=Y.view(-1))
    assert Q.last_path() == (Q.PATH_GEMV if path == "gemv" else Q.PATH_GENERIC)
    assert_within(Y.cpu().numpy(), y, tol, f"{kind} K={K}")


# ---------------------------------------------------------------------------
# failure path: a bounded wait that runs out is reported, the context survives
# ---------------------------------------------------------------------------
def test_device_timeout_is_reported_and_context_survives(Q, orc):
    assert Q.check_device_error() == 0
    Q.selftest_wait_timeout(1 << 22)           # a few milliseconds of waiting
    assert Q.check_device_error() == Q.STATUS_ID["QMM_ERR_DEVICE_TIMEOUT"]
    assert Q.check_device_error() == 0         # the latch was cleared
    # the context is still usable: a GEMV right after matches the oracle
    M, K = 96, 1024
    w = synth.quant_weights("Q8_0", M, K, 51)
    x = synth.activations(1, K, 52)
    y, tol = orc.gemm("Q8_0", w, M, K, x, 1)
    Y = sentinel((1, M))
    Q.qgemv("Q8_0", dev(w), dev(x), M, K, y=Y.view(-1))
    assert_within(Y.cpu().numpy(), y, tol, "after timeout")
    assert Q.check_device_error() == 0


# ---------------------------------------------------------------------------
# grouped product: limits of the streaming kernel, crowded experts, f16, odd K
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["experts_1024", "experts_1025", "crowded_expert", "f16_x", "k96"])
def test_grouped_edge_cases(Q, orc, case):
    rng = np.random.default_rng(sum(map(ord, case)))
    kind, M, K, E, T = "Q4_0", 64, 256, 16, 6
    xdt = "f32"
    if case == "experts_1024":
        E = 1024
    elif case == "experts_1025":
        E = 1025
    elif case == "f16_x":
        xdt = "f16"
    elif case == "k96":
        K = 96
    rb = synth.row_bytes(kind, K)
    w = synth.quant_weights(kind, E * M, K, 71)
    x = synth.activations(T, K, 72, xdt)
    n = 24
    x_row = rng.integers(0, T, n).astype(np.int32)
    eid = rng.integers(0, E, n).astype(np.int32)
    if case == "crowded_expert":
        eid[:11] = 3                      # eleven assignments of one expert, some repeated rows
        x_row[:11] = np.array([0, 1, 1, 2, 5, 5, 5, 4, 3, 0, 2], dtype=np.int32)
    Y = sentinel((n, M))
    Q.qgemm_grouped(kind, dev(w), M * rb, E, dev(x), dev(x_row), dev(eid), M, K, Y=Y)
    streaming = case in ("experts_1024", "crowded_expert", "f16_x")
    assert Q.last_path() == (Q.PATH_GROUPED if streaming else Q.PATH_GENERIC)
    assert Q.check_device_error() == 0
    y, tol = orc.grouped(kind, w, M * rb, E, x, x_row, eid, M, K)
    assert_within(Y.cpu().numpy(), y, tol, f"grouped {case}")


# ---------------------------------------------------------------------------
# fp32 activations on the tensor-core path, 16-bit outputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg,kind", [(synth.KQUANT, "Q4_K"), (synth.KQUANT, "Q6_K"), (synth.KQUANT, "Q2_K"),
                                      (synth.CODEBOOK, "IQ4_NL"), (synth.CODEBOOK, "MXFP4"),
                                      (synth.LEGACY1, "Q5_1")])
def test_prefill_gemm_fp32_activations(Q, orc, cfg, kind):
    """fp32 activations at the workload shapes run on the tensor cores as
    (hi, lo) f16 pairs; every output against the oracle."""
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    w = synth.workload_weights(cfg, kind)
    x = synth.workload_x(cfg, kind).astype(np.float32)
    x = x + synth.activations(N, K, 123, "f32") * 1e-3      # bits below f16's precision
    Y = sentinel((N, M))
    Q.qgemm(kind, dev(w), dev(x), M, K, N, Y=Y)
    assert Q.last_path() == Q.PATH_TC
    y, tol = oracle_full_product(orc, kind, w, M, K, x)
    assert_within(Y.cpu().numpy(), y, tol, f"{kind} fp32 X, all {N * M} outputs")


@pytest.mark.parametrize("kind", ["Q4_K", "Q5_K", "IQ4_XS", "Q8_0", "Q4_1", "Q5_1"])
def test_fp32_activations_of_any_magnitude(Q, orc, kind):
    """Token rows far outside f16's range (1e30, 1e-30, mixed): the per-row
    power-of-two scale keeps the (hi, lo) split exact to about 2^-22."""
    M, K, N = 256, 1024, 40
    w = synth.quant_weights(kind, M, K, 61)
    x = synth.activations(N, K, 62, "f32").astype(np.float64)
    mag = np.array([1e30, 1e-30, 3e4, 7e4, 1e-7, 1.0, 2.0 ** -140, 1e20] * 5)[:N]
    x = (x * mag[:, None]).astype(np.float32)
    x[5, 7] = 0.0
    x[9, :] = 0.0                                            # an all-zero row
    Y = sentinel((N, M))
    Q.qgemm(kind, dev(w), dev(x), M, K, N, Y=Y)
    assert Q.last_path() == Q.PATH_TC
    y, tol = orc.gemm(kind, w, M, K, x, N)
    assert_within(Y.cpu().numpy(), y, tol, f"{kind} fp32 X wide range")


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("kind,N,path", [("Q4_0", 1, "gemv"), ("Q6_K", 3, "gemv"), ("Q4_K", 33, "tc"),
                                         ("IQ4_NL", 130, "tc_shared"), ("MXFP4", 40, "tc_fp32"),
                                         ("Q5_0", 5, "generic")])
def test_sixteen_bit_outputs(Q, orc, out, kind, N, path):
    """f16 / bf16 outputs are the product rounded once at the store: within
    the stated bar plus half an ulp of the output type, on every kernel."""
    import torch
    M, K = (1000, 4096) if path == "tc_shared" else (300, 2048)
    xdt = "f32" if path in ("gemv", "generic", "tc_fp32") else "f16"
    w = synth.quant_weights(kind, M, K, 70 + N)
    x = synth.activations(N, K, 71 + N, xdt)
    y, tol = orc.gemm(kind, w, M, K, x, N)
    tdt = torch.float16 if out == "f16" else torch.bfloat16
    Y = torch.full((N, M), float("nan"), dtype=tdt, device="cuda")
    if path == "generic":
        Q.set_path(Q.PATH_GENERIC)
    try:
        Q.qgemm(kind, dev(w), dev(x), M, K, N, Y=Y)
    finally:
        Q.set_path(0)
    want_path = {"gemv": Q.PATH_GEMV, "generic": Q.PATH_GENERIC}.get(path, Q.PATH_TC)
    assert Q.last_path() == want_path
    got = Y.float().cpu().numpy().astype(np.float64)
    assert not np.isnan(got).any(), "outputs never written"
    half_ulp = np.abs(y) * (2.0 ** -11 if out == "f16" else 2.0 ** -8)
    bad = ~(np.abs(got - y) <= tol + half_ulp)
    assert not bad.any(), f"{int(bad.sum())} outputs outside the bar"


# ---------------------------------------------------------------------------
# the tensor-core GEMM's f16 operand fold at its worst case
# ---------------------------------------------------------------------------
def fold_worst_block(kind):
    """A block whose every element's code times sub-scale is an odd integer just
    above 2048, where f16 rounds by half a spacing of 2 (relative 4.8e-4), all
    with the same sign: Q6_K sc = 77, q - 32 = 27 (2079); IQ4_XS ls - 32 = -25,
    KV = -83 (2075). d has 11 significant bits."""
    bb, _ = synth.block_geometry(kind)
    b = np.zeros(bb, dtype=np.uint8)
    d = (0x1BFF).to_bytes(2, "little")
    if kind == "Q6_K":
        b[0:128] = 0xBB                  # low nibbles 11 (q = 59 = 11 + 16 * 3)
        b[128:192] = 0xFF                # high 2-bit fields 3
        b[192:208] = 77                  # int8 sub-scales
        b[208:210] = list(d)
    else:
        b[0:2] = list(d)
        b[2:4] = 0x00                    # scales_h: high bits 0
        b[4:8] = 0x77                    # scales_l: ls = 7 -> ls - 32 = -25
        b[8:136] = 0x22                  # codes 2 -> KV = -83
    return b


@pytest.mark.parametrize("kind", ["Q6_K", "IQ4_XS"])
def test_operand_fold_worst_case(Q, orc, kind):
    """Every weight of a long row rounds the same way when its integer operand
    is folded into f16, and every activation is positive, so the rounding adds
    up coherently over K = 16384: the product stays within the bar."""
    M, K, N = 128, 16384, 33
    w = np.tile(fold_worst_block(kind), M * (K // 256))
    x = (0.5 + 0.5 * synth.Stream(91).uniform(N * K)).astype(np.float16).reshape(N, K)
    deq = orc.dequant(kind, w, 1, K)[0]
    assert np.all(deq == deq[0]) and deq[0] != 0, "one value everywhere"
    y, tol = orc.gemm(kind, w, M, K, x, N)
    Y = sentinel((N, M))
    Q.qgemm(kind, dev(w), dev(x), M, K, N, Y=Y)
    assert Q.last_path() == Q.PATH_TC
    assert_within(Y.cpu().numpy(), y, tol, f"{kind} operand fold, worst case")


@pytest.mark.parametrize("lo,hi", [(100, 140), (103, 127), (118, 142)])
def test_mxfp4_exponent_spread_on_tensor_cores(Q, orc, lo, hi):
    """MXFP4 on the tensor cores folds each block's exponent into its operands
    relative to the largest of its 256-element super-step: spreads up to 23
    are exact; at 24 the odd halves round, beyond it a block contributes
    nothing (f16 subnormals end at 2^-24). With random codes the largest
    block dominates and the loss stays far inside the bar."""
    M, K, N = 256, 4096, 40
    w = synth.quant_weights("MXFP4", M, K, 31 + lo, e8m0_lo=lo, e8m0_hi=hi)
    x = synth.activations(N, K, 32 + lo, "f16")
    y, tol = orc.gemm("MXFP4", w, M, K, x, N)
    Y = sentinel((N, M))
    Q.qgemm("MXFP4", dev(w), dev(x), M, K, N, Y=Y)
    assert Q.last_path() == Q.PATH_TC
    assert_within(Y.cpu().numpy(), y, tol, f"MXFP4 exponents {lo}..{hi}")
