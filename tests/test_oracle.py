"""The oracle against its pins (CPU only): golden values the pages print,
exhaustive scalar sweeps, hand-built blocks, one-hot fields, round trips,
cross-format invariants and brute force -- plus sabotage builds showing that
each pin fires on a plausible mistake."""
import numpy as np
import pytest

import oracle
from tests import pins

PIN_CHECKS = [
    pins.check_f16_exhaustive, pins.check_e8m0_exhaustive, pins.check_scalar_golden,
    pins.check_iq4nl_codebook, pins.check_e2m1_codebook, pins.check_mxfp4_scale,
    pins.check_q4_0_nibbles, pins.check_q8_0, pins.check_q5_0_qh,
    pins.check_q4_k, pins.check_q5_k, pins.check_q6_k, pins.check_q2_k, pins.check_q3_k,
    pins.check_iq4_xs, pins.check_q4_1, pins.check_q5_1, pins.check_q8_1,
    pins.check_legacy_min_formats_reduce, pins.check_gemm_brute_force,
]


@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda c: c.__name__)
def test_pin(orc, check):
    bad = check(orc)
    assert not bad, "\n".join(bad[:20])


# sabotage id -> the pin that must fire (planted in the oracle, on the CPU)
SABOTAGE = {
    1: pins.check_q5_0_qh,        # Q5_0 fifth-bit shift off by four for the high half
    2: pins.check_iq4_xs,         # IQ4_XS scales_h shifted by sub-block, not group
    3: pins.check_q3_k,           # Q3_K hmask bias inverted
    4: pins.check_q4_0_nibbles,   # Q4_0 nibble halves swapped
    5: pins.check_q6_k,           # Q6_K scale index per 32 instead of per 16
    6: pins.check_q4_k,           # Q4_K min term dropped
    7: pins.check_e2m1_codebook,  # MXFP4 code 8 as +0.0
    8: pins.check_gemm_brute_force,  # activation index transposed inside a pair
    9: pins.check_q4_1,           # Q4_1 min subtracted instead of added
    10: pins.check_q8_1,          # Q8_1 codes read from byte 2, as in Q8_0
}


@pytest.mark.parametrize("sab", sorted(SABOTAGE))
def test_pin_fires_on_sabotage(sab):
    bad = oracle.load(sabotage=sab)
    assert bad.lib.oracle_sabotage_id() == sab
    assert SABOTAGE[sab](bad), f"sabotage {sab} went unnoticed by {SABOTAGE[sab].__name__}"


def test_geometry(orc):
    want = {"Q8_0": (34, 32), "Q4_0": (18, 32), "Q5_0": (22, 32), "Q4_K": (144, 256),
            "Q5_K": (176, 256), "Q6_K": (210, 256), "Q2_K": (84, 256), "Q3_K": (110, 256),
            "IQ4_NL": (18, 32), "IQ4_XS": (136, 256), "MXFP4": (17, 32),
            "Q4_1": (20, 32), "Q5_1": (24, 32), "Q8_1": (36, 32)}
    for k, g in want.items():
        assert orc.geometry(k) == g


def test_gemm_is_fp64_matmul_of_dequant(orc):
    """The product reduces to a library fp64 matmul of the dequantized matrix."""
    from gemv_mul_mm_gb300 import synth
    for kind in oracle.KINDS:
        be = orc.geometry(kind)[1]
        M, K, N = 37, 2 * 256, 5
        w = synth.quant_weights(kind, M, K, seed=99 + oracle.KIND_ID[kind])
        x = synth.activations(N, K, seed=5)
        deq = orc.dequant(kind, w, M, K).astype(np.float64)
        y, tol = orc.gemm(kind, w, M, K, x, N)
        ref = x.astype(np.float64) @ deq.T
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
        mag = np.abs(x.astype(np.float64)) @ np.abs(deq).T
        np.testing.assert_allclose(tol, 1e-3 * mag + 1e-6, rtol=1e-12)
        assert be in (32, 256)


def test_gemm_f16_activations(orc):
    from gemv_mul_mm_gb300 import synth
    M, K, N = 9, 256, 3
    w = synth.quant_weights("Q4_K", M, K, seed=3)
    x16 = synth.activations(N, K, seed=4, dtype="f16")
    y16, _ = orc.gemm("Q4_K", w, M, K, x16, N)
    y32, _ = orc.gemm("Q4_K", w, M, K, x16.astype(np.float32), N)
    np.testing.assert_array_equal(y16, y32)


def test_gemm_at_matches_gemm(orc):
    from gemv_mul_mm_gb300 import synth
    M, K, N = 50, 512, 4
    w = synth.quant_weights("Q6_K", M, K, seed=11)
    x = synth.activations(N, K, seed=12)
    y, tol = orc.gemm("Q6_K", w, M, K, x, N)
    n_idx = np.array([0, 3, 2, 1, 3])
    m_idx = np.array([0, 49, 17, 3, 0])
    ys, ts = orc.gemm_at("Q6_K", w, M, K, x, n_idx, m_idx)
    np.testing.assert_array_equal(ys, y[n_idx, m_idx])
    np.testing.assert_array_equal(ts, tol[n_idx, m_idx])


def test_grouped_is_per_assignment_gemm(orc):
    from gemv_mul_mm_gb300 import synth
    E, M, K = 5, 24, 64
    rb = orc.row_bytes("Q4_0", K)
    w = synth.quant_weights("Q4_0", E * M, K, seed=21)
    x = synth.activations(4, K, seed=22)
    x_row = np.array([0, 0, 3, 2, 1, 3], dtype=np.int32)
    eid = np.array([4, 1, 0, 4, 2, 3], dtype=np.int32)
    y, tol = orc.grouped("Q4_0", w, M * rb, E, x, x_row, eid, M, K)
    for r in range(x_row.size):
        we = w[eid[r] * M * rb:(eid[r] + 1) * M * rb]
        yr, tr = orc.gemm("Q4_0", we, M, K, x[x_row[r]:x_row[r] + 1], 1)
        np.testing.assert_array_equal(y[r], yr[0])
        np.testing.assert_array_equal(tol[r], tr[0])
    ys, _ = orc.grouped("Q4_0", w, M * rb, E, x, x_row, eid, M, K,
                        r_idx=np.array([5, 0]), m_idx=np.array([23, 1]))
    np.testing.assert_array_equal(ys, [y[5, 23], y[0, 1]])


def test_bad_expert_rejected(orc):
    w = np.zeros(18 * 2, dtype=np.uint8)
    x = np.zeros((1, 32), dtype=np.float32)
    with pytest.raises(ValueError):
        orc.grouped("Q4_0", w, 18, 1, x, np.array([0], np.int32), np.array([1], np.int32), 1, 32)
