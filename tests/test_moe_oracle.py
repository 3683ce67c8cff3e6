"""Pins of the MoE-layer oracle (oracle/moe.py) -- CPU only.

Closed forms chosen so that a plausible mistake in the composition fails one
of them (the sabotage tests show it):
  * odd symmetry: silu(v) - silu(-v) = v, so two experts with gates +I and -I,
    up and down I, routing weights +1 and -1 give y = x^2 exactly;
  * a large positive gate makes silu the identity (error e^-v): y = up-scale
    times x^2;
  * a zero gate gives y = 0 whatever up and down are (silu(0) = 0);
  * the combine is linear in the routing weights and blind to slot order, and
    k slots of one expert with weights summing to one equal that expert alone.
Weights are hand-built Q8_0 blocks with scale 1.0, so every dequantized weight
is the integer code itself.
"""
import numpy as np
import pytest

from gemv_mul_mm_gb300 import synth

D = 32   # d_model = d_ff: one Q8_0 block per row


def q8_rows(mat):
    """Q8_0 bytes of an integer matrix (rows of 32 codes), scale 1.0."""
    mat = np.asarray(mat, dtype=np.int64)
    out = np.zeros((mat.shape[0], 34), dtype=np.uint8)
    out[:, 0], out[:, 1] = 0x00, 0x3C
    out[:, 2:] = mat.astype(np.int8).view(np.uint8)
    return out.reshape(-1)


def experts(gates, ups, downs):
    """gate_up (gate rows then up rows) and down weights of each expert."""
    gu = np.concatenate([q8_rows(np.vstack([g, u])) for g, u in zip(gates, ups)])
    dn = np.concatenate([q8_rows(d) for d in downs])
    return gu, 2 * D * 34, dn, D * 34


def run(orc, gates, ups, downs, x, ids, w, sabotage=0):
    gu, gus, dn, dns = experts(gates, ups, downs)
    return orc.moe_ffn("Q8_0", gu, gus, dn, dns, len(gates), x, ids, w, D, D, sabotage=sabotage)


I = np.eye(D, dtype=np.int64)


def odd_symmetry(orc, sabotage=0):
    x = (np.arange(D) - 15.5).astype(np.float32)[None, :] / 4
    y, tol = run(orc, [I, -I], [I, I], [I, I], x, np.array([[0, 1]]), np.array([[1.0, -1.0]]), sabotage)
    return y[0], (x[0].astype(np.float64)) ** 2, tol[0]


def test_odd_symmetry_gives_x_squared(orc):
    y, want, tol = odd_symmetry(orc)
    # h is rounded to fp32 before the down projection: 2^-24 of each |h|
    assert np.max(np.abs(y - want) / (1.0 + want)) <= 1e-6
    assert np.all(tol > 0)


@pytest.mark.parametrize("sab", [1, 2, 3, 4])
def test_odd_symmetry_pin_fires_on_sabotage(orc, sab):
    y, want, _ = odd_symmetry(orc, sabotage=sab)
    assert np.max(np.abs(y - want)) > 1e-3


def test_large_gate_makes_silu_the_identity(orc):
    x = (20.0 + np.arange(D)).astype(np.float32)[None, :]
    y, _ = run(orc, [I], [2 * I], [I], x, np.array([[0]]), np.array([[0.5]]))
    want = x[0].astype(np.float64) ** 2
    assert np.max(np.abs(y[0] - want) / want) <= 1e-8


def test_zero_gate_gives_zero(orc):
    rng = np.random.default_rng(3)
    up = rng.integers(-9, 9, (D, D))
    dn = rng.integers(-9, 9, (D, D))
    x = rng.standard_normal((2, D)).astype(np.float32)
    y, _ = run(orc, [0 * I], [up], [dn], x, np.array([[0], [0]]), np.array([[0.7], [1.3]]))
    assert np.all(y == 0.0)


def random_layer(seed, E=4, k=3, T=3):
    rng = np.random.default_rng(seed)
    gates = [rng.integers(-3, 4, (D, D)) for _ in range(E)]
    ups = [rng.integers(-3, 4, (D, D)) for _ in range(E)]
    downs = [rng.integers(-3, 4, (D, D)) for _ in range(E)]
    x = (rng.standard_normal((T, D)) / 4).astype(np.float32)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    return gates, ups, downs, x, ids, rng


def test_combine_is_linear_and_blind_to_slot_order(orc):
    gates, ups, downs, x, ids, rng = random_layer(5)
    w1, w2 = rng.random(ids.shape), rng.random(ids.shape)
    y1, _ = run(orc, gates, ups, downs, x, ids, w1)
    y2, _ = run(orc, gates, ups, downs, x, ids, w2)
    y12, _ = run(orc, gates, ups, downs, x, ids, w1 + w2)
    assert np.allclose(y12, y1 + y2, rtol=1e-12, atol=1e-12)
    perm = np.array([2, 0, 1])
    yp, _ = run(orc, gates, ups, downs, x, ids[:, perm], w1[:, perm])
    assert np.allclose(yp, y1, rtol=1e-12, atol=1e-12)


def test_slots_of_one_expert_with_unit_weight_sum_equal_the_expert(orc):
    gates, ups, downs, x, _, rng = random_layer(7, T=2)
    ids = np.full((2, 3), 2, dtype=np.int32)
    w = rng.random((2, 3))
    w /= w.sum(axis=1, keepdims=True)
    y, _ = run(orc, gates, ups, downs, x, ids, w)
    y1, _ = run(orc, gates, ups, downs, x, ids[:, :1], np.ones((2, 1)))
    assert np.allclose(y, y1, rtol=1e-12, atol=1e-12)


def test_tolerance_covers_a_perturbed_intermediate(orc):
    # the derived bar must admit a device whose gate_up output is off by its
    # own bar: recompute the layer by hand from perturbed g, u and check
    gates, ups, downs, x, ids, rng = random_layer(9, E=3, k=2, T=2)
    w = rng.random(ids.shape)
    y, tol = run(orc, gates, ups, downs, x, ids, w)
    gu, gus, dn, dns = experts(gates, ups, downs)
    T, k = ids.shape
    eid = ids.reshape(-1)
    g_u, gu_tol = orc.grouped("Q8_0", gu, gus, len(gates), x, np.repeat(np.arange(T, dtype=np.int32), k),
                              eid, 2 * D, D)
    sgn = np.where(rng.random(g_u.shape) < 0.5, -1.0, 1.0)
    pert = g_u + sgn * gu_tol                    # every gate/up output off by its whole bar
    g, u = pert[:, :D], pert[:, D:]
    h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
    o, _ = orc.grouped("Q8_0", dn, dns, len(gates), h, np.arange(T * k, dtype=np.int32), eid, D, D)
    yp = np.einsum("tk,tkm->tm", w, o.reshape(T, k, D))
    assert np.all(np.abs(yp - y) <= tol)
