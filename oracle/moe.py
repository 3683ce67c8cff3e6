"""CPU oracle of a mixture-of-experts feed-forward layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and bench.py's CPU-oracle leg may
use this module; the product path never imports it.

The layer around the expert-grouped product (the Qwen3-30B-A3B decode that the
inferencelayer 0.2.8 ``src/cublas_prefill.rs`` page quotes its per-token
weight traffic for). The pages do not spell the layer out; the reading taken:
for token t and routing slot j (expert e = ids[t, j], weight w[t, j]):

    g = W_gate_e x_t,  u = W_up_e x_t          (the gate_up projection: gate
                                                 rows first, then up rows)
    h = silu(g) * u,   silu(v) = v / (1 + e^-v)  (SwiGLU)
    o = W_down_e h
    y_t = sum_j w[t, j] o                        (top-k weighted combine)

The two projections are the oracle's own grouped product (fp32 element
dequant, fp64 sums; pinned in tests/test_oracle.py); SwiGLU and the combine
are evaluated in fp64 here. The activation h fed to the down projection is
rounded to fp32, as the grouped product takes fp32 activations.

Tolerance. Each projection's bar is 1e-3 * sum |w x| + 1e-6 per output. A
device that meets it on g and u (errors dg, du) produces h with error at most

    dh = |silu'(g)| |u| dg + |silu(g)| du + 1.1 dg du + 2^-21 |h|

(|silu'| <= 1.1 everywhere; the last term covers fp32 evaluation of silu and
the product), and the down projection of that h, against the down bar of the
exact h, adds sum_k |W_down[m, k]| (dh[k] + 2^-23 |h[k]|). The combine adds
the weighted sum of those, plus fp32 rounding of the sum. This is the bound
the per-product bar implies for the composed layer; parity unpinned beyond
the closed-form pins (the pages fix neither SwiGLU nor the combine).

``sabotage`` plants one mistake for the pin tests: 1 swaps gate and up, 2
drops the silu, 3 ignores the routing weights, 4 sums silu over the up half.
"""
from __future__ import annotations

import numpy as np


def silu(v):
    return v / (1.0 + np.exp(-v))


def moe_ffn(orc, kind, w_gu, gu_stride, w_down, down_stride, n_experts, x, ids, weights,
            d_model, d_ff, sabotage: int = 0, nthreads: int = 1):
    """(y, tol), float64 arrays of shape (T, d_model)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, d_model)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.asarray(weights, dtype=np.float64)
    T, k = ids.shape
    A = T * k
    x_row = np.repeat(np.arange(T, dtype=np.int32), k)
    eid = ids.reshape(-1)
    gu, gu_tol = orc.grouped(kind, w_gu, gu_stride, n_experts, x, x_row, eid, 2 * d_ff, d_model,
                             nthreads=nthreads)
    g, u = gu[:, :d_ff], gu[:, d_ff:]
    dg, du = gu_tol[:, :d_ff], gu_tol[:, d_ff:]
    if sabotage == 1:
        g, u = u, g
    if sabotage == 2:
        h = g * u
    elif sabotage == 4:
        h = silu(u) * u
    else:
        h = silu(g) * u
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = np.minimum(np.abs(sig * (1.0 + g * (1.0 - sig))), 1.1)
    dh = dsilu * np.abs(u) * dg + np.abs(silu(g)) * du + 1.1 * dg * du + 2.0 ** -21 * np.abs(h)
    h32 = h.astype(np.float32)
    o, o_tol = orc.grouped(kind, w_down, down_stride, n_experts, h32, np.arange(A, dtype=np.int32), eid,
                           d_model, d_ff, nthreads=nthreads)
    # propagate dh (and the fp32 rounding of h) through |W_down| of each used expert
    rb = orc.row_bytes(kind, d_ff)
    prop = np.zeros((A, d_model))
    for e in np.unique(eid):
        rows = np.flatnonzero(eid == e)
        we = w_down[int(e) * down_stride:int(e) * down_stride + d_model * rb]
        absw = np.abs(orc.dequant(kind, we, d_model, d_ff).astype(np.float64))
        prop[rows] = (dh[rows] + 2.0 ** -23 * np.abs(h[rows])) @ absw.T
    wts = np.ones_like(weights) if sabotage == 3 else weights
    o3 = o.reshape(T, k, d_model)
    y = np.einsum("tk,tkm->tm", wts, o3)
    aw = np.abs(weights)[:, :, None]
    tol = ((o_tol + prop).reshape(T, k, d_model) * aw).sum(axis=1)
    tol += 2.0 ** -21 * (aw * np.abs(o3)).sum(axis=1) + 1e-6
    return y, tol
