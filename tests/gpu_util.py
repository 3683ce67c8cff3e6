"""Helpers shared by the GPU parity tests (comparison against the oracle)."""
from __future__ import annotations

import numpy as np

SENTINEL = -1.0e30


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def sentinel(shape, offset_elems: int = 0):
    """fp32 device buffer prefilled with the sentinel; optionally offset by a few
    elements so that the view is not 16-byte aligned."""
    import torch
    n = int(np.prod(shape))
    buf = torch.full((n + offset_elems,), SENTINEL, dtype=torch.float32, device="cuda")
    return buf[offset_elems:].view(*shape)


def assert_bits(got: np.ndarray, want: np.ndarray, tag: str = ""):
    """Bit-exact fp32 equality; any NaN matches any NaN."""
    got = np.ascontiguousarray(got, dtype=np.float32)
    want = np.ascontiguousarray(want, dtype=np.float32)
    assert got.shape == want.shape, (got.shape, want.shape)
    gb, wb = got.view(np.uint32), want.view(np.uint32)
    bad = (gb != wb) & ~(np.isnan(got) & np.isnan(want))
    n = int(bad.sum())
    if n:
        i = np.flatnonzero(bad.reshape(-1))[:5]
        raise AssertionError(f"{tag}: {n} of {got.size} elements differ in bits; first at {i}: "
                             f"got {got.reshape(-1)[i]} want {want.reshape(-1)[i]}")


def assert_within(got: np.ndarray, y: np.ndarray, tol: np.ndarray, tag: str = ""):
    """|got - y| <= tol per element (tol = 1e-3 * sum|w x| + 1e-6 from the
    oracle) and no sentinel left behind."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == y.shape, (got.shape, y.shape)
    untouched = int((got == SENTINEL).sum())
    assert untouched == 0, f"{tag}: {untouched} outputs never written"
    err = np.abs(got - y)
    bad = ~(err <= tol)
    n = int(bad.sum())
    if n:
        i = np.flatnonzero(bad.reshape(-1))[:5]
        raise AssertionError(f"{tag}: {n} of {got.size} outputs outside tolerance; first at {i}: "
                             f"got {got.reshape(-1)[i]} want {y.reshape(-1)[i]} tol {tol.reshape(-1)[i]}")
    return float(np.max(err / tol)) if err.size else 0.0
