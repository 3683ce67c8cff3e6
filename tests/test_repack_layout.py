"""The repacked layout (qrepack) pinned on the CPU, as the Vulkore
quant_test.cpp page checks its load-time repack: the repacked tensor must
reconstruct every element bit-exactly. The repack and the reconstruction here
are written from the layout's description (include/qmm.h, qrepack); the
element values come from the oracle's dequant of the native blocks."""
import numpy as np
import pytest

import oracle
from gemv_mul_mm_gb300 import synth

CODE = {"Q8_0": 32, "Q4_0": 16}


def repack_np(kind, w, rows, cols):
    """Native blocks -> units of eight blocks: the eight code fields, then the
    eight f16 scales."""
    bb = CODE[kind] + 2
    units = w.reshape(rows * cols // 256, 8, bb)
    codes = units[:, :, 2:].reshape(units.shape[0], -1)
    scales = units[:, :, :2].reshape(units.shape[0], -1)
    return np.concatenate([codes, scales], axis=1).reshape(-1)


def reconstruct(kind, rp, rows, cols):
    """Every element of the repacked tensor, from its code and scale fields."""
    cb = CODE[kind]
    u = rp.reshape(rows * cols // 256, 8 * (cb + 2))
    d = u[:, 8 * cb:].copy().view(np.float16).astype(np.float32)            # [units, 8]
    c = u[:, :8 * cb].reshape(-1, 8, cb)
    if kind == "Q8_0":
        q = c.view(np.int8).astype(np.float32)                               # element j = code byte j
    else:
        lo, hi = (c & 15).astype(np.int32), (c >> 4).astype(np.int32)
        q = (np.concatenate([lo, hi], axis=2) - 8).astype(np.float32)        # j < 16 low, j + 16 high
    return (d[:, :, None] * q).reshape(rows, cols)


@pytest.mark.parametrize("kind", ["Q8_0", "Q4_0"])
def test_repacked_layout_reconstructs_every_element(orc, kind):
    rows, cols = 130, 1024                    # 130: not a multiple of any tile
    w = synth.quant_weights(kind, rows, cols, 40 + oracle.KIND_ID[kind])
    rp = repack_np(kind, w, rows, cols)
    assert rp.size == w.size                  # the same bytes as the native tensor
    got = reconstruct(kind, rp, rows, cols)
    want = orc.dequant(kind, w, rows, cols)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_reconstruction_notices_a_misplaced_scale(orc):
    kind, rows, cols = "Q4_0", 8, 256
    w = synth.quant_weights(kind, rows, cols, 44)
    rp = repack_np(kind, w, rows, cols).reshape(-1, 144)
    rp[:, 128:] = np.roll(rp[:, 128:].reshape(-1, 8, 2), 1, axis=1).reshape(-1, 16)   # scales shifted one block
    got = reconstruct(kind, rp.reshape(-1), rows, cols)
    assert not np.array_equal(got, orc.dequant(kind, w, rows, cols))
