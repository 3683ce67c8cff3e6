"""Exactness of the element formulas (CPU only).

Every element of every format is a product of an fp32 block scale, an integer
sub-scale and an integer code (or a codebook value), minus, for the affine-min
formats (Q4_K, Q5_K, Q2_K), a second product of a scale and an integer min
(Q4_1 and Q5_1 add an f16 min instead).
The significant bits of each product stay within fp32's 24, so the product is
exact and its association order does not matter; the affine formats round
once, at the subtraction, which an FMA also does. This is what makes a
bit-exact dequant possible on any evaluation order, and what lets the kernels
multiply block scales into partial sums instead of operands.

The check: factors are extracted here, in numpy, straight from the block bytes
(the byte layouts of the Vulkore `ref::` CPU references for Q8_0, Q5_0, Q4_K
and Q6_K, the ferrox-cuda codebook.rs page for IQ4_NL, IQ4_XS and MXFP4, the
GGUF reading for Q5_K, Q2_K, Q3_K, Q4_1, Q5_1 and Q8_1); for every element, (a * b) * c,
a * (b * c) and the exact product (fp64, where it is exact) must agree
bitwise, the FMA-contracted affine form must equal the subtract form, and the
result must equal the oracle's dequant bit for bit.
"""
import numpy as np
import pytest

import oracle
from gemv_mul_mm_gb300 import synth

KV_IQ4 = np.array([-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113], np.float32)
KV_E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], np.float32)


def _f16(b, off):
    return b[:, off:off + 2].copy().view(np.float16)[:, 0].astype(np.float32)


def _nib(codes, e):
    """Element e of a 32-element nibble run: low nibble of byte e (e < 16),
    high nibble of byte e - 16."""
    byte = codes[:, e % 16].astype(np.int64)
    return (byte & 15) if e < 16 else (byte >> 4)


def _k4_scale_min(s, j):
    s = s.astype(np.int64)
    if j < 4:
        return s[:, j] & 63, s[:, j + 4] & 63
    return ((s[:, j + 4] & 15) | ((s[:, j - 4] >> 6) << 4),
            (s[:, j + 4] >> 4) | ((s[:, j] >> 6) << 4))


def factors(kind, b):
    """Per block row of `b` (n_blocks x block_bytes) and per element e:
    (a, sub, q, dmin, mn) with value = (a * sub) * q - dmin * mn, all fp32
    arrays of shape (n_blocks, elems); dmin = mn = 0 where there is no min."""
    nb = b.shape[0]
    be = synth.block_geometry(kind)[1]
    a = np.zeros((nb, be), np.float32)
    sub = np.ones((nb, be), np.float32)
    q = np.zeros((nb, be), np.float32)
    dmin = np.zeros((nb, be), np.float32)
    mn = np.zeros((nb, be), np.float32)
    bi = b.astype(np.int64)
    for e in range(be):
        if kind == "Q8_0":
            a[:, e] = _f16(b, 0)
            q[:, e] = b[:, 2 + e].view(np.int8)
        elif kind == "Q4_0":
            a[:, e] = _f16(b, 0)
            q[:, e] = _nib(b[:, 2:18], e) - 8
        elif kind == "IQ4_NL":
            a[:, e] = _f16(b, 0)
            q[:, e] = KV_IQ4[_nib(b[:, 2:18], e)]
        elif kind == "MXFP4":
            eb = bi[:, 0]
            a[:, e] = np.where(eb == 0, np.float32(2.0 ** -127),
                               np.ldexp(np.float32(1), (eb - 127).astype(np.int32)).astype(np.float32))
            q[:, e] = KV_E2M1[_nib(b[:, 1:17], e)]
        elif kind == "Q5_0":
            qh = bi[:, 2] | (bi[:, 3] << 8) | (bi[:, 4] << 16) | (bi[:, 5] << 24)
            a[:, e] = _f16(b, 0)
            q[:, e] = (_nib(b[:, 6:22], e) | (((qh >> e) & 1) << 4)) - 16
        elif kind in ("Q4_K", "Q5_K"):
            j = e // 32
            sc, m = _k4_scale_min(b[:, 4:16], j)
            qs = 16 if kind == "Q4_K" else 48
            byte = bi[:, qs + (e // 64) * 32 + e % 32]
            nib = (byte & 15) if (e % 64) < 32 else (byte >> 4)
            if kind == "Q5_K":
                nib = nib + 16 * ((bi[:, 16 + e % 32] >> (e // 32)) & 1)
            a[:, e], sub[:, e], q[:, e] = _f16(b, 0), sc, nib
            dmin[:, e], mn[:, e] = _f16(b, 2), m
        elif kind == "Q6_K":
            h, w = e // 128, e % 128
            l, g = w % 32, w // 32
            byte = bi[:, h * 64 + l + (g & 1) * 32]
            lo = (byte & 15) if g < 2 else (byte >> 4)
            hi = (bi[:, 128 + h * 32 + l] >> (2 * g)) & 3
            a[:, e] = _f16(b, 208)
            sub[:, e] = b[:, 192 + e // 16].view(np.int8)
            q[:, e] = (lo | (hi << 4)) - 32
        elif kind == "Q2_K":
            h, w = e // 128, e % 128
            l, g = w % 32, w // 32
            s = bi[:, e // 16]
            a[:, e], sub[:, e] = _f16(b, 80), s & 15
            q[:, e] = (bi[:, 16 + h * 32 + l] >> (2 * g)) & 3
            dmin[:, e], mn[:, e] = _f16(b, 82), s >> 4
        elif kind == "Q3_K":
            h, w = e // 128, e % 128
            l, g = w % 32, w // 32
            q2 = (bi[:, 32 + h * 32 + l] >> (2 * g)) & 3
            hb = (bi[:, e % 32] >> (e // 32)) & 1
            j = e // 16
            lo = (bi[:, 96 + j] & 15) if j < 8 else (bi[:, 96 + j - 8] >> 4)
            hi = (bi[:, 96 + 8 + j % 4] >> (2 * (j // 4))) & 3
            a[:, e], sub[:, e] = _f16(b, 108), (lo | (hi << 4)) - 32
            q[:, e] = q2 - np.where(hb == 1, 0, 4)
        elif kind == "IQ4_XS":
            ib, f = e // 32, e % 32
            byte = bi[:, 8 + 16 * ib + f % 16]
            c = (byte & 15) if f < 16 else (byte >> 4)
            sh = bi[:, 2] | (bi[:, 3] << 8)
            ls = ((bi[:, 4 + ib // 2] >> (4 * (ib & 1))) & 15) | (((sh >> (2 * ib)) & 3) << 4)
            a[:, e], sub[:, e], q[:, e] = _f16(b, 0), ls - 32, KV_IQ4[c]
        elif kind == "Q8_1":
            a[:, e] = _f16(b, 0)
            q[:, e] = b[:, 4 + e].view(np.int8)
        elif kind == "Q4_1":
            # w = d * q + m: the min enters as dmin = -m times mn = 1
            a[:, e], q[:, e] = _f16(b, 0), _nib(b[:, 4:20], e)
            dmin[:, e], mn[:, e] = -_f16(b, 2), 1.0
        elif kind == "Q5_1":
            qh = bi[:, 4] | (bi[:, 5] << 8) | (bi[:, 6] << 16) | (bi[:, 7] << 24)
            a[:, e], q[:, e] = _f16(b, 0), _nib(b[:, 8:24], e) | (((qh >> e) & 1) << 4)
            dmin[:, e], mn[:, e] = -_f16(b, 2), 1.0
        else:
            raise ValueError(kind)
    return a, sub, q, dmin, mn


def blocks_for(kind, n_rows, seed):
    K = synth.block_geometry(kind)[1] * 8
    w = synth.quant_weights(kind, n_rows, K, seed)
    bb = synth.block_geometry(kind)[0]
    return w, w.reshape(-1, bb), K


@pytest.mark.parametrize("kind", oracle.KINDS)
def test_products_exact_in_any_order(orc, kind):
    w, b, K = blocks_for(kind, 48, 700 + oracle.KIND_ID[kind])
    a, sub, q, dmin, mn = factors(kind, b)
    with np.errstate(over="ignore", invalid="ignore"):
        p1 = (a * sub) * q                      # (d * sc) * q
        p2 = a * (sub * q)                      # d * (sc * q)
        exact = a.astype(np.float64) * sub.astype(np.float64) * q.astype(np.float64)
        t2 = dmin * mn
        t2_exact = dmin.astype(np.float64) * mn.astype(np.float64)
    fin = np.isfinite(exact)
    assert fin.mean() > 0.99
    # every product is exact: both orders give the fp64 product bit for bit
    assert np.array_equal(p1[fin].astype(np.float64), exact[fin])
    assert np.array_equal(p2.view(np.uint32)[fin], p1.view(np.uint32)[fin])
    assert np.array_equal(t2.astype(np.float64), t2_exact)
    # affine form: subtract of two exact products == the FMA-contracted form,
    # i.e. one rounding of the exact difference (exact in fp64 here: the
    # workload scales span a few decades, far inside fp64's 53 bits)
    sub_form = (p1 - t2).astype(np.float32)
    fma_form = (exact - t2_exact).astype(np.float32)
    assert np.array_equal(sub_form.view(np.uint32)[fin], fma_form.view(np.uint32)[fin])
    # and the oracle's dequant is exactly that value
    deq = orc.dequant(kind, w, 48, K).reshape(-1, synth.block_geometry(kind)[1])
    assert np.array_equal(deq.view(np.uint32)[fin], sub_form.view(np.uint32)[fin])


@pytest.mark.parametrize("kind", ["Q6_K", "IQ4_XS", "Q5_K", "Q4_K"])
def test_products_exact_at_extreme_codes(orc, kind):
    """The widest products: every code and sub-scale at its extreme magnitude
    (Q6_K sc = -128 with q - 32 = -32; IQ4_XS ls - 32 = -32 with KV = -127;
    Q4_K / Q5_K sc = m = 63 with q = 15 / 31), scales with all 11 significant
    bits set."""
    bb, be = synth.block_geometry(kind)
    b = np.zeros((4, bb), np.uint8)
    dbits = np.array([0x3BFF, 0x1BFF, 0x07FF, 0x5BFF], np.uint16)   # 11-bit significands, wide exponents
    for r in range(4):
        d = np.frombuffer(dbits[r].tobytes(), np.uint8)
        if kind == "Q6_K":
            b[r, 0:128] = 0x00              # low nibbles 0, high bits 0 -> q = -32
            b[r, 192:208] = 0x80            # sc = -128
            b[r, 208:210] = d
        elif kind == "IQ4_XS":
            b[r, 0:2] = d
            b[r, 2:4] = 0x00                # scales_h 0 ...
            b[r, 4:8] = 0x00                # ... and scales_l 0 -> ls - 32 = -32
            b[r, 8:136] = 0x00              # codes 0 -> KV = -127
        else:
            b[r, 0:2] = d
            b[r, 2:4] = d
            b[r, 4:16] = 0xFF               # sc = m = 63 for all eight sub-blocks
            b[r, 16:bb] = 0xFF              # q = 15 (Q4_K) / qh all set, q = 31 (Q5_K)
    a, sub, q, dmin, mn = factors(kind, b)
    exact = a.astype(np.float64) * sub.astype(np.float64) * q.astype(np.float64)
    assert np.array_equal(((a * sub) * q).astype(np.float64), exact)
    assert np.array_equal((a * (sub * q)).astype(np.float64), exact)
    want = (exact - dmin.astype(np.float64) * mn.astype(np.float64)).astype(np.float32)
    deq = orc.dequant(kind, b.reshape(-1), 4, be)
    assert np.array_equal(deq.view(np.uint32), want.view(np.uint32))


def test_mxfp4_operand_fold_range():
    """The tensor-core GEMM folds each MXFP4 block's exponent into its f16
    operands relative to the largest exponent e_max of the 256-element
    super-step: operand = E2M1 value * 2^-(e_max - e), rounded once to f16.
    An E2M1 value is m * 2^-1 with m <= 12, so the operand is exact while the
    spread e_max - e is at most 23 (f16 subnormals are the multiples of
    2^-24); at 24 the odd halves (+-0.5, +-1.5) round to even; past 24 the
    kernel zeroes the scale and the block contributes nothing. The scale words
    themselves are f16 powers of two down to 2^-24 (normal through 2^-14,
    subnormal below)."""
    for d in range(0, 24):
        exact = KV_E2M1.astype(np.float64) * 2.0 ** -d
        assert np.array_equal(exact.astype(np.float16).astype(np.float64), exact), d
    at24 = KV_E2M1.astype(np.float64) * 2.0 ** -24
    r = at24.astype(np.float16).astype(np.float64)
    odd_half = np.isin(np.abs(KV_E2M1), [0.5, 1.5])
    assert np.array_equal(r[~odd_half], at24[~odd_half])
    assert np.array_equal(np.abs(r[odd_half]), np.where(np.abs(KV_E2M1[odd_half]) == 0.5, 0.0, 2.0 ** -23))
    # the scale word for a spread k: f16 bits (15 - k) << 10 (normal) or
    # 1 << (24 - k) (subnormal), 2^-k either way
    for k in range(0, 25):
        bits = ((15 - k) << 10) if k <= 14 else (1 << (24 - k))
        assert np.array([bits], np.uint16).view(np.float16)[0] == np.float16(2.0 ** -k), k
