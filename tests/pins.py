"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each `check_*` takes an oracle build and returns a list of mismatch strings
(empty when the pin holds), so that the same pin can be run against the
sabotaged oracle builds to show that it fires.

Expected values are derived by hand from the pages' descriptions (cited per
check) -- not by re-typing the oracle's formulas. Blocks are hand-built with
scale 1.0 (f16 0x3C00) so the scale drops out of every product.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ONE = (0x00, 0x3C)          # f16 1.0, little-endian
BLOCK = {"Q8_0": 34, "Q4_0": 18, "Q5_0": 22, "Q4_K": 144, "Q5_K": 176, "Q6_K": 210,
         "Q2_K": 84, "Q3_K": 110, "IQ4_NL": 18, "IQ4_XS": 136, "MXFP4": 17,
         "Q4_1": 20, "Q5_1": 24, "Q8_1": 36}
ELEMS = {"Q8_0": 32, "Q4_0": 32, "Q5_0": 32, "Q4_K": 256, "Q5_K": 256, "Q6_K": 256,
         "Q2_K": 256, "Q3_K": 256, "IQ4_NL": 32, "IQ4_XS": 256, "MXFP4": 32,
         "Q4_1": 32, "Q5_1": 32, "Q8_1": 32}


def load_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def blk(kind):
    return np.zeros(BLOCK[kind], dtype=np.uint8)


def put16(b, off, v):
    b[off] = v & 0xFF
    b[off + 1] = (v >> 8) & 0xFF


def decode(orc, kind, b):
    return orc.dequant(kind, b, 1, ELEMS[kind])[0]


def f32bits(v):
    return int(np.float32(v).view(np.uint32))


def _diff(tag, got, want):
    bad = []
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    for i in range(want.size):
        g, w = got.flat[i], want.flat[i]
        if np.isnan(w) and np.isnan(g):
            continue
        if f32bits(g) != f32bits(w):
            bad.append(f"{tag}[{i}]: got {g!r} want {w!r}")
    return bad


# ---------------------------------------------------------------------------
# scalar decoders
# ---------------------------------------------------------------------------
def check_f16_exhaustive(orc):
    """All 65,536 binary16 patterns against numpy's float16 -> float32 (an
    independent route); NaN matches NaN (Vulkore quant_test.cpp, section 1)."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = pats.view(np.float16).astype(np.float32)
    got = np.array([orc.f16(int(h)) for h in range(65536)], dtype=np.float32)
    return _diff("f16", got, want)


def check_e8m0_exhaustive(orc):
    """Every E8M0 byte is 2^(e-127), computed another way (ferrox-cuda 0.20.0
    codebook.rs, every_e8m0_byte_is_two_to_the_e_minus_127)."""
    want = [np.ldexp(np.float32(1.0), e - 127) if e < 255 else np.float32(np.inf)
            for e in range(256)]
    with np.errstate(over="ignore"):
        want = np.array([np.float32(w) for w in want], dtype=np.float32)
    got = np.array([orc.e8m0(e) for e in range(256)], dtype=np.float32)
    return _diff("e8m0", got, want)


def check_scalar_golden(orc):
    bad = []
    for kind, inp, want in load_table("scalar_decoders.txt"):
        v = int(inp, 0)
        got = orc.f16(v) if kind == "f16" else orc.e8m0(v)
        if want == "nan":
            if not np.isnan(got):
                bad.append(f"{kind} {inp}: got {got}, want NaN")
        elif f32bits(got) != int(want, 16):
            bad.append(f"{kind} {inp}: got {f32bits(got):#010x}, want {want}")
    return bad


# ---------------------------------------------------------------------------
# codebooks by decode (ferrox-cuda 0.20.0 codebook.rs tests)
# ---------------------------------------------------------------------------
def check_iq4nl_codebook(orc):
    """d = 1.0 and byte j = code j in both nibbles: elements 0..15 and again
    16..31 must read the 16 table values in order."""
    table = [float(v) for _, v in load_table("iq4nl_codebook.txt")]
    b = blk("IQ4_NL")
    b[0], b[1] = ONE
    for j in range(16):
        b[2 + j] = j | (j << 4)
    got = decode(orc, "IQ4_NL", b)
    return _diff("iq4nl", got, table + table)


def check_e2m1_codebook(orc):
    """Scale byte 127 (= 2^0) and byte j = code j | code j << 4: decodes to the
    E2M1 table, compared by BITS so code 8 must be -0.0."""
    rows = load_table("e2m1_codebook.txt")
    bits = [int(r[2], 16) for r in rows]
    b = blk("MXFP4")
    b[0] = 127
    for j in range(16):
        b[1 + j] = j | (j << 4)
    got = decode(orc, "MXFP4", b)
    want = np.array(bits + bits, dtype=np.uint32).view(np.float32)
    bad = _diff("e2m1", got, want)
    # closed form of E2M1: sign s, exponent x, mantissa m
    for c in range(16):
        s, x, m = c >> 3, (c >> 1) & 3, c & 1
        mag = m / 2 if x == 0 else 2.0 ** (x - 1) * (1 + m / 2)
        cf = np.float32(-mag if s else mag)
        if f32bits(cf) != bits[c]:
            bad.append(f"e2m1 closed form code {c}: {cf} vs golden {bits[c]:#x}")
    return bad


def check_mxfp4_scale(orc):
    """E8M0 multiplies the code value: 128 doubles it, 0 gives 2^-127 times it
    (an exact fp32 subnormal)."""
    rows = load_table("e2m1_codebook.txt")
    vals = np.array([int(r[2], 16) for r in rows], dtype=np.uint32).view(np.float32)
    bad = []
    for e, f in ((128, np.float32(2.0)), (0, np.float32(2.0) ** np.float32(-127)),
                 (130, np.float32(8.0))):
        b = blk("MXFP4")
        b[0] = e
        for j in range(16):
            b[1 + j] = j | (j << 4)
        got = decode(orc, "MXFP4", b)
        want = np.concatenate([vals, vals]) * f
        bad += _diff(f"mxfp4 e={e}", got, want)
    return bad


# ---------------------------------------------------------------------------
# legacy 32-element formats
# ---------------------------------------------------------------------------
def check_q4_0_nibbles(orc):
    """Byte j = (j) | (15 - j) << 4 with d = 1: element j = j - 8 and element
    j + 16 = (15 - j) - 8 = 7 - j (BASELINE tiny Q4_0 workload; ferrox-cuda
    codebook.rs IQ4_NL doc: Q4_0's packing, -8 bias)."""
    b = blk("Q4_0")
    b[0], b[1] = ONE
    for j in range(16):
        b[2 + j] = j | ((15 - j) << 4)
    want = [j - 8 for j in range(16)] + [7 - j for j in range(16)]
    return _diff("q4_0", decode(orc, "Q4_0", b), want)


def check_q8_0(orc):
    """d = 1 and the 32 code bytes 0x00, 0x7F, 0x80, 0xFF, ...: int8 codes are
    two's complement (Vulkore quant_test.cpp, ref::q8_0)."""
    b = blk("Q8_0")
    b[0], b[1] = ONE
    codes = [0x00, 0x7F, 0x80, 0xFF, 0x01, 0x81, 0x40, 0xC0] * 4
    b[2:34] = codes
    want = [0, 127, -128, -1, 1, -127, 64, -64] * 4
    bad = _diff("q8_0", decode(orc, "Q8_0", b), want)
    # d = 2^-24 (smallest f16 subnormal) times 127 is exact in fp32
    put16(b, 0, 0x0001)
    want2 = [np.float32(w) * np.float32(2.0 ** -24) for w in want]
    return bad + _diff("q8_0 subnormal d", decode(orc, "Q8_0", b), want2)


def check_q5_0_qh(orc):
    """The fifth bit of element e is bit e of qh (Vulkore quant_test.cpp,
    ref::q5_0 comment). With zero nibbles every element is -16; setting one qh
    bit lifts exactly that element to 0."""
    bad = []
    for e0 in (0, 5, 15, 16, 20, 31):
        b = blk("Q5_0")
        b[0], b[1] = ONE
        qh = 1 << e0
        b[2:6] = [qh & 0xFF, (qh >> 8) & 0xFF, (qh >> 16) & 0xFF, (qh >> 24) & 0xFF]
        want = [-16.0] * 32
        want[e0] = 0.0
        bad += _diff(f"q5_0 qh bit {e0}", decode(orc, "Q5_0", b), want)
    # nibble order as Q4_0: byte 3 = 0xA7 -> element 3 = 7-16, element 19 = 10-16
    b = blk("Q5_0")
    b[0], b[1] = ONE
    b[6 + 3] = 0xA7
    want = [-16.0] * 32
    want[3], want[19] = -9.0, -6.0
    return bad + _diff("q5_0 nibbles", decode(orc, "Q5_0", b), want)


# ---------------------------------------------------------------------------
# the kinds with no mul_mm kernel on the pages (GGUF reading): Q4_1, Q5_1, Q8_1
# ---------------------------------------------------------------------------
F16_MINUS_8 = 0xC800       # -8.0
F16_MINUS_16 = 0xCC00      # -16.0
F16_60000 = 0x7B53         # 60000.0
F16_TINY = 0x0401          # 2^-14 * (1 + 2^-10), the smallest normal f16 plus one ulp


def check_q4_1(orc):
    """Q4_1 = Q4_0's nibble packing with unsigned codes plus an f16 min after
    d: with d = 1, m = 0 and byte j = j | (15 - j) << 4, element j is j and
    element j + 16 is 15 - j. With m = -8 (d = 1) every element is Q4_0's
    value of the same code bytes, j - 8 and 7 - j. With d = 0 every element
    is m. d*q + m rounds once: d = 2^-14 (1 + 2^-10), q = 15, m = 60000 gives
    60000 exactly (the product is far below half an fp32 ulp of 60000)."""
    bad = []
    b = blk("Q4_1")
    b[0], b[1] = ONE
    for j in range(16):
        b[4 + j] = j | ((15 - j) << 4)
    bad += _diff("q4_1 codes", decode(orc, "Q4_1", b), [j for j in range(16)] + [15 - j for j in range(16)])
    put16(b, 2, F16_MINUS_8)
    bad += _diff("q4_1 m = -8", decode(orc, "Q4_1", b), [j - 8 for j in range(16)] + [7 - j for j in range(16)])
    b0 = blk("Q4_1")
    put16(b0, 2, 0x3E00)   # m = 1.5, d = 0
    b0[4:20] = 0xFF
    bad += _diff("q4_1 d = 0", decode(orc, "Q4_1", b0), [1.5] * 32)
    b1 = blk("Q4_1")
    put16(b1, 0, F16_TINY)
    put16(b1, 2, F16_60000)
    b1[4:20] = 0xFF
    bad += _diff("q4_1 rounds once", decode(orc, "Q4_1", b1), [60000.0] * 32)
    return bad


def check_q5_1(orc):
    """Q5_1 = Q5_0's bit layout after an f16 min, unsigned codes: with d = 1,
    m = 0 and zero nibbles every element is 0 except the one whose qh bit is
    set, which is 16; with m = -16 it reduces to Q5_0 (-16 everywhere, 0
    where the bit is set); the nibble order is Q4_0's."""
    bad = []
    for e0 in (0, 7, 15, 16, 23, 31):
        b = blk("Q5_1")
        b[0], b[1] = ONE
        qh = 1 << e0
        b[4:8] = [qh & 0xFF, (qh >> 8) & 0xFF, (qh >> 16) & 0xFF, (qh >> 24) & 0xFF]
        want = [0.0] * 32
        want[e0] = 16.0
        bad += _diff(f"q5_1 qh bit {e0}", decode(orc, "Q5_1", b), want)
        put16(b, 2, F16_MINUS_16)
        want = [-16.0] * 32
        want[e0] = 0.0
        bad += _diff(f"q5_1 qh bit {e0}, m = -16", decode(orc, "Q5_1", b), want)
    b = blk("Q5_1")
    b[0], b[1] = ONE
    b[8 + 3] = 0xA7
    want = [0.0] * 32
    want[3], want[19] = 7.0, 10.0
    return bad + _diff("q5_1 nibbles", decode(orc, "Q5_1", b), want)


def check_q8_1(orc):
    """Q8_1 = Q8_0's int8 codes after an extra f16 field (d times the code sum),
    which no element reads: the codes of check_q8_0 at byte 4 give the same
    values whatever the field holds (0, a NaN, an infinity)."""
    bad = []
    codes = [0x00, 0x7F, 0x80, 0xFF, 0x01, 0x81, 0x40, 0xC0] * 4
    want = [0, 127, -128, -1, 1, -127, 64, -64] * 4
    for sfield in (0x0000, 0x7E00, 0x7C00, 0x3C00):
        b = blk("Q8_1")
        b[0], b[1] = ONE
        put16(b, 2, sfield)
        b[4:36] = codes
        bad += _diff(f"q8_1 s = {sfield:#06x}", decode(orc, "Q8_1", b), want)
    return bad


def check_legacy_min_formats_reduce(orc):
    """Cross-format invariants on random blocks: Q4_1 with m = -8 d is Q4_0,
    Q5_1 with m = -16 d is Q5_0, Q8_1 is Q8_0 (same d and code bytes). d is a
    power of two so that -8 d and -16 d are exact f16 values."""
    bad = []
    rng = np.random.default_rng(7)
    for _ in range(64):
        e = int(rng.integers(-10, 4))
        d_bits = (15 + e) << 10                      # 2^e
        codes = rng.integers(0, 256, 32, dtype=np.uint8)
        qh = rng.integers(0, 256, 4, dtype=np.uint8)
        q40 = blk("Q4_0"); put16(q40, 0, d_bits); q40[2:18] = codes[:16]
        q41 = blk("Q4_1"); put16(q41, 0, d_bits); put16(q41, 2, 0x8000 | ((18 + e) << 10)); q41[4:20] = codes[:16]
        bad += _diff("q4_1 vs q4_0", decode(orc, "Q4_1", q41), decode(orc, "Q4_0", q40))
        q50 = blk("Q5_0"); put16(q50, 0, d_bits); q50[2:6] = qh; q50[6:22] = codes[:16]
        q51 = blk("Q5_1"); put16(q51, 0, d_bits); put16(q51, 2, 0x8000 | ((19 + e) << 10))
        q51[4:8] = qh; q51[8:24] = codes[:16]
        bad += _diff("q5_1 vs q5_0", decode(orc, "Q5_1", q51), decode(orc, "Q5_0", q50))
        q80 = blk("Q8_0"); put16(q80, 0, d_bits); q80[2:34] = codes
        q81 = blk("Q8_1"); put16(q81, 0, d_bits); q81[2:4] = rng.integers(0, 256, 2, dtype=np.uint8)
        q81[4:36] = codes
        bad += _diff("q8_1 vs q8_0", decode(orc, "Q8_1", q81), decode(orc, "Q8_0", q80))
    return bad


# ---------------------------------------------------------------------------
# K-quants
# ---------------------------------------------------------------------------
def pack_k4_scales(sc, mn):
    """Encoder for the Q4_K/Q5_K 12-byte 6-bit (scale, min) field, written as the
    inverse of the unpack in Vulkore quant_test.cpp `q4k_scale_min`: sub-blocks
    0..3 keep 6 bits in bytes 0..3 (scale) and 4..7 (min); sub-blocks 4..7 keep
    their low 4 bits in the nibbles of bytes 8..11 and their top 2 bits in the
    top 2 bits of bytes 0..7."""
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return s


def check_q4_k(orc):
    bad = []
    # 1. nibble order: chunk c's 32 bytes give elements 64c..64c+31 (low) then
    #    64c+32..64c+63 (high). All sc = 1, mins 0 (Vulkore ref::q4_k).
    b = blk("Q4_K")
    b[0], b[1] = ONE
    b[4:16] = pack_k4_scales([1] * 8, [0] * 8)
    for i in range(128):
        b[16 + i] = (i % 16) | ((15 - i % 16) << 4)
    want = []
    for c in range(4):
        want += [i % 16 for i in range(32)] + [15 - i % 16 for i in range(32)]
    bad += _diff("q4_k nibbles", decode(orc, "Q4_K", b), want)
    # 2. distinct 6-bit scales and mins per sub-block, round trip through the packer
    sc = [1, 2, 3, 63, 33, 17, 48, 5]
    mn = [0, 7, 63, 1, 40, 2, 31, 60]
    b = blk("Q4_K")
    b[0], b[1] = ONE
    b[2], b[3] = ONE                       # dmin = 1
    b[4:16] = pack_k4_scales(sc, mn)
    for i in range(128):
        b[16 + i] = 0x93                   # low nibble 3, high nibble 9
    want = []
    for c in range(4):
        want += [sc[2 * c] * 3 - mn[2 * c]] * 32 + [sc[2 * c + 1] * 9 - mn[2 * c + 1]] * 32
    bad += _diff("q4_k scales/mins", decode(orc, "Q4_K", b), want)
    return bad


def check_q5_k(orc):
    bad = []
    sc = [4, 9, 1, 62, 35, 2, 11, 40]
    mn = [3, 0, 5, 9, 63, 32, 1, 7]
    head = pack_k4_scales(sc, mn)
    # 1. with qh = 0 a Q5_K block equals the Q4_K block with the same head and codes
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 256, 128, dtype=np.uint8)
    a = blk("Q5_K")
    a[0], a[1] = ONE
    put16(a, 2, 0x3800)                    # dmin = 0.5
    a[4:16] = head
    a[48:176] = codes
    q4 = blk("Q4_K")
    q4[0:16] = a[0:16]
    q4[16:144] = codes
    bad += _diff("q5_k(qh=0) vs q4_k", decode(orc, "Q5_K", a), decode(orc, "Q4_K", q4))
    # 2. one qh bit: qh[l] bit t is the fifth bit of element 32t + l
    for l, t in ((7, 2), (0, 0), (31, 7), (12, 5)):
        b = a.copy()
        b[16 + l] = 1 << t
        want = decode(orc, "Q4_K", q4).copy()
        e = 32 * t + l
        want[e] = np.float32(np.float32(sc[t] * (int(want_code(codes, e)) + 16))
                             - np.float32(0.5 * mn[t]))
        bad += _diff(f"q5_k qh[{l}] bit {t}", decode(orc, "Q5_K", b), want)
    return bad


def want_code(codes, e):
    """4-bit code of element e in the Q4_K/Q5_K nibble layout (64-element chunks:
    low nibbles of the chunk's 32 bytes, then the high nibbles)."""
    byte = codes[(e // 64) * 32 + e % 32]
    return (byte >> 4) if (e % 64) >= 32 else (byte & 15)


def check_q6_k(orc):
    """Hand-placed bits (Vulkore quant_test.cpp ref::q6_k: ql 128 B, qh 64 B, 16
    int8 scales, f16 d at 208; each 128-element half is four interleaved
    32-element quarters). All codes zero decode to -32."""
    def base():
        b = blk("Q6_K")
        put16(b, 208, 0x3C00)
        b[192:208] = 1
        return b
    cases = [
        # (byte index, value, {element: value})
        (0, 0x05, {0: -27}),            # ql[0] low nibble -> element 0
        (0, 0x50, {64: -27}),           # ql[0] high nibble -> quarter 2 of half 0
        (32, 0x03, {32: -29}),          # ql[32] low -> quarter 1
        (32, 0x30, {96: -29}),          # ql[32] high -> quarter 3
        (64 + 7, 0x01, {135: -31}),     # ql of half 1, lane 7
        (128 + 0, 0x04, {32: -16}),     # qh[0] bits 2..3 = 1 -> quarter 1, +16
        (128 + 32 + 5, 0xC0, {229: 16}),  # qh of half 1, lane 5, bits 6..7 = 3 -> +48
        (128 + 9, 0x03, {9: 16}),       # qh[9] bits 0..1 = 3 -> element 9, +48
    ]
    bad = []
    for idx, val, changed in cases:
        b = base()
        b[idx] = val
        want = np.full(256, -32.0, dtype=np.float32)
        for e, v in changed.items():
            want[e] = v
        bad += _diff(f"q6_k byte {idx}={val:#x}", decode(orc, "Q6_K", b), want)
    # one scale: int8 scale j covers elements 16j..16j+15; 0xFE is -2
    b = base()
    b[192 + 3] = 0xFE
    want = np.full(256, -32.0, dtype=np.float32)
    want[48:64] = 64.0
    bad += _diff("q6_k scale 3", decode(orc, "Q6_K", b), want)
    b = base()
    b[192 + 13] = 0x80                    # -128
    want = np.full(256, -32.0, dtype=np.float32)
    want[208:224] = 4096.0
    bad += _diff("q6_k scale 13", decode(orc, "Q6_K", b), want)
    return bad


def check_q2_k(orc):
    """GGUF reading (layout not on the pages): scales[16] at 0 (low nibble scale,
    high nibble min), qs[64] at 16, f16 d at 80, f16 dmin at 82."""
    def base():
        b = blk("Q2_K")
        put16(b, 80, 0x3C00)
        put16(b, 82, 0x3C00)
        b[0:16] = 0x01
        return b
    bad = []
    for idx, val, changed in ((16, 0x03, {0: 3}), (16, 0x0C, {32: 3}),
                              (16 + 32 + 1, 0xC0, {225: 3}), (16 + 17, 0x20, {81: 2})):
        b = base()
        b[idx] = val
        want = np.zeros(256, dtype=np.float32)
        for e, v in changed.items():
            want[e] = v
        bad += _diff(f"q2_k byte {idx}={val:#x}", decode(orc, "Q2_K", b), want)
    b = base()
    b[16:80] = 0xFF                        # every code 3
    b[5] = 0x52                            # sub-block 5: scale 2, min 5
    want = np.full(256, 3.0, dtype=np.float32)
    want[80:96] = 2 * 3 - 5
    bad += _diff("q2_k scale/min 5", decode(orc, "Q2_K", b), want)
    return bad


def pack_q3k_scales(sc):
    """Encoder for the Q3_K 12-byte field of sixteen 6-bit scales (GGUF reading):
    low 4 bits of scale j in the low nibble of byte j (j < 8) or the high nibble
    of byte j-8; top 2 bits in byte 8 + j%4 at bit 2*(j//4)."""
    s = [0] * 12
    for j in range(16):
        if j < 8:
            s[j] |= sc[j] & 15
        else:
            s[j - 8] |= (sc[j] & 15) << 4
        s[8 + j % 4] |= ((sc[j] >> 4) & 3) << (2 * (j // 4))
    return s


def check_q3_k(orc):
    """GGUF reading: hmask[32] at 0, qs[64] at 32, scales[12] at 96, f16 d at 108;
    a CLEAR hmask bit subtracts 4 (ferrox-cuda mul_mm.rs names an hmask bias)."""
    def base(hm=0xFF, qs=0x00, sc=None):
        b = blk("Q3_K")
        b[0:32] = hm
        b[32:96] = qs
        b[96:108] = pack_q3k_scales(sc or [33] * 16)   # every scale 33 - 32 = 1
        put16(b, 108, 0x3C00)
        return b
    bad = []
    bad += _diff("q3_k all set", decode(orc, "Q3_K", base()), np.zeros(256))
    bad += _diff("q3_k all clear", decode(orc, "Q3_K", base(hm=0x00)), np.full(256, -4.0))
    b = base()
    b[3] = 0xDF                            # hmask[3] bit 5 clear -> element 5*32+3
    want = np.zeros(256)
    want[163] = -4
    bad += _diff("q3_k hmask one bit", decode(orc, "Q3_K", b), want)
    b = base()
    b[32 + 0] = 0x02                       # qs[0] bits 0..1 = 2 -> element 0
    want = np.zeros(256)
    want[0] = 2
    bad += _diff("q3_k qs[0]", decode(orc, "Q3_K", b), want)
    sc = [33] * 16
    sc[9] = 35
    sc[14] = 0                             # 0 - 32 = -32
    want = np.ones(256)
    want[144:160] = 3
    want[224:240] = -32
    bad += _diff("q3_k scales", decode(orc, "Q3_K", base(qs=0x55, sc=sc)), want)
    # round trip of all 64 scale values
    sc = [(7 * j + 3) % 64 for j in range(16)]
    want = np.repeat(np.array(sc, dtype=np.float32) - 32, 16)
    bad += _diff("q3_k scale round trip", decode(orc, "Q3_K", base(qs=0x55, sc=sc)), want)
    return bad


def pack_iq4xs_scales(ls):
    """Encoder for IQ4_XS group scales (ferrox-cuda 0.20.0 codebook.rs, IQ4_XS
    doc): low 4 bits in nibble (ib & 1) of scales_l[ib / 2], top 2 bits in bits
    2ib..2ib+1 of scales_h."""
    sh = 0
    sl = [0] * 4
    for ib in range(8):
        sl[ib // 2] |= (ls[ib] & 15) << (4 * (ib & 1))
        sh |= ((ls[ib] >> 4) & 3) << (2 * ib)
    return sh, sl


def check_iq4_xs(orc):
    table = np.array([float(v) for _, v in load_table("iq4nl_codebook.txt")], dtype=np.float32)
    bad = []
    for ls in ([33] * 8, [33, 34, 33, 1, 63, 32, 49, 20]):
        b = blk("IQ4_XS")
        b[0], b[1] = ONE
        sh, sl = pack_iq4xs_scales(ls)
        put16(b, 2, sh)
        b[4:8] = sl
        for ib in range(8):
            for j in range(16):
                b[8 + 16 * ib + j] = j | (j << 4)
        want = np.concatenate([np.concatenate([table, table]) * (l - 32) for l in ls])
        bad += _diff(f"iq4_xs ls={ls}", decode(orc, "IQ4_XS", b), want)
    # group g equals an IQ4_NL block whose scale is d * (ls - 32)
    rng = np.random.default_rng(12345)
    b = rng.integers(0, 256, 136, dtype=np.uint8)
    put16(b, 0, 0x3000)                     # d = 0.125: d * (ls - 32) stays an exact f16
    got = decode(orc, "IQ4_XS", b)
    d = 0.125
    sh = int(b[2]) | (int(b[3]) << 8)
    for ib in range(8):
        ls = ((b[4 + ib // 2] >> (4 * (ib & 1))) & 15) | (((sh >> (2 * ib)) & 3) << 4)
        nl = blk("IQ4_NL")
        dd = np.float16(d * (int(ls) - 32))
        if float(dd) != d * (int(ls) - 32):
            continue                        # not representable as an f16 scale
        put16(nl, 0, int(np.array(dd, dtype=np.float16).view(np.uint16)))
        nl[2:18] = b[8 + 16 * ib: 24 + 16 * ib]
        bad += _diff(f"iq4_xs group {ib} vs iq4_nl", got[32 * ib:32 * ib + 32],
                     decode(orc, "IQ4_NL", nl))
    return bad


# ---------------------------------------------------------------------------
# products
# ---------------------------------------------------------------------------
def check_gemm_brute_force(orc):
    """1-block inputs: the fp64 product is the hand-expanded sum over the block's
    elements; the N x M output layout is token-major (ferrox-cuda mul_mm.rs:
    dst[token * n_rows + row])."""
    bad = []
    rng = np.random.default_rng(1)
    for kind in BLOCK:
        K = ELEMS[kind]
        M, N = 3, 2
        w = rng.integers(0, 256, M * BLOCK[kind], dtype=np.uint8)
        for r in range(M):                 # keep f16 scale fields finite and small
            o = r * BLOCK[kind]
            for off in {"Q6_K": (208,), "Q2_K": (80, 82), "Q3_K": (108,),
                        "MXFP4": ()}.get(kind, (0, 2) if kind in ("Q4_K", "Q5_K", "Q4_1", "Q5_1") else (0,)):
                put16(w, o + off, 0x2000 + int(rng.integers(0, 0x400)))
            if kind == "MXFP4":
                w[o] = 120 + int(rng.integers(0, 8))
        x = rng.standard_normal((N, K)).astype(np.float32)
        deq = orc.dequant(kind, w, M, K)
        y, tol = orc.gemm(kind, w, M, K, x, N)
        for n in range(N):
            for m in range(M):
                acc = 0.0
                mag = 0.0
                for k in range(K):
                    p = float(deq[m, k]) * float(x[n, k])
                    acc += p
                    mag += abs(p)
                if abs(y[n, m] - acc) > 1e-12 * max(1.0, mag):
                    bad.append(f"{kind} y[{n},{m}] = {y[n, m]} vs hand sum {acc}")
                if abs(tol[n, m] - (1e-3 * mag + 1e-6)) > 1e-12 * max(1.0, mag):
                    bad.append(f"{kind} tol[{n},{m}] = {tol[n, m]} vs {1e-3 * mag + 1e-6}")
    return bad
