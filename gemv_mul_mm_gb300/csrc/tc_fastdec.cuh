// tc_fastdec.cuh -- register-level decoders that turn one 64-element sub-step
// of a quantized row (raw block bytes in shared memory) into the f16 operand
// codes of the tensor-core GEMM.
//
// The codes are those of the table in decode.cuh (integer code times integer
// sub-scale, or the codebook value); the fp32 block / super-block scales are
// applied to the partial sums in the epilogue, not here.
//
// Output: o[e / 2] holds elements e and e + 1 of the sub-step (e even) as an
// f16x2 word, low half = element e. The K-quants and IQ4_XS (FastDecPre) split the work:
// pre() turns the super-block's integer sub-scales into f16 words once,
// sub_pre() decodes a sub-step with them; the other formats decode a sub-step
// with sub(). The GEMM stores o[4c .. 4c + 3] as the
// 16-byte chunk c (elements 8c .. 8c + 7) of the row's K-major operand row.
//
// Techniques (no per-element conversions, no table loads from memory):
//   * f16 "magic number": OR-ing a small unsigned field v into the mantissa of
//     1024.0h (bits 0x6400) gives the f16 value 1024 + v exactly (the f16 ulp
//     is 1 in [1024, 2048)); a field at bits 4..7 gives 1024 + 16 v. One packed
//     f16 add / fma then removes the bias and applies an integer sub-scale;
//     whenever the result is an integer below 2048 in magnitude it is exact, and
//     otherwise (Q6_K, IQ4_XS codes above 2048) the single rounding of the fused
//     operation equals rounding the exact integer to f16.
//   * 16-entry codebooks (IQ4_NL / IQ4_XS values, E2M1) live in four 32-bit
//     registers as biased bytes; a byte permute (prmt) looks up four nibbles at
//     once, two permutes cover the two halves of the table and a third picks
//     per byte by the nibble's top bit.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "sm100_async.cuh"

namespace qmm {

// ------------------------------------------------------------ bit helpers
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// (a & b) | c
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hadd2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// f16 bits of v (exactly representable here) in both halves
__device__ __forceinline__ uint32_t h2dup(float v) {
    const uint32_t b = __half_as_ushort(__float2half_rn(v));
    return b | (b << 16);
}

// f16 bit pattern of an integer |v| < 2048 (exact), duplicated into both halves
__host__ __device__ constexpr uint32_t h2int(int v) {
    const uint32_t s = v < 0 ? 0x8000u : 0u;
    const uint32_t a = static_cast<uint32_t>(v < 0 ? -v : v);
    if (a == 0) return (s << 16) | s;
    int e = 0;
    while ((a >> (e + 1)) != 0) ++e;
    const uint32_t m = (a << (10 - e)) & 0x3FFu;
    const uint32_t h = s | (static_cast<uint32_t>(e + 15) << 10) | m;
    return (h << 16) | h;
}
static_assert(h2int(1024) == 0x64006400u && h2int(-1152) == 0xE480E480u && h2int(1) == 0x3C003C00u, "f16 ints");
constexpr uint32_t kH2Sixteenth = 0x2C002C00u;   // 1/16 in both halves
constexpr uint32_t kMag16 = 0x64006400u;         // 1024.0h, 1024.0h
constexpr uint32_t kMagB = 0x64646464u;          // high byte of 1024.0h in every byte
constexpr uint32_t kMagB512 = 0x60606060u;       // high byte of 512.0h (ulp 0.5)

// four table bytes packed little-endian
__host__ __device__ constexpr uint32_t pack4(int a, int b, int c, int d) {
    return (static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8) |
           ((static_cast<uint32_t>(c) & 0xFFu) << 16) | ((static_cast<uint32_t>(d) & 0xFFu) << 24);
}
// IQ4_NL / IQ4_XS codebook (ferrox-cuda 0.20.0 src/mul_mm_kinds/codebook.rs),
// each value biased by +128 into an unsigned byte.
struct KvTable {
    static constexpr uint32_t T0 = pack4(-127 + 128, -104 + 128, -83 + 128, -65 + 128);
    static constexpr uint32_t T1 = pack4(-49 + 128, -35 + 128, -22 + 128, -10 + 128);
    static constexpr uint32_t T2 = pack4(1 + 128, 13 + 128, 25 + 128, 38 + 128);
    static constexpr uint32_t T3 = pack4(53 + 128, 69 + 128, 89 + 128, 113 + 128);
};
// E2M1 values (same page; code 8 is -0.0, stored here as 0) times 2, biased
// by +128: with the 512.0h magic (ulp 0.5) the byte b decodes to b / 2 - 64.
struct E2m1Table {
    static constexpr uint32_t T0 = pack4(128 + 0, 128 + 1, 128 + 2, 128 + 3);
    static constexpr uint32_t T1 = pack4(128 + 4, 128 + 6, 128 + 8, 128 + 12);
    static constexpr uint32_t T2 = pack4(128 - 0, 128 - 1, 128 - 2, 128 - 3);
    static constexpr uint32_t T3 = pack4(128 - 4, 128 - 6, 128 - 8, 128 - 12);
};

// Table bytes of the four nibbles in the low 16 bits of idx: result byte k is
// entry (idx >> 4k) & 15.
template <typename T>
__device__ __forceinline__ uint32_t lut16(uint32_t idx) {
    const uint32_t i3 = idx & 0x7777u;
    const uint32_t lo = prmt(T::T0, T::T1, i3);
    const uint32_t hi = prmt(T::T2, T::T3, i3);
    const uint32_t pick = lop_and_or(idx >> 1, 0x4444u, 0x3210u);   // byte k of hi if bit 3 of nibble k
    return prmt(lo, hi, pick);
}

// NW consecutive little-endian 32-bit words starting at shared-memory byte
// address p, which is ALIGN-byte aligned (1, 2 or 4; 16 allows 16-byte loads).
template <int NW, int ALIGN>
__device__ __forceinline__ void ld_words(const uint8_t* p, uint32_t (&w)[NW]) {
    if constexpr (ALIGN % 16 == 0 && NW % 4 == 0) {
#pragma unroll
        for (int i = 0; i < NW / 4; ++i) {
            const uint4 v = reinterpret_cast<const uint4*>(p)[i];
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
    } else if constexpr (ALIGN % 4 == 0) {
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = reinterpret_cast<const uint32_t*>(p)[i];
    } else {
        const uint32_t mis = smem_u32(p) & 3u;
        const uint32_t* q = reinterpret_cast<const uint32_t*>(p - mis);
        const uint32_t sh = mis * 8u;
        uint32_t prev = q[0];
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const uint32_t nx = q[i + 1];
            w[i] = __funnelshift_r(prev, nx, sh);
            prev = nx;
        }
    }
}

template <int KIND> struct FastDec;
// Formats whose decoder takes per-super-block scale words (pre / sub_pre).
template <int KIND> struct FastDecPre {
    static constexpr bool ON = KIND == Q4_K || KIND == Q5_K || KIND == Q6_K || KIND == Q2_K || KIND == Q3_K ||
                               KIND == IQ4_XS || KIND == MXFP4;
};

// ---------------------------------------------------------------------------
// 32-element formats: sub-step q covers blocks 2q and 2q + 1 of the super-step.
// In each block, byte j of the nibble field holds element j (low nibble) and
// element j + 16 (high nibble). Block b's elements land in o[16 b' + e / 2].
// ---------------------------------------------------------------------------
template <> struct FastDec<Q8_0> {
    __device__ __forceinline__ static void sub(const uint8_t* row, int q, uint32_t (&o)[32]) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t w[8];
            ld_words<8, 2>(row + (2 * q + hb) * 34 + 2, w);
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
                const uint32_t u = w[wi] ^ 0x80808080u;   // int8 -> byte + 128
                o[16 * hb + 2 * wi] = hadd2_u(prmt(u, kMagB, 0x4140), h2int(-1152));
                o[16 * hb + 2 * wi + 1] = hadd2_u(prmt(u, kMagB, 0x4342), h2int(-1152));
            }
        }
    }
};

template <> struct FastDec<Q4_0> {
    __device__ __forceinline__ static void sub(const uint8_t* row, int q, uint32_t (&o)[32]) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t w[4];
            ld_words<4, 2>(row + (2 * q + hb) * 18 + 2, w);
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const uint32_t t01 = prmt(w[wi], 0u, 0x4140), t23 = prmt(w[wi], 0u, 0x4342);
                // low nibble: 1024 + n - 1032 = n - 8; high: (1024 + 16 n) / 16 - 72 = n - 8
                o[16 * hb + 2 * wi] = hadd2_u(lop_and_or(t01, 0x000F000Fu, kMag16), h2int(-1032));
                o[16 * hb + 2 * wi + 1] = hadd2_u(lop_and_or(t23, 0x000F000Fu, kMag16), h2int(-1032));
                o[16 * hb + 8 + 2 * wi] = hfma2_u(lop_and_or(t01, 0x00F000F0u, kMag16), kH2Sixteenth, h2int(-72));
                o[16 * hb + 9 + 2 * wi] = hfma2_u(lop_and_or(t23, 0x00F000F0u, kMag16), kH2Sixteenth, h2int(-72));
            }
        }
    }
};

template <> struct FastDec<Q5_0> {
    __device__ __forceinline__ static void sub(const uint8_t* row, int q, uint32_t (&o)[32]) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t w[5];   // qh, then the 16 nibble bytes
            ld_words<5, 2>(row + (2 * q + hb) * 22 + 2, w);
            const uint32_t qh = w[0];
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const uint32_t t01 = prmt(w[1 + wi], 0u, 0x4140), t23 = prmt(w[1 + wi], 0u, 0x4342);
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const uint32_t t = p ? t23 : t01;
                    const int e = 4 * wi + 2 * p;   // element pair (e, e + 1) and (16 + e, 17 + e)
                    // 5th bits of elements e, e + 1 to bits 4 / 20 (low) and of 16 + e, 17 + e to
                    // bits 8 / 24 (high, where the nibble sits at bits 4..7)
                    const uint32_t ml = lop_and_or(((qh >> e) & 3u) * 0x00080010u, 0x00100010u, kMag16);
                    const uint32_t mh = lop_and_or(((qh >> (16 + e)) & 3u) * 0x00800100u, 0x01000100u, kMag16);
                    o[16 * hb + e / 2] = hadd2_u(lop_and_or(t, 0x000F000Fu, ml), h2int(-1040));
                    o[16 * hb + 8 + e / 2] = hfma2_u(lop_and_or(t, 0x00F000F0u, mh), kH2Sixteenth, h2int(-80));
                }
            }
        }
    }
};

// Q8_1: Q8_0's codes after a 4-byte head (d and an unread f16), 36-byte blocks
// (every field 4-byte aligned).
template <> struct FastDec<Q8_1> {
    __device__ __forceinline__ static void sub(const uint8_t* row, int q, uint32_t (&o)[32]) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t w[8];
            ld_words<8, 4>(row + (2 * q + hb) * 36 + 4, w);
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
                const uint32_t u = w[wi] ^ 0x80808080u;
                o[16 * hb + 2 * wi] = hadd2_u(prmt(u, kMagB, 0x4140), h2int(-1152));
                o[16 * hb + 2 * wi + 1] = hadd2_u(prmt(u, kMagB, 0x4342), h2int(-1152));
            }
        }
    }
};

// Q4_1 (20-byte blocks, codes at byte 4) and Q5_1 (24-byte blocks, qh at byte
// 4, codes at byte 8): Q4_0's and Q5_0's unpack with unsigned codes (no bias);
// the min term comes from the min MMA, the scale d from the epilogue.
template <> struct FastDec<Q4_1> {
    __device__ __forceinline__ static void sub(const uint8_t* row, int q, uint32_t (&o)[32]) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t w[4];
            ld_words<4, 4>(row + (2 * q + hb) * 20 + 4, w);
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const uint32_t t01 = prmt(w[wi], 0u, 0x4140), t23 = prmt(w[wi], 0u, 0x4342);
                // low nibble: 1024 + n - 1024; high: (1024 + 16 n) / 16 - 64
                o[16 * hb + 2 * wi] = hadd2_u(lop_and_or(t01, 0x000F000Fu, kMag16), h2int(-1024));
                o[16 * hb + 2 * wi + 1] = hadd2_u(lop_and_or(t23, 0x000F000Fu, kMag16), h2int(-1024));
                o[16 * hb + 8 + 2 * wi] = hfma2_u(lop_and_or(t01, 0x00F000F0u, kMag16), kH2Sixteenth, h2int(-64));
                o[16 * hb + 9 + 2 * wi] = hfma2_u(lop_and_or(t23, 0x00F000F0u, kMag16), kH2Sixteenth, h2int(-64));
            }
        }
    }
};

template <> struct FastDec<Q5_1> {
    __device__ __forceinline__ static void sub(const uint8_t* row, int q, uint32_t (&o)[32]) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t w[5];   // qh, then the 16 nibble bytes
            ld_words<5, 4>(row + (2 * q + hb) * 24 + 4, w);
            const uint32_t qh = w[0];
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const uint32_t t01 = prmt(w[1 + wi], 0u, 0x4140), t23 = prmt(w[1 + wi], 0u, 0x4342);
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const uint32_t t = p ? t23 : t01;
                    const int e = 4 * wi + 2 * p;
                    const uint32_t ml = lop_and_or(((qh >> e) & 3u) * 0x00080010u, 0x00100010u, kMag16);
                    const uint32_t mh = lop_and_or(((qh >> (16 + e)) & 3u) * 0x00800100u, 0x01000100u, kMag16);
                    o[16 * hb + e / 2] = hadd2_u(lop_and_or(t, 0x000F000Fu, ml), h2int(-1024));
                    o[16 * hb + 8 + e / 2] = hfma2_u(lop_and_or(t, 0x00F000F0u, mh), kH2Sixteenth, h2int(-64));
                }
            }
        }
    }
};

// Codebook formats with one 16-byte nibble field per 32 elements.
template <typename T, uint32_t MAGB, uint32_t BIAS>
__device__ __forceinline__ void lut_block(const uint32_t (&w)[4], uint32_t scale, uint32_t bias, bool scaled,
                                          uint32_t* o) {
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        // ra = values of elements 4wi, 16 + 4wi, 4wi + 1, 17 + 4wi; rb = the next two pairs
        const uint32_t ra = lut16<T>(w[wi]), rb = lut16<T>(w[wi] >> 16);
        const uint32_t c[4] = {prmt(ra, MAGB, 0x4240), prmt(rb, MAGB, 0x4240), prmt(ra, MAGB, 0x4341),
                               prmt(rb, MAGB, 0x4341)};
        const int dst[4] = {2 * wi, 2 * wi + 1, 8 + 2 * wi, 9 + 2 * wi};
#pragma unroll
        for (int k = 0; k < 4; ++k) o[dst[k]] = scaled ? hfma2_u(c[k], scale, bias) : hadd2_u(c[k], BIAS);
    }
}

template <> struct FastDec<IQ4_NL> {
    __device__ __forceinline__ static void sub(const uint8_t* row, int q, uint32_t (&o)[32]) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t w[4];
            ld_words<4, 2>(row + (2 * q + hb) * 18 + 2, w);
            lut_block<KvTable, kMagB, h2int(-1152)>(w, 0u, 0u, false, o + 16 * hb);
        }
    }
};

// MXFP4 on the super-block pipeline: the eight block exponents of a
// 256-element super-step are folded into the operands relative to the largest
// one, e_max (2^(e_max - 127) multiplies the super-block's partial sums): a
// block's codes are scaled by 2^-(e_max - e), an exact f16 power of two (zero
// below 2^-24, when the exponents of one super-step span more than 24). The
// operand E2M1 * 2^-(e_max - e) is exact for spreads up to 23; at 24 the codes
// +-0.5 and +-1.5 round to even.
__device__ __forceinline__ uint32_t h2pow2neg(uint32_t k) {
    const uint32_t h = k <= 14u ? ((15u - k) << 10) : (k <= 24u ? (1u << (24u - k)) : 0u);
    return h | (h << 16);
}
template <> struct FastDec<MXFP4> {
    // scw[b] = 2^-(e_max - e_b) for the super-step's eight blocks, f16x2
    __device__ __forceinline__ static void pre(const uint8_t* row, uint32_t (&scw)[8]) {
        uint32_t e[8], emax = 0;
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
            e[blk] = row[17 * blk];
            emax = max(emax, e[blk]);
        }
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) scw[blk] = h2pow2neg(emax - e[blk]);
    }
    __device__ __forceinline__ static void sub_pre(const uint8_t* row, int q, uint32_t (&o)[32],
                                                   const uint32_t (&scw)[8]) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            const int j = 2 * q + hb;
            const uint32_t sc = q == 0 ? (hb ? scw[1] : scw[0])
                              : q == 1 ? (hb ? scw[3] : scw[2])
                              : q == 2 ? (hb ? scw[5] : scw[4])
                                       : (hb ? scw[7] : scw[6]);
            uint32_t w[4];
            ld_words<4, 1>(row + 17 * j + 1, w);
            // (512 + b / 2) * s - 576 * s = E2M1 value * s, one rounding
            lut_block<E2m1Table, kMagB512, 0u>(w, sc, hmul2_u(sc, h2int(-576)), true, o + 16 * hb);
        }
    }
};

// ---------------------------------------------------------------------------
// 256-element formats: sub-step q covers 32-element sub-blocks 2q and 2q + 1.
// ---------------------------------------------------------------------------
template <> struct FastDec<IQ4_XS> {
    // the eight 6-bit group scales minus 32 as exact f16: low nibbles from
    // scales_l (even groups low, odd groups high nibble of each byte), the two
    // high bits from scales_h spread one nibble per byte. scw[0..1] hold the
    // even groups (0, 2), (4, 6); scw[2..3] the odd ones (1, 3), (5, 7).
    __device__ __forceinline__ static void pre(const uint8_t* row, uint32_t (&scw)[8]) {
        uint32_t hdr[2];   // d | scales_h << 16, scales_l
        ld_words<2, 8>(row, hdr);
        const uint32_t sh = hdr[0] >> 16, sl = hdr[1];
        const uint32_t t = (sh & 0xFu) | ((sh & 0xF0u) << 4) | ((sh & 0xF00u) << 8) | ((sh & 0xF000u) << 12);
        const uint32_t ce = (sl & 0x0F0F0F0Fu) | ((t & 0x03030303u) << 4);
        const uint32_t co = ((sl >> 4) & 0x0F0F0F0Fu) | (((t >> 2) & 0x03030303u) << 4);
        scw[0] = hadd2_u(prmt(ce, kMagB, 0x4140u), h2int(-1056));
        scw[1] = hadd2_u(prmt(ce, kMagB, 0x4342u), h2int(-1056));
        scw[2] = hadd2_u(prmt(co, kMagB, 0x4140u), h2int(-1056));
        scw[3] = hadd2_u(prmt(co, kMagB, 0x4342u), h2int(-1056));
    }
    __device__ __forceinline__ static void sub_pre(const uint8_t* row, int q, uint32_t (&o)[32],
                                                   const uint32_t (&scw)[8]) {
        const uint32_t sel = (q & 1) ? 0x3232u : 0x1010u;
        const uint32_t we = (q < 2) ? scw[0] : scw[1], wo = (q < 2) ? scw[2] : scw[3];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            const int j = 2 * q + hb;
            const uint32_t sc = prmt(hb ? wo : we, hb ? wo : we, sel);
            uint32_t w[4];
            ld_words<4, 8>(row + 8 + 16 * j, w);
            // (1024 + b) * sc - 1152 * sc = KV * sc, one rounding
            lut_block<KvTable, kMagB, 0u>(w, sc, hmul2_u(sc, h2int(-1152)), true, o + 16 * hb);
        }
    }
};

// Q4_K / Q5_K integer sub-scales, once per super-block: the eight 6-bit
// scales of the 12-byte field (bytes 0..3 low 6 bits; bytes 8..11 low nibble
// with the top 2 bits of bytes 0..3), extracted word-wide and made exact f16
// pairs (1024 + sc under the 0x64 magic byte, minus 1024): scw[i] holds the
// scales of sub-blocks 2i and 2i + 1.
__device__ __forceinline__ void k4_scale_words(const uint8_t* row, uint32_t (&scw)[8]) {
    const uint32_t* f = reinterpret_cast<const uint32_t*>(row + 4);   // 4-byte aligned in the stage
    const uint32_t s0 = f[0], s2 = f[2];
    const uint32_t lo4 = s0 & 0x3F3F3F3Fu;
    const uint32_t hi4 = (s2 & 0x0F0F0F0Fu) | (((s0 >> 6) & 0x03030303u) << 4);
    scw[0] = hadd2_u(prmt(lo4, kMagB, 0x4140u), h2int(-1024));
    scw[1] = hadd2_u(prmt(lo4, kMagB, 0x4342u), h2int(-1024));
    scw[2] = hadd2_u(prmt(hi4, kMagB, 0x4140u), h2int(-1024));
    scw[3] = hadd2_u(prmt(hi4, kMagB, 0x4342u), h2int(-1024));
}

// The four f16x2 operands of sub-step q from the scale words: the low
// sub-block's scale sc0 (a0 = sc0, b0 = -1024 sc0) and the high one's
// (a1 = sc1 / 16, b1 = -64 sc1), all exact in f16.
__device__ __forceinline__ void k4_sub_operands(const uint32_t (&scw)[8], int q, uint32_t& a0, uint32_t& b0,
                                                uint32_t& a1, uint32_t& b1) {
    const uint32_t w = q == 0 ? scw[0] : q == 1 ? scw[1] : q == 2 ? scw[2] : scw[3];
    a0 = prmt(w, w, 0x1010u);
    const uint32_t s1 = prmt(w, w, 0x3232u);
    b0 = hmul2_u(a0, h2int(-1024));
    a1 = hmul2_u(s1, kH2Sixteenth);
    b1 = hmul2_u(s1, h2int(-64));
}

// The four per-16-element scales of sub-step q (groups 4q .. 4q + 3) from
// eight precomputed f16x2 words, each duplicated into both halves.
__device__ __forceinline__ void group_scales(const uint32_t (&scw)[8], int q, uint32_t (&S)[4]) {
    const uint32_t w0 = q == 0 ? scw[0] : q == 1 ? scw[2] : q == 2 ? scw[4] : scw[6];
    const uint32_t w1 = q == 0 ? scw[1] : q == 1 ? scw[3] : q == 2 ? scw[5] : scw[7];
    S[0] = prmt(w0, w0, 0x1010u);
    S[1] = prmt(w0, w0, 0x3232u);
    S[2] = prmt(w1, w1, 0x1010u);
    S[3] = prmt(w1, w1, 0x3232u);
}

// Q4_K: code bytes 16 + 32q .. +32; low nibbles are sub-block 2q, high 2q + 1.
template <> struct FastDec<Q4_K> {
    __device__ __forceinline__ static void pre(const uint8_t* row, uint32_t (&scw)[8]) { k4_scale_words(row, scw); }
    // sub-step q with the super-block's scale words precomputed
    __device__ __forceinline__ static void sub_pre(const uint8_t* row, int q, uint32_t (&o)[32],
                                                   const uint32_t (&scw)[8]) {
        uint32_t a0, b0, a1, b1;
        k4_sub_operands(scw, q, a0, b0, a1, b1);
        uint32_t w[8];
        ld_words<8, 16>(row + 16 + 32 * q, w);
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            const uint32_t t01 = prmt(w[wi], 0u, 0x4140), t23 = prmt(w[wi], 0u, 0x4342);
            o[2 * wi] = hfma2_u(lop_and_or(t01, 0x000F000Fu, kMag16), a0, b0);
            o[2 * wi + 1] = hfma2_u(lop_and_or(t23, 0x000F000Fu, kMag16), a0, b0);
            o[16 + 2 * wi] = hfma2_u(lop_and_or(t01, 0x00F000F0u, kMag16), a1, b1);
            o[17 + 2 * wi] = hfma2_u(lop_and_or(t23, 0x00F000F0u, kMag16), a1, b1);
        }
    }
};

// Q5_K: as Q4_K with code bytes at 48 + 32q and the 5th bit of element i of
// sub-block j in bit j of qh[i] (qh at byte 16).
template <> struct FastDec<Q5_K> {
    __device__ __forceinline__ static void pre(const uint8_t* row, uint32_t (&scw)[8]) { k4_scale_words(row, scw); }
    // sub-step q with the super-block's scale words precomputed
    __device__ __forceinline__ static void sub_pre(const uint8_t* row, int q, uint32_t (&o)[32],
                                                   const uint32_t (&scw)[8]) {
        uint32_t a0, b0, a1, b1;
        k4_sub_operands(scw, q, a0, b0, a1, b1);
        uint32_t w[8], h[8];
        ld_words<8, 16>(row + 48 + 32 * q, w);
        ld_words<8, 16>(row + 16, h);
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const uint32_t sel = p ? 0x4342u : 0x4140u;
                const uint32_t t = prmt(w[wi], 0u, sel);
                const uint32_t x = prmt(h[wi], 0u, sel) >> (2 * q);   // bit 0/16: sub-block 2q; 1/17: 2q + 1
                const uint32_t ml = lop_and_or(x << 4, 0x00100010u, kMag16);
                const uint32_t mh = lop_and_or(x << 7, 0x01000100u, kMag16);
                o[2 * wi + p] = hfma2_u(lop_and_or(t, 0x000F000Fu, ml), a0, b0);
                o[16 + 2 * wi + p] = hfma2_u(lop_and_or(t, 0x00F000F0u, mh), a1, b1);
            }
        }
    }
};

// Q6_K: sub-block j = 2q + hb reads ql[64 (q >> 1) + 32 hb + i] (high nibble
// when q is odd) and bits 2 (j & 3) .. +1 of qh[128 + 32 (q >> 1) + i];
// int8 scale per 16 elements at 192 + 2j + i / 16.
// Four codes at a time: the low nibbles and the two high bits of four
// elements are merged into four bytes with word-wide shifts and masks, and
// each byte pair becomes an f16 pair 1024 + code under the 0x64 magic byte.
template <> struct FastDec<Q6_K> {
    // the sixteen int8 scales (bytes 192..207) as exact f16: byte ^ 0x80
    // under the 0x64 magic byte is 1024 + b + 128, minus 1152
    __device__ __forceinline__ static void pre(const uint8_t* row, uint32_t (&scw)[8]) {
        uint32_t sw[4];
        ld_words<4, 2>(row + 192, sw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t u = sw[i] ^ 0x80808080u;
            scw[2 * i] = hadd2_u(prmt(u, kMagB, 0x4140u), h2int(-1152));
            scw[2 * i + 1] = hadd2_u(prmt(u, kMagB, 0x4342u), h2int(-1152));
        }
    }
    __device__ __forceinline__ static void sub_pre(const uint8_t* row, int q, uint32_t (&o)[32],
                                                   const uint32_t (&scw)[8]) {
        const int h = q >> 1, nib = q & 1;
        uint32_t hq[8], S[4];
        ld_words<8, 2>(row + 128 + 32 * h, hq);
        group_scales(scw, q, S);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t w[8];
            ld_words<8, 2>(row + 64 * h + 32 * hb, w);
            const int gs = 4 * nib + 2 * hb;
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
                const uint32_t hi = ((hq[wi] >> gs) << 4) & 0x30303030u;
                const uint32_t code = lop_and_or(w[wi] >> (4 * nib), 0x0F0F0F0Fu, hi);
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const uint32_t c = hadd2_u(prmt(code, kMagB, p ? 0x4342u : 0x4140u), h2int(-1056));
                    o[16 * hb + 2 * wi + p] = hmul2_u(c, S[2 * hb + (wi >> 2)]);
                }
            }
        }
    }
};

// Q2_K: sub-block j = 2q + hb reads bits 2 (j & 3) .. +1 of qs[16 + 32 (q >> 1) + i];
// 4-bit scale per 16 elements in the low nibble of byte 2j + i / 16.
template <> struct FastDec<Q2_K> {
    // the sixteen 4-bit scales (low nibbles of bytes 0..15) as exact f16
    __device__ __forceinline__ static void pre(const uint8_t* row, uint32_t (&scw)[8]) {
        uint32_t sw[4];
        ld_words<4, 4>(row, sw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t m = sw[i] & 0x0F0F0F0Fu;
            scw[2 * i] = hadd2_u(prmt(m, kMagB, 0x4140u), h2int(-1024));
            scw[2 * i + 1] = hadd2_u(prmt(m, kMagB, 0x4342u), h2int(-1024));
        }
    }
    __device__ __forceinline__ static void sub_pre(const uint8_t* row, int q, uint32_t (&o)[32],
                                                   const uint32_t (&scw)[8]) {
        uint32_t w[8], A[4], B[4];
        ld_words<8, 4>(row + 16 + 32 * (q >> 1), w);
        group_scales(scw, q, A);
#pragma unroll
        for (int k = 0; k < 4; ++k) B[k] = hmul2_u(A[k], h2int(-1024));
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            const int gs = 4 * (q & 1) + 2 * hb;
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const uint32_t t = prmt(w[wi], 0u, p ? 0x4342u : 0x4140u) >> gs;
                    const int k = 2 * hb + (wi >> 2);
                    o[16 * hb + 2 * wi + p] = hfma2_u(lop_and_or(t, 0x00030003u, kMag16), A[k], B[k]);
                }
            }
        }
    }
};

// Q3_K: sub-block j = 2q + hb reads bits 2 (j & 3) .. +1 of qs[32 + 32 (q >> 1) + i]
// and bit j of hmask[i] (clear = subtract 4); 6-bit scale per 16 elements.
template <> struct FastDec<Q3_K> {
    // the sixteen 6-bit scales of the 12-byte field at 96, minus 32, as exact
    // f16: low nibbles from bytes 0..7 (low / high halves), the 2 high bits
    // from bytes 8..11 shifted by 2 per group of four
    __device__ __forceinline__ static void pre(const uint8_t* row, uint32_t (&scw)[8]) {
        uint32_t f[3];
        ld_words<3, 2>(row + 96, f);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t lo = (g == 0) ? (f[0] & 0x0F0F0F0Fu) : (g == 1) ? (f[1] & 0x0F0F0F0Fu)
                              : (g == 2) ? ((f[0] >> 4) & 0x0F0F0F0Fu) : ((f[1] >> 4) & 0x0F0F0F0Fu);
            const uint32_t code = lo | (((f[2] >> (2 * g)) & 0x03030303u) << 4);
            scw[2 * g] = hadd2_u(prmt(code, kMagB, 0x4140u), h2int(-1056));
            scw[2 * g + 1] = hadd2_u(prmt(code, kMagB, 0x4342u), h2int(-1056));
        }
    }
    __device__ __forceinline__ static void sub_pre(const uint8_t* row, int q, uint32_t (&o)[32],
                                                   const uint32_t (&scw)[8]) {
        uint32_t hm[8], w[8], S[4];
        ld_words<8, 2>(row, hm);
        ld_words<8, 2>(row + 32 + 32 * (q >> 1), w);
        group_scales(scw, q, S);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            const int j = 2 * q + hb;
            const int gs = 4 * (q & 1) + 2 * hb;
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const uint32_t sel = p ? 0x4342u : 0x4140u;
                    const uint32_t mk = lop_and_or(prmt(hm[wi], 0u, sel) >> j << 2, 0x00040004u, kMag16);
                    const uint32_t c16 = lop_and_or(prmt(w[wi], 0u, sel) >> gs, 0x00030003u, mk);
                    o[16 * hb + 2 * wi + p] = hmul2_u(hadd2_u(c16, h2int(-1028)), S[2 * hb + (wi >> 2)]);
                }
            }
        }
    }
};

}  // namespace qmm
