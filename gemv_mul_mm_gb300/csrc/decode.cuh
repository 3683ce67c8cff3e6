// decode.cuh -- device-side block-format decoders for sm_103a.
//
// Each format is decoded per 32-element sub-block ("chunk" j of a block):
// chunk j of a 256-element super-block covers elements [32j, 32j + 32), and the
// 32-element formats have a single chunk. The byte layouts are those of the
// pages: Vulkore examples/llm/quant_test.cpp (`ref::q8_0`, `ref::q5_0`,
// `ref::q4_k`, `ref::q6_k`), ferrox-cuda 0.20.0 src/mul_mm_kinds/codebook.rs
// (IQ4_NL, IQ4_XS, MXFP4 and their codebooks), ferrox-cuda 0.21.0
// src/mul_mm.rs (Q4_0 packing, Q5_K sharing Q4_K's 6-bit scale/min unpack, the
// Q3_K hmask bias) and, where the pages name a format without its layout
// (Q5_K, Q2_K, Q3_K), the public GGUF block definitions.
//
// Arithmetic: every product is exact in fp32 (f16 scale <= 11 significant bits
// times small integers), so any evaluation order gives the same bits; the
// affine-min formats round once at the final subtraction. f16 -> f32 uses the
// hardware conversion (exact, subnormals kept). Kernels are built without
// -ftz / fast-math so fp32 subnormals (MXFP4 with small E8M0) survive.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace qmm {

enum Kind : int {
    Q8_0 = 0, Q4_0 = 1, Q5_0 = 2, Q4_K = 3, Q5_K = 4, Q6_K = 5,
    Q2_K = 6, Q3_K = 7, IQ4_NL = 8, IQ4_XS = 9, MXFP4 = 10,
    Q4_1 = 11, Q5_1 = 12, Q8_1 = 13, NKINDS = 14,
    // Library-internal layouts made by qrepack (not block formats of the ABI):
    // Q8_0 / Q4_0 rows as units of eight blocks, the eight code fields back to
    // back (32 / 16 bytes each) and then the eight f16 scales (16 bytes).
    Q8_0R = 32, Q4_0R = 33
};

template <int KIND> struct Geo;
template <> struct Geo<Q8_0>   { static constexpr int BB = 34,  BE = 32;  };
template <> struct Geo<Q4_0>   { static constexpr int BB = 18,  BE = 32;  };
template <> struct Geo<Q5_0>   { static constexpr int BB = 22,  BE = 32;  };
template <> struct Geo<Q4_K>   { static constexpr int BB = 144, BE = 256; };
template <> struct Geo<Q5_K>   { static constexpr int BB = 176, BE = 256; };
template <> struct Geo<Q6_K>   { static constexpr int BB = 210, BE = 256; };
template <> struct Geo<Q2_K>   { static constexpr int BB = 84,  BE = 256; };
template <> struct Geo<Q3_K>   { static constexpr int BB = 110, BE = 256; };
template <> struct Geo<IQ4_NL> { static constexpr int BB = 18,  BE = 32;  };
template <> struct Geo<IQ4_XS> { static constexpr int BB = 136, BE = 256; };
template <> struct Geo<MXFP4>  { static constexpr int BB = 17,  BE = 32;  };
template <> struct Geo<Q4_1>   { static constexpr int BB = 20,  BE = 32;  };
template <> struct Geo<Q5_1>   { static constexpr int BB = 24,  BE = 32;  };
template <> struct Geo<Q8_1>   { static constexpr int BB = 36,  BE = 32;  };
template <> struct Geo<Q8_0R>  { static constexpr int BB = 34,  BE = 32;  };
template <> struct Geo<Q4_0R>  { static constexpr int BB = 18,  BE = 32;  };

// 16-entry codebooks. IQ4_NL/IQ4_XS values and the E2M1 values (code 8 is
// negative zero) as the codebook.rs page lists them.
static __constant__ float c_kv_iq4nl[16] = {-127.f, -104.f, -83.f, -65.f, -49.f, -35.f, -22.f, -10.f,
                                            1.f, 13.f, 25.f, 38.f, 53.f, 69.f, 89.f, 113.f};
static __constant__ float c_kv_e2m1[16] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f,
                                           -0.f, -0.5f, -1.f, -1.5f, -2.f, -3.f, -4.f, -6.f};

__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xFFFFu)));
}

// E8M0: the byte is an fp32 exponent field; 0 means 2^-127, the fp32
// subnormal with only mantissa bit 22 set (codebook.rs, `ferrox_e8m0_to_f32`).
__device__ __forceinline__ float e8m0f(uint32_t e) {
    return e == 0 ? __int_as_float(0x00400000) : __int_as_float(static_cast<int>(e << 23));
}

template <typename P>
__device__ __forceinline__ uint32_t ld8(const P* b, int o) { return reinterpret_cast<const uint8_t*>(b)[o]; }
template <typename P>
__device__ __forceinline__ uint32_t ld16(const P* b, int o) { return ld8(b, o) | (ld8(b, o + 1) << 8); }

// Q4_K / Q5_K (scale, min) of 32-element sub-block j from the 12-byte field.
__device__ __forceinline__ void k4_sm(const uint8_t* s, int j, int& sc, int& mn) {
    if (j < 4) {
        sc = s[j] & 63;
        mn = s[j + 4] & 63;
    } else {
        sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

// Q3_K 6-bit scale of 16-element sub-block j (unbiased value, 0..63).
__device__ __forceinline__ int q3_scale(const uint8_t* s, int j) {
    const int lo = (j < 8) ? (s[j] & 15) : (s[j - 8] >> 4);
    const int hi = (s[8 + (j & 3)] >> (2 * (j >> 2))) & 3;
    return lo | (hi << 4);
}

// Element i (0..31) of chunk j of the block at b. Byte loads only: no
// alignment is assumed (MXFP4's 17-byte stride puts blocks on odd addresses).
template <int KIND>
__device__ __forceinline__ float elem32(const uint8_t* b, int j, int i) {
    if constexpr (KIND == Q8_0) {
        return h2f(ld16(b, 0)) * static_cast<float>(static_cast<int8_t>(b[2 + i]));
    } else if constexpr (KIND == Q4_0 || KIND == IQ4_NL) {
        const uint32_t byte = b[2 + (i & 15)];
        const int c = (i < 16) ? (byte & 15) : (byte >> 4);
        if constexpr (KIND == Q4_0) return h2f(ld16(b, 0)) * static_cast<float>(c - 8);
        else return h2f(ld16(b, 0)) * c_kv_iq4nl[c];
    } else if constexpr (KIND == Q5_0) {
        const uint32_t qh = ld8(b, 2) | (ld8(b, 3) << 8) | (ld8(b, 4) << 16) | (ld8(b, 5) << 24);
        const uint32_t byte = b[6 + (i & 15)];
        const int lo = (i < 16) ? (byte & 15) : (byte >> 4);
        const int q = lo | (((qh >> i) & 1) << 4);
        return h2f(ld16(b, 0)) * static_cast<float>(q - 16);
    } else if constexpr (KIND == Q4_K || KIND == Q5_K) {
        int sc, mn;
        k4_sm(b + 4, j, sc, mn);
        const int qs = (KIND == Q4_K) ? 16 : 48;
        const uint32_t byte = b[qs + (j >> 1) * 32 + i];
        int q = (j & 1) ? (byte >> 4) : (byte & 15);
        if constexpr (KIND == Q5_K) q += ((b[16 + i] >> j) & 1) << 4;
        const float ds = h2f(ld16(b, 0)) * static_cast<float>(sc);
        const float dm = h2f(ld16(b, 2)) * static_cast<float>(mn);
        return __fsub_rn(__fmul_rn(ds, static_cast<float>(q)), dm);
    } else if constexpr (KIND == Q6_K) {
        const int h = j >> 2, g = j & 3;
        const uint32_t lob = b[h * 64 + i + (g & 1) * 32];
        const int lo = (g >= 2) ? (lob >> 4) : (lob & 15);
        const int hi = (b[128 + h * 32 + i] >> (2 * g)) & 3;
        const int sc = static_cast<int8_t>(b[192 + 2 * j + (i >> 4)]);
        return h2f(ld16(b, 208)) * static_cast<float>(sc) * static_cast<float>((lo | (hi << 4)) - 32);
    } else if constexpr (KIND == Q2_K) {
        const int h = j >> 2, g = j & 3;
        const int q = (b[16 + h * 32 + i] >> (2 * g)) & 3;
        const int s = b[2 * j + (i >> 4)];
        const float dl = h2f(ld16(b, 80)) * static_cast<float>(s & 15);
        const float ml = h2f(ld16(b, 82)) * static_cast<float>(s >> 4);
        return __fsub_rn(__fmul_rn(dl, static_cast<float>(q)), ml);
    } else if constexpr (KIND == Q3_K) {
        const int h = j >> 2, g = j & 3;
        const int q2 = (b[32 + h * 32 + i] >> (2 * g)) & 3;
        const int q = q2 - (((b[i] >> j) & 1) ? 0 : 4);
        const int sc = q3_scale(b + 96, 2 * j + (i >> 4)) - 32;
        return h2f(ld16(b, 108)) * static_cast<float>(sc) * static_cast<float>(q);
    } else if constexpr (KIND == IQ4_XS) {
        const uint32_t byte = b[8 + 16 * j + (i & 15)];
        const int c = (i < 16) ? (byte & 15) : (byte >> 4);
        const uint32_t sh = ld16(b, 2);
        const int ls = ((b[4 + (j >> 1)] >> (4 * (j & 1))) & 15) | (((sh >> (2 * j)) & 3) << 4);
        return h2f(ld16(b, 0)) * static_cast<float>(ls - 32) * c_kv_iq4nl[c];
    } else if constexpr (KIND == Q4_1 || KIND == Q5_1) {
        constexpr int QS = (KIND == Q5_1) ? 8 : 4;
        const uint32_t byte = b[QS + (i & 15)];
        int q = (i < 16) ? (byte & 15) : (byte >> 4);
        if constexpr (KIND == Q5_1) q |= static_cast<int>((b[4 + (i >> 3)] >> (i & 7)) & 1) << 4;
        return __fadd_rn(__fmul_rn(h2f(ld16(b, 0)), static_cast<float>(q)), h2f(ld16(b, 2)));
    } else if constexpr (KIND == Q8_1) {
        return h2f(ld16(b, 0)) * static_cast<float>(static_cast<int8_t>(b[4 + i]));
    } else {  // MXFP4
        static_assert(KIND == MXFP4, "every format has an element decoder");
        const uint32_t byte = b[1 + (i & 15)];
        const int c = (i < 16) ? (byte & 15) : (byte >> 4);
        return e8m0f(b[0]) * c_kv_e2m1[c];
    }
}

// Element e (0 <= e < BE) of the block at b.
template <int KIND>
__device__ __forceinline__ float elem(const uint8_t* b, int e) {
    return elem32<KIND>(b, e >> 5, e & 31);
}

// Elements e .. e + 3 (e a multiple of 4) of the block at b, the same values
// as elem() bit for bit: the four share one scale group (every format's
// groups are 16 or 32 elements), so the scale factors are derived once. The
// codebook formats read their table from `tbl` (16 floats: the IQ4_NL values,
// or E2M1 for MXFP4), a copy the caller keeps in shared memory -- one entry
// per bank, so lanes with different codes never serialize, as they do on a
// per-lane-indexed __constant__ array. Byte loads only (any alignment).
template <int KIND>
__device__ __forceinline__ float4 elem4(const uint8_t* b, int e, const float* tbl) {
    float v[4];
    const int j = e >> 5, i0 = e & 31;
    if constexpr (KIND == Q8_0) {
        const float d = h2f(ld16(b, 0));
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = d * static_cast<float>(static_cast<int8_t>(b[2 + i0 + t]));
    } else if constexpr (KIND == Q4_0 || KIND == IQ4_NL) {
        const float d = h2f(ld16(b, 0));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const uint32_t byte = b[2 + (i & 15)];
            const int c = (i < 16) ? (byte & 15) : (byte >> 4);
            v[t] = (KIND == Q4_0) ? d * static_cast<float>(c - 8) : d * tbl[c];
        }
    } else if constexpr (KIND == Q5_0) {
        const float d = h2f(ld16(b, 0));
        const uint32_t qh = ld8(b, 2) | (ld8(b, 3) << 8) | (ld8(b, 4) << 16) | (ld8(b, 5) << 24);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const uint32_t byte = b[6 + (i & 15)];
            const int lo = static_cast<int>((i < 16) ? (byte & 15) : (byte >> 4));
            const int q = lo | static_cast<int>(((qh >> i) & 1u) << 4);   // signed: q - 16 may be negative
            v[t] = d * static_cast<float>(q - 16);
        }
    } else if constexpr (KIND == Q4_K || KIND == Q5_K) {
        int sc, mn;
        k4_sm(b + 4, j, sc, mn);
        const float ds = h2f(ld16(b, 0)) * static_cast<float>(sc);
        const float dm = h2f(ld16(b, 2)) * static_cast<float>(mn);
        const int qs = (KIND == Q4_K) ? 16 : 48;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const uint32_t byte = b[qs + (j >> 1) * 32 + i];
            int q = (j & 1) ? (byte >> 4) : (byte & 15);
            if constexpr (KIND == Q5_K) q += ((b[16 + i] >> j) & 1) << 4;
            v[t] = __fsub_rn(__fmul_rn(ds, static_cast<float>(q)), dm);
        }
    } else if constexpr (KIND == Q6_K) {
        const int h = j >> 2, g = j & 3;
        const float ds = h2f(ld16(b, 208)) * static_cast<float>(static_cast<int8_t>(b[192 + 2 * j + (i0 >> 4)]));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const uint32_t lob = b[h * 64 + i + (g & 1) * 32];
            const int lo = (g >= 2) ? (lob >> 4) : (lob & 15);
            const int hi = (b[128 + h * 32 + i] >> (2 * g)) & 3;
            v[t] = ds * static_cast<float>((lo | (hi << 4)) - 32);
        }
    } else if constexpr (KIND == Q2_K) {
        const int h = j >> 2, g = j & 3;
        const int s = b[2 * j + (i0 >> 4)];
        const float dl = h2f(ld16(b, 80)) * static_cast<float>(s & 15);
        const float ml = h2f(ld16(b, 82)) * static_cast<float>(s >> 4);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int q = (b[16 + h * 32 + i0 + t] >> (2 * g)) & 3;
            v[t] = __fsub_rn(__fmul_rn(dl, static_cast<float>(q)), ml);
        }
    } else if constexpr (KIND == Q3_K) {
        const int h = j >> 2, g = j & 3;
        const float ds = h2f(ld16(b, 108)) * static_cast<float>(q3_scale(b + 96, 2 * j + (i0 >> 4)) - 32);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const int q2 = (b[32 + h * 32 + i] >> (2 * g)) & 3;
            v[t] = ds * static_cast<float>(q2 - (((b[i] >> j) & 1) ? 0 : 4));
        }
    } else if constexpr (KIND == IQ4_XS) {
        const uint32_t sh = ld16(b, 2);
        const int ls = ((b[4 + (j >> 1)] >> (4 * (j & 1))) & 15) | (((sh >> (2 * j)) & 3) << 4);
        const float ds = h2f(ld16(b, 0)) * static_cast<float>(ls - 32);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const uint32_t byte = b[8 + 16 * j + (i & 15)];
            v[t] = ds * tbl[(i < 16) ? (byte & 15) : (byte >> 4)];
        }
    } else if constexpr (KIND == Q4_1 || KIND == Q5_1) {
        constexpr int QS = (KIND == Q5_1) ? 8 : 4;
        const float d = h2f(ld16(b, 0)), m = h2f(ld16(b, 2));
        const uint32_t qh = (KIND == Q5_1) ? (ld8(b, 4) | (ld8(b, 5) << 8) | (ld8(b, 6) << 16) | (ld8(b, 7) << 24)) : 0u;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const uint32_t byte = b[QS + (i & 15)];
            const uint32_t q = ((i < 16) ? (byte & 15) : (byte >> 4)) | (((qh >> i) & 1u) << 4);
            v[t] = __fadd_rn(__fmul_rn(d, static_cast<float>(q)), m);
        }
    } else if constexpr (KIND == Q8_1) {
        const float d = h2f(ld16(b, 0));
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = d * static_cast<float>(static_cast<int8_t>(b[4 + i0 + t]));
    } else {  // MXFP4
        static_assert(KIND == MXFP4, "every format has an element decoder");
        const float s = e8m0f(b[0]);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const uint32_t byte = b[1 + (i & 15)];
            v[t] = s * tbl[(i < 16) ? (byte & 15) : (byte >> 4)];
        }
    }
    return make_float4(v[0], v[1], v[2], v[3]);
}

// The 16-entry table elem4 reads for a format (nullptr-safe for the others).
template <int KIND>
__device__ __forceinline__ float codebook_entry(int c) {
    return KIND == MXFP4 ? c_kv_e2m1[c] : c_kv_iq4nl[c];
}


// ---------------------------------------------------------------------------
// Tensor-core operand decoding: integer codes (times integer sub-scales) and
// the fp32 scales that multiply the partial sums.
//
//   format  code (exact in f16 unless noted)        scale on partial sums
//   Q8_0    q                                        d        per 32
//   Q4_0    q - 8                                    d        per 32
//   Q5_0    q - 16                                   d        per 32
//   IQ4_NL  KV[c]                                    d        per 32
//   MXFP4   E2M1[c] * 2^(e - e_max)  (exact while e_max - e <= 23)  2^(e_max-127) per 256
//   Q8_1    q                                        d        per 32
//   Q4_1    q                                        d        per 32;   mins: m (an f16)
//   Q5_1    q                                        d        per 32;   mins: m (an f16)
//   Q4_K    sc_j * q            (<= 945)             d per 256;  mins: dmin * m_j
//   Q5_K    sc_j * q            (<= 1953)            d per 256;  mins: dmin * m_j
//   Q6_K    sc * (q - 32)       (<= 4096; rounds once above 2048)   d per 256
//   Q2_K    (s & 15) * q        (<= 45)              d per 256;  mins: dmin * (s >> 4)
//   Q3_K    (sc - 32) * q       (<= 128)             d per 256
//   IQ4_XS  (ls - 32) * KV[c]   (<= 4064; rounds once above 2048)   d per 256
// ---------------------------------------------------------------------------
template <int KIND> struct TcGeo {
    // scale per 32-element block (MXFP4 folds its block exponents into the
    // operands and keeps one power of two per 256 elements instead)
    static constexpr bool PER32 = Geo<KIND>::BE == 32 && KIND != MXFP4;
    static constexpr bool MINS = KIND == Q4_K || KIND == Q5_K || KIND == Q2_K || KIND == Q4_1 || KIND == Q5_1;
    static constexpr int MIN_GROUPS = KIND == Q2_K ? 16 : 8;                 // min groups per 256
};

// The codes themselves are produced per sub-step, in registers, by the fast
// decoders of tc_fastdec.cuh.

// fp32 scale of a 32-element block (PER32 formats).
template <int KIND>
__device__ __forceinline__ float scale32(const uint8_t* b) {
    static_assert(TcGeo<KIND>::PER32, "per-32 formats: an f16 scale at byte 0");
    return h2f(ld16(b, 0));
}

// Super-block d and dmin (PER32 == false).
template <int KIND>
__device__ __forceinline__ float2 scale256(const uint8_t* b) {
    if constexpr (KIND == Q4_K || KIND == Q5_K) return make_float2(h2f(ld16(b, 0)), h2f(ld16(b, 2)));
    else if constexpr (KIND == Q6_K) return make_float2(h2f(ld16(b, 208)), 0.f);
    else if constexpr (KIND == Q2_K) return make_float2(h2f(ld16(b, 80)), h2f(ld16(b, 82)));
    else if constexpr (KIND == Q3_K) return make_float2(h2f(ld16(b, 108)), 0.f);
    else if constexpr (KIND == MXFP4) {
        // the largest of the eight block exponents: 2^(e_max - 127)
        uint32_t e = 0;
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) e = max(e, static_cast<uint32_t>(b[17 * blk]));
        return make_float2(e8m0f(e), 0.f);
    } else return make_float2(h2f(ld16(b, 0)), 0.f);  // IQ4_XS
}

// Runtime kind -> template dispatch helper for the streaming GEMV, which also
// reads the repacked layouts.
#define QMM_DISPATCH_GEMV_KIND(kind, FN, ...)                     \
    switch (kind) {                                               \
    case ::qmm::Q8_0R: FN<::qmm::Q8_0R>(__VA_ARGS__); break;      \
    case ::qmm::Q4_0R: FN<::qmm::Q4_0R>(__VA_ARGS__); break;      \
    default: QMM_DISPATCH_KIND(kind, FN, __VA_ARGS__);            \
    }

// Runtime kind -> template dispatch helper.
#define QMM_DISPATCH_KIND(kind, FN, ...)                          \
    switch (kind) {                                               \
    case ::qmm::Q8_0: FN<::qmm::Q8_0>(__VA_ARGS__); break;        \
    case ::qmm::Q4_0: FN<::qmm::Q4_0>(__VA_ARGS__); break;        \
    case ::qmm::Q5_0: FN<::qmm::Q5_0>(__VA_ARGS__); break;        \
    case ::qmm::Q4_K: FN<::qmm::Q4_K>(__VA_ARGS__); break;        \
    case ::qmm::Q5_K: FN<::qmm::Q5_K>(__VA_ARGS__); break;        \
    case ::qmm::Q6_K: FN<::qmm::Q6_K>(__VA_ARGS__); break;        \
    case ::qmm::Q2_K: FN<::qmm::Q2_K>(__VA_ARGS__); break;        \
    case ::qmm::Q3_K: FN<::qmm::Q3_K>(__VA_ARGS__); break;        \
    case ::qmm::IQ4_NL: FN<::qmm::IQ4_NL>(__VA_ARGS__); break;    \
    case ::qmm::IQ4_XS: FN<::qmm::IQ4_XS>(__VA_ARGS__); break;    \
    case ::qmm::Q4_1: FN<::qmm::Q4_1>(__VA_ARGS__); break;        \
    case ::qmm::Q5_1: FN<::qmm::Q5_1>(__VA_ARGS__); break;        \
    case ::qmm::Q8_1: FN<::qmm::Q8_1>(__VA_ARGS__); break;        \
    default: FN<::qmm::MXFP4>(__VA_ARGS__); break;                \
    }

}  // namespace qmm
