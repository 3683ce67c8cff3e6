// k_gemv.cu -- weight-streaming quantized GEMV for small N (decode), plain and
// expert-grouped.
//
// y[n, m] = sum_k W[m, k] * x[n, k] for up to 8 activation rows, and the
// expert-indexed form where output row r reads expert expert_id[r]'s weights
// and activation row x_row[r]. A decode-time GEMV spends its time reading the
// weights from HBM, once (the `Q4_GEMV_KERNEL` notes of inferencelayer 0.2.8
// src/cublas_prefill.rs make the same point), so the design is about bytes in
// flight, coalescing and a lean decode:
//
//   * Work items are groups of 32 weight rows (one row per lane) of one
//     "problem": the plain product is one problem; the grouped product has one
//     problem per (expert, block of up to NCMAX <= 4 assignments of that
//     expert), so an expert's rows stream from HBM once per block of its
//     tokens (once for most experts), not once per token. Each CTA
//     (persistent, one per SM) takes a contiguous, equal share of the items.
//   * One producer thread moves K-chunks of an item's 32 rows from HBM into a
//     ring of shared-memory stages, one TMA tensor copy per stage
//     (`cp.async.bulk.tensor.3d`, completing on an mbarrier, L2 evict-first).
//     The tensor map sees the weights as (8-byte word of the row, row,
//     expert); the box takes an odd number of 16-byte granules per row (the
//     chunk, plus one slack granule when the chunk's count is even), so staged
//     rows sit an odd number of 16-byte words apart and the 32 lanes reading
//     32 rows hit distinct banks, while each box row is one contiguous run in
//     memory (a 16-byte innermost box dimension would cost one L2 request per
//     16 bytes). Rows past M and words past the row end read as zeros. One
//     copy per stage (not one per row) keeps the copy engine's per-request
//     cost off the critical path, so stages can be small and consumption
//     starts as soon as the first one lands.
//   * The consumer warps form G groups of NWU warps; group g consumes chunks
//     g, g + G, g + 2G, ... of the CTA's chunk stream, warp u of the group the
//     u-th unit of each (lane = row, 16-byte shared loads, row stride padded to
//     an odd number of 16-byte words so the 32 lanes hit distinct banks;
//     activations by broadcast loads). Per-row partial sums of all warps are
//     added through shared memory at the end of each item.
//   * Activations are staged once per problem, by the consumers, in a
//     per-format layout. Q4_0: each nibble is OR-ed into the mantissa of
//     128.0f at the bit position it already has in its 32-bit word (no shifts
//     but one per word), which gives exactly 128 + q * 2^p; one packed subtract
//     leaves exactly (q - 8) * 2^p, and the activation is staged pre-multiplied
//     by 2^-p, so every product is the exact (q - 8) * x. Q8_0: the code byte
//     XOR 0x80 in the low byte under 2^23 gives 2^23 + q + 128 exactly, one
//     packed subtract leaves q. Both multiply with packed fp32x2 FMAs; the fp32
//     block scale multiplies the block's partial sum.
//   * Programmatic dependent launch: the kernel lets the next one on the stream
//     launch at once. When the caller declares the weights constant
//     (QMM_FLAG_WEIGHTS_CONST), each CTA
//     of the next GEMV streams its first weight stages as soon as it is
//     resident -- beside this kernel's CTAs when the stage ring fits two CTAs
//     per SM, else as this kernel's CTAs retire -- while this one drains.
//     Activations and expert ids are read only after `griddepcontrol.wait`.
//
// The P4 page's v3 lesson (stage x in shared memory, keep lanes on distinct
// banks, keep loads in flight) is kept; its f16x2 accumulation is not (too
// lossy for the 1e-3 relative bar over K = 4096), nor its structure-of-arrays
// layout. Every wait is bounded; a timeout latches DEV_ERR_TIMEOUT and the
// CTA unwinds.
#include <cstdlib>

#include <cuda_fp16.h>

#include "decode.cuh"
#include "qmm.h"
#include "qmm_internal.cuh"
#include "sm100_async.cuh"
#include "tc_fastdec.cuh"

namespace qmm {
namespace {

constexpr int kRows = 32;
constexpr int kMaxStages = 16;
constexpr int kCoresident = 112 * 1024;   // two CTAs (this kernel and the next) fit on one SM
constexpr int kSmemBudget = 224 * 1024;
constexpr int kMaxGroupedExperts = 1024;
constexpr int kMaxGroupedAssign = 4096;

// Per format: blocks per warp unit (UB), consumer warps (NW) and preferred
// warps per chunk (NWU). A unit is a multiple of 16 bytes where the format
// allows it. Measured on the decode workload (M = 14336, K = 4096): Q8_0 runs
// best with 1088-byte chunks (4 warps of 8), Q4_0 with 1152-byte chunks (8
// warps of 16; its decode needs the extra warps).
template <int KIND> struct SG;
template <> struct SG<Q8_0>   { static constexpr int UB = 8,  NW = 8,  NWU = 4; };
template <> struct SG<Q4_0>   { static constexpr int UB = 8,  NW = 16, NWU = 8; };
template <> struct SG<Q5_0>   { static constexpr int UB = 8,  NW = 8,  NWU = 2; };
template <> struct SG<IQ4_NL> { static constexpr int UB = 8,  NW = 8,  NWU = 2; };
template <> struct SG<MXFP4>  { static constexpr int UB = 16, NW = 8,  NWU = 2; };
template <> struct SG<Q4_K>   { static constexpr int UB = 1,  NW = 8,  NWU = 4; };
template <> struct SG<Q5_K>   { static constexpr int UB = 1,  NW = 8,  NWU = 4; };
template <> struct SG<Q6_K>   { static constexpr int UB = 1,  NW = 8,  NWU = 4; };
template <> struct SG<Q2_K>   { static constexpr int UB = 1,  NW = 8,  NWU = 4; };
template <> struct SG<Q3_K>   { static constexpr int UB = 1,  NW = 8,  NWU = 4; };
template <> struct SG<IQ4_XS> { static constexpr int UB = 1,  NW = 8,  NWU = 4; };
template <> struct SG<Q4_1>   { static constexpr int UB = 8,  NW = 8,  NWU = 2; };
template <> struct SG<Q5_1>   { static constexpr int UB = 8,  NW = 8,  NWU = 2; };
template <> struct SG<Q8_1>   { static constexpr int UB = 8,  NW = 8,  NWU = 4; };
template <> struct SG<Q8_0R>  { static constexpr int UB = 8,  NW = 8,  NWU = 4; };
template <> struct SG<Q4_0R>  { static constexpr int UB = 8,  NW = 16, NWU = 8; };

template <int KIND> struct SGeo {
    static constexpr int NW = SG<KIND>::NW;
    static constexpr int UNIT_B = SG<KIND>::UB * Geo<KIND>::BB;
    static constexpr int UNIT_E = SG<KIND>::UB * Geo<KIND>::BE;
};

struct GemvArgs {
    const uint8_t* W;
    size_t row_bytes;
    int64_t M;
    int K;
    const void* X;
    int x_dtype;
    float* Y;
    int y_dtype;              // 0 fp32, 1 f16, 2 bf16
    int x_mode;               // 0 plain rows, 1 SwiGLU of gate_up rows (see Problem)
    int64_t x_stride;         // elements per activation row
    int ncols;                // plain: N
    // grouped (x_row == nullptr for the plain product)
    const int32_t* x_row;
    const int32_t* expert_id;
    size_t expert_stride;
    int n_experts;
    int n_assign;
    int64_t n_x_rows;
    // pipeline
    int stages;
    int nwu;                  // warps per chunk
    int stride;               // shared bytes per staged row: box granules * 16 (odd multiple of 16)
    int upr;                  // units per row
    int cpr;                  // chunks per row
    int flags;
    unsigned* err;
};

constexpr int kFlagPrefetchW = 1;  // weights may be read before the previous grid completes

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 3-D tiled TMA load (coordinates innermost first), completing on `bar`, with
// an L2 cache policy.
__device__ __forceinline__ void tma3d(void* dst, const CUtensorMap* tm, int c0, int c1, int c2, uint64_t* bar,
                                      uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// (a & b) | c in one LOP3, all operands in registers.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------------------
// unit decoders: acc[n] += sum over the unit's elements of W * x[n]
// ---------------------------------------------------------------------------

// Q4_0 staged-activation order. The decoder walks four 32-bit words of code
// bytes per block. Odd blocks start 4-byte aligned at their codes (word j =
// code bytes 4j..4j+3); even blocks start 2 bytes off, so their word 0 is
// (c14, c15, c0, c1) and word j >= 1 holds code bytes 4j-2..4j+1. Nibble i of a
// word (bits 4i..4i+3; i = 2 * byte + high) feeds slot 8j + i.
__host__ __device__ __forceinline__ int q4_slot(int e, bool even) {
    const int hi = e >> 4, c = e & 15;       // nibble half, code byte
    int j, k;                                // word, byte within word
    if (!even) {
        j = c >> 2;
        k = c & 3;
    } else if (c >= 14) {
        j = 0;
        k = c - 14;
    } else if (c < 2) {
        j = 0;
        k = c + 2;
    } else {
        j = (c + 2) >> 2;
        k = (c + 2) & 3;
    }
    return 8 * j + 2 * k + hi;
}

// Nibble i of a word is OR-ed into 128.0f at mantissa bits 4i..4i+3 (i <= 4)
// or, from the word shifted right by 12, at bits 4(i-3)..4(i-3)+3 (i >= 5):
// its weight there is 2^(4i-16) resp. 2^(4(i-3)-16). The activation staged for
// that slot is multiplied by the inverse power of two (exact).
__host__ __device__ __forceinline__ int q4_pow(int i) {
    return (i <= 4) ? 4 * i - 16 : 4 * (i - 3) - 16;
}

// Formats whose minimum term needs the activation sums of each 16-element group.
template <int KIND> struct XSum {
    static constexpr bool ON = KIND == Q4_K || KIND == Q5_K || KIND == Q2_K || KIND == Q4_1 || KIND == Q5_1;
};

// Codebook formats (IQ4_NL, IQ4_XS, MXFP4) stage the activations of each
// 32-element group in the order their decoder meets the elements: a code word
// holds elements 4w .. 4w + 3 in its low nibbles and 16 + 4w .. in its high
// nibbles, and the register table lookup returns them interleaved, element
// 16 h + 4 w + j at slot 8 w + 2 j + h.
__host__ __device__ __forceinline__ int cb_slot(int e) { return 8 * ((e >> 2) & 3) + 2 * (e & 3) + (e >> 4); }
template <int KIND> struct CbOrder { static constexpr bool ON = KIND == IQ4_NL || KIND == IQ4_XS || KIND == MXFP4; };

// Q4_0, one activation column: 8 blocks of 18 bytes (144 B, 16-byte aligned
// in shared memory), fully unrolled (the fastest form for a single column).
template <int NC>
__device__ __forceinline__ void unit_q4_0_flat(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(u)[i];
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    const uint32_t mask[5] = {0xFu, 0xF0u, 0xF00u, 0xF000u, 0xF0000u};
    const uint32_t kMagic = 0x43000000u;   // 128.0f
    // 128 + 8 * 2^p for the four nibble pairs (0,1) (2,3) (4,5) (6,7)
    const float2 bias0 = make_float2(128.f + 8.f * 0x1p-16f, 128.f + 8.f * 0x1p-12f);
    const float2 bias1 = make_float2(128.f + 8.f * 0x1p-8f, 128.f + 8.f * 0x1p-4f);
    const float2 bias2 = make_float2(136.f, 128.f + 8.f * 0x1p-8f);
    const float2 bias3 = make_float2(128.f + 8.f * 0x1p-4f, 136.f);
#pragma unroll
    for (int blk = 0; blk < 8; ++blk) {
        const int o = 18 * blk, a = o >> 2;
        const bool even = (o & 3) == 0;
        const float d = h2f(even ? w[a] : (w[a] >> 16));
        uint32_t words[4];
        if (even) {
            words[0] = __byte_perm(w[a], w[a + 4], 0x3254);
            words[1] = w[a + 1];
            words[2] = w[a + 2];
            words[3] = w[a + 3];
        } else {
            words[0] = w[a + 1];
            words[1] = w[a + 2];
            words[2] = w[a + 3];
            words[3] = w[a + 4];
        }
        const int kb = k0 + 32 * blk;
        float2 S[NC][2];
#pragma unroll
        for (int n = 0; n < NC; ++n) S[n][0] = S[n][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t v = words[j], sh = v >> 12;
            const float2 f01 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[0], kMagic)),
                                                      __uint_as_float(and_or(v, mask[1], kMagic))),
                                          make_float2(-bias0.x, -bias0.y));
            const float2 f23 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[2], kMagic)),
                                                      __uint_as_float(and_or(v, mask[3], kMagic))),
                                          make_float2(-bias1.x, -bias1.y));
            const float2 f45 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[4], kMagic)),
                                                      __uint_as_float(and_or(sh, mask[2], kMagic))),
                                          make_float2(-bias2.x, -bias2.y));
            const float2 f67 = __fadd2_rn(make_float2(__uint_as_float(and_or(sh, mask[3], kMagic)),
                                                      __uint_as_float(and_or(sh, mask[4], kMagic))),
                                          make_float2(-bias3.x, -bias3.y));
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float4 xl = *reinterpret_cast<const float4*>(xs + n * K + kb + 8 * j);
                const float4 xh = *reinterpret_cast<const float4*>(xs + n * K + kb + 8 * j + 4);
                S[n][0] = __ffma2_rn(f01, make_float2(xl.x, xl.y), S[n][0]);
                S[n][1] = __ffma2_rn(f23, make_float2(xl.z, xl.w), S[n][1]);
                S[n][0] = __ffma2_rn(f45, make_float2(xh.x, xh.y), S[n][0]);
                S[n][1] = __ffma2_rn(f67, make_float2(xh.z, xh.w), S[n][1]);
            }
        }
#pragma unroll
        for (int n = 0; n < NC; ++n) {
            const float2 t2 = __fadd2_rn(S[n][0], S[n][1]);
            acc[n] = fmaf(d, t2.x + t2.y, acc[n]);
        }
    }
}

// Q4_0, several activation columns: the same arithmetic, walked as four pairs
// of blocks with a rolled loop -- a pair is 36 bytes starting 4-byte aligned
// (nine 32-bit loads) -- which keeps the multi-column decoder small enough for
// the instruction cache.
template <int NC>
__device__ __forceinline__ void unit_q4_0(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    const uint32_t mask[5] = {0xFu, 0xF0u, 0xF00u, 0xF000u, 0xF0000u};
    const uint32_t kMagic = 0x43000000u;   // 128.0f
    // 128 + 8 * 2^p for the four nibble pairs (0,1) (2,3) (4,5) (6,7)
    const float2 nb0 = make_float2(-(128.f + 8.f * 0x1p-16f), -(128.f + 8.f * 0x1p-12f));
    const float2 nb1 = make_float2(-(128.f + 8.f * 0x1p-8f), -(128.f + 8.f * 0x1p-4f));
    const float2 nb2 = make_float2(-136.f, -(128.f + 8.f * 0x1p-8f));
    const float2 nb3 = make_float2(-(128.f + 8.f * 0x1p-4f), -136.f);
#pragma unroll 1
    for (int pr = 0; pr < 4; ++pr) {
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(u + 36 * pr);
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = pw[i];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // block 2pr (h = 0) starts at the pair's first byte: d in the low
            // half of word 0, codes 0..1 in its high half, 14..15 in word 4;
            // block 2pr + 1 (h = 1) has d in the high half of word 4 and its
            // codes in words 5..8
            const float d = h2f(h ? (w[4] >> 16) : w[0]);
            uint32_t words[4];
            if (h == 0) {
                words[0] = __byte_perm(w[0], w[4], 0x3254);
                words[1] = w[1];
                words[2] = w[2];
                words[3] = w[3];
            } else {
                words[0] = w[5];
                words[1] = w[6];
                words[2] = w[7];
                words[3] = w[8];
            }
            const int kb = k0 + 32 * (2 * pr + h);
            float2 S[NC][2];
#pragma unroll
            for (int n = 0; n < NC; ++n) S[n][0] = S[n][1] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t v = words[j], sh = v >> 12;
                const float2 f01 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[0], kMagic)),
                                                          __uint_as_float(and_or(v, mask[1], kMagic))), nb0);
                const float2 f23 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[2], kMagic)),
                                                          __uint_as_float(and_or(v, mask[3], kMagic))), nb1);
                const float2 f45 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[4], kMagic)),
                                                          __uint_as_float(and_or(sh, mask[2], kMagic))), nb2);
                const float2 f67 = __fadd2_rn(make_float2(__uint_as_float(and_or(sh, mask[3], kMagic)),
                                                          __uint_as_float(and_or(sh, mask[4], kMagic))), nb3);
#pragma unroll
                for (int n = 0; n < NC; ++n) {
                    const float4 xl = *reinterpret_cast<const float4*>(xs + n * K + kb + 8 * j);
                    const float4 xh = *reinterpret_cast<const float4*>(xs + n * K + kb + 8 * j + 4);
                    S[n][0] = __ffma2_rn(f01, make_float2(xl.x, xl.y), S[n][0]);
                    S[n][1] = __ffma2_rn(f23, make_float2(xl.z, xl.w), S[n][1]);
                    S[n][0] = __ffma2_rn(f45, make_float2(xh.x, xh.y), S[n][0]);
                    S[n][1] = __ffma2_rn(f67, make_float2(xh.z, xh.w), S[n][1]);
                }
            }
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float2 t2 = __fadd2_rn(S[n][0], S[n][1]);
                acc[n] = fmaf(d, t2.x + t2.y, acc[n]);
            }
        }
    }
}

// Q8_0: 8 blocks of 34 bytes (272 B). Code byte c (two's complement) XOR 0x80
// is c + 128; placed in the low byte under 0x4B000000 it reads 2^23 + c + 128,
// and one packed subtract of (2^23 + 128) leaves c exactly.
template <int NC>
__device__ __forceinline__ void unit_q8_0(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    uint32_t w[68];
#pragma unroll
    for (int i = 0; i < 17; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(u)[i];
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    const float2 off = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
#pragma unroll
    for (int blk = 0; blk < 8; ++blk) {
        const int o = 34 * blk;
        const uint32_t dw = w[o >> 2];
        const float d = h2f((o & 3) ? (dw >> 16) : dw);
        const int kb = k0 + 32 * blk;
        float2 S[NC][2];
#pragma unroll
        for (int n = 0; n < NC; ++n) S[n][0] = S[n][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            float4 xv[NC];
#pragma unroll
            for (int n = 0; n < NC; ++n) xv[n] = *reinterpret_cast<const float4*>(xs + n * K + kb + i);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int b0 = o + 2 + i + 2 * h, b1 = b0 + 1;
                const float f0 = __int_as_float(static_cast<int>(
                    __byte_perm(w[b0 >> 2] ^ 0x80808080u, 0x4B000000u, 0x7650u | static_cast<unsigned>(b0 & 3))));
                const float f1 = __int_as_float(static_cast<int>(
                    __byte_perm(w[b1 >> 2] ^ 0x80808080u, 0x4B000000u, 0x7650u | static_cast<unsigned>(b1 & 3))));
                const float2 q = __fadd2_rn(make_float2(f0, f1), off);
#pragma unroll
                for (int n = 0; n < NC; ++n) {
                    const float2 xp = h ? make_float2(xv[n].z, xv[n].w) : make_float2(xv[n].x, xv[n].y);
                    S[n][h] = __ffma2_rn(q, xp, S[n][h]);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < NC; ++n) {
            const float2 t2 = __fadd2_rn(S[n][0], S[n][1]);
            acc[n] = fmaf(d, t2.x + t2.y, acc[n]);
        }
    }
}

// ---------------------------------------------------------------------------
// Byte-code decoders for the other formats. A word of four code bytes c_k
// (unsigned, biased) becomes four exact fp32 values: byte k placed under the
// exponent of 2^23 (one byte permute) reads 2^23 + c_k, and one packed
// subtract of 2^23 + bias leaves c_k - bias exactly. Packed FMAs then add
// (c_k - bias) * x_k into per-group partial sums, which the group's fp32 scale
// multiplies afterwards (the minimum term of Q4_K / Q5_K / Q2_K / Q4_1 / Q5_1 multiplies
// the group's activation sum). Codebooks are looked up four nibbles at a time
// in registers (byte permutes, see lut16), never in memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 nbias(float bias) { return make_float2(-(8388608.f + bias), -(8388608.f + bias)); }

// s[n] += sum_k (byte k of w + nb) * x[n * K + k], k = 0..3 (x 16-byte aligned)
template <int NC>
__device__ __forceinline__ void dot4(uint32_t w, float2 nb, const float* x, int K, float2 (&s)[NC]) {
    const float2 q01 = __fadd2_rn(make_float2(__uint_as_float(prmt(w, 0x4B000000u, 0x7540u)),
                                              __uint_as_float(prmt(w, 0x4B000000u, 0x7541u))), nb);
    const float2 q23 = __fadd2_rn(make_float2(__uint_as_float(prmt(w, 0x4B000000u, 0x7542u)),
                                              __uint_as_float(prmt(w, 0x4B000000u, 0x7543u))), nb);
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        const float4 xv = *reinterpret_cast<const float4*>(x + n * K);
        s[n] = __ffma2_rn(q01, make_float2(xv.x, xv.y), s[n]);
        s[n] = __ffma2_rn(q23, make_float2(xv.z, xv.w), s[n]);
    }
}

template <int NC>
__device__ __forceinline__ void zero2(float2 (&s)[NC]) {
#pragma unroll
    for (int n = 0; n < NC; ++n) s[n] = make_float2(0.f, 0.f);
}

// the four bits v (bits 0..3) moved to bit 4 of bytes 0..3
__device__ __forceinline__ uint32_t bit4_to_bytes(uint32_t v) { return ((v * 0x00204081u) & 0x01010101u) << 4; }

// Q5_0: pairs of 22-byte blocks (44 bytes, 4-byte aligned in the unit).
template <int NC>
__device__ __forceinline__ void unit_q5_0(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    const float2 nb = nbias(16.f);
#pragma unroll 1
    for (int pr = 0; pr < 4; ++pr) {
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(u + 44 * pr);
        uint32_t w[11];
#pragma unroll
        for (int i = 0; i < 11; ++i) w[i] = pw[i];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            // block 2pr: d at bytes 0-1, qh 2-5, codes 6-21; block 2pr + 1: d 22-23, qh 24-27, codes 28-43
            const float d = h2f(hb ? (w[5] >> 16) : w[0]);
            const uint32_t qh = hb ? w[6] : __funnelshift_r(w[0], w[1], 16);
            const int kb = k0 + 32 * (2 * pr + hb);
            float2 S[NC];
            zero2(S);
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const uint32_t q = hb ? w[7 + wi] : __funnelshift_r(w[1 + wi], w[2 + wi], 16);
                const uint32_t lo = (q & 0x0F0F0F0Fu) | bit4_to_bytes((qh >> (4 * wi)) & 0xFu);
                const uint32_t hi = ((q >> 4) & 0x0F0F0F0Fu) | bit4_to_bytes((qh >> (16 + 4 * wi)) & 0xFu);
                dot4<NC>(lo, nb, xs + kb + 4 * wi, K, S);
                dot4<NC>(hi, nb, xs + kb + 16 + 4 * wi, K, S);
            }
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[n] = fmaf(d, S[n].x + S[n].y, acc[n]);
        }
    }
}

// Q4_1 (20 B), Q5_1 (24 B) and Q8_1 (36 B) keep every field 4-byte aligned:
// four blocks are 80 / 96 / 144 bytes, whole 16-byte vectors from the
// 16-byte aligned unit. Block scale d on the partial sum; Q4_1 / Q5_1 add
// their f16 min times the block's activation sum (two per-16 sums).
template <int KIND, int NC>
__device__ __forceinline__ void unit_legacy1(const uint8_t* u, const float* xs, const float* xsum, int K, int k0,
                                             float (&acc)[NC]) {
    constexpr int BW = Geo<KIND>::BB / 4;   // words per block: 5, 6 or 9
    const float2 nb = nbias(KIND == Q8_1 ? 128.f : 0.f);
#pragma unroll 1
    for (int qd = 0; qd < 2; ++qd) {
        uint32_t w[4 * BW];
#pragma unroll
        for (int i = 0; i < BW; ++i) {
            const uint4 v = reinterpret_cast<const uint4*>(u + 16 * BW * qd)[i];
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int bi = 0; bi < 4; ++bi) {
            const uint32_t* bw = w + BW * bi;
            const float d = h2f(bw[0]);
            const int kb = k0 + 32 * (4 * qd + bi);
            float2 S[NC];
            zero2(S);
            if constexpr (KIND == Q8_1) {
#pragma unroll
                for (int wi = 0; wi < 8; ++wi) dot4<NC>(bw[1 + wi] ^ 0x80808080u, nb, xs + kb + 4 * wi, K, S);
            } else {
                constexpr int QS = (KIND == Q5_1) ? 2 : 1;   // first code word
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    uint32_t lo = bw[QS + wi] & 0x0F0F0F0Fu, hi = (bw[QS + wi] >> 4) & 0x0F0F0F0Fu;
                    if constexpr (KIND == Q5_1) {
                        lo |= bit4_to_bytes((bw[1] >> (4 * wi)) & 0xFu);
                        hi |= bit4_to_bytes((bw[1] >> (16 + 4 * wi)) & 0xFu);
                    }
                    dot4<NC>(lo, nb, xs + kb + 4 * wi, K, S);
                    dot4<NC>(hi, nb, xs + kb + 16 + 4 * wi, K, S);
                }
            }
            if constexpr (KIND == Q8_1) {
#pragma unroll
                for (int n = 0; n < NC; ++n) acc[n] = fmaf(d, S[n].x + S[n].y, acc[n]);
            } else {
                const float m = h2f(bw[0] >> 16);
#pragma unroll
                for (int n = 0; n < NC; ++n) {
                    const float* xsn = xsum + n * (K >> 4) + (kb >> 4);
                    acc[n] = fmaf(m, xsn[0] + xsn[1], fmaf(d, S[n].x + S[n].y, acc[n]));
                }
            }
        }
    }
}

// One 32-element codebook group from its four code words (activations in
// codebook order, see cb_slot); table T biased by +128.
template <typename T, int NC>
__device__ __forceinline__ void cb_group(const uint32_t (&q)[4], const float* x, int K, float2 (&S)[NC]) {
    const float2 nb = nbias(128.f);
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        dot4<NC>(lut16<T>(q[wi]), nb, x + 8 * wi, K, S);
        dot4<NC>(lut16<T>(q[wi] >> 16), nb, x + 8 * wi + 4, K, S);
    }
}

// IQ4_NL: pairs of 18-byte blocks, as Q4_0.
template <int NC>
__device__ __forceinline__ void unit_iq4nl(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
#pragma unroll 1
    for (int pr = 0; pr < 4; ++pr) {
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(u + 36 * pr);
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = pw[i];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            const float d = h2f(hb ? (w[4] >> 16) : w[0]);
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = hb ? w[5 + i] : __funnelshift_r(w[i], w[i + 1], 16);
            float2 S[NC];
            zero2(S);
            cb_group<KvTable, NC>(q, xs + k0 + 32 * (2 * pr + hb), K, S);
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[n] = fmaf(d, S[n].x + S[n].y, acc[n]);
        }
    }
}

// MXFP4: groups of four 17-byte blocks (68 bytes, 4-byte aligned in the unit).
template <int NC>
__device__ __forceinline__ void unit_mxfp4(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
#pragma unroll 1
    for (int gq = 0; gq < 4; ++gq) {
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(u + 68 * gq);
        uint32_t w[17];
#pragma unroll
        for (int i = 0; i < 17; ++i) w[i] = pw[i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // block j: exponent byte 17 j, codes 17 j + 1 .. 17 j + 16
            const int bo = 17 * j, wo = (bo + 1) >> 2, sh = ((bo + 1) & 3) * 8;
            const uint32_t e = (w[bo >> 2] >> ((bo & 3) * 8)) & 0xFFu;
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = sh ? __funnelshift_r(w[wo + i], w[wo + i + 1], sh) : w[wo + i];
            float2 S[NC];
            zero2(S);
            cb_group<E2m1Table, NC>(q, xs + k0 + 32 * (4 * gq + j), K, S);
            const float sc = e8m0f(e);
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[n] = fmaf(sc, S[n].x + S[n].y, acc[n]);
        }
    }
}

// Q4_K / Q5_K (6-bit scale and min of sub-block j from the 12-byte field,
// held as three words s0 = bytes 0-3, s1 = 4-7, s2 = 8-11).
__device__ __forceinline__ void k4_sm_words(uint32_t s0, uint32_t s1, uint32_t s2, int j, int& sc, int& mn) {
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63;
        mn = (s1 >> (8 * j)) & 63;
    } else {
        const int b = 8 * (j - 4);
        sc = ((s2 >> b) & 15) | (((s0 >> b) >> 6 & 3) << 4);
        mn = ((s2 >> b) >> 4 & 15) | (((s1 >> b) >> 6 & 3) << 4);
    }
}

// Q4_K (144 B, 16-byte aligned) and Q5_K (176 B, 16-byte aligned): one
// super-block per unit, 64 elements (sub-blocks 2c and 2c + 1) per step.
template <int KIND, int NC>
__device__ __forceinline__ void unit_k45(const uint8_t* u, const float* xs, const float* xsum, int K, int k0,
                                         float (&acc)[NC]) {
    const uint4 h = *reinterpret_cast<const uint4*>(u);
    const float d = h2f(h.x), dmin = h2f(h.x >> 16);
    uint32_t qh[8];
    if constexpr (KIND == Q5_K) {
        const uint4 a = *reinterpret_cast<const uint4*>(u + 16), b = *reinterpret_cast<const uint4*>(u + 32);
        qh[0] = a.x; qh[1] = a.y; qh[2] = a.z; qh[3] = a.w;
        qh[4] = b.x; qh[5] = b.y; qh[6] = b.z; qh[7] = b.w;
    }
    constexpr int QS = (KIND == Q4_K) ? 16 : 48;
    const float2 nb = nbias(0.f);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(u + QS + 32 * c);
        const uint4 v1 = *reinterpret_cast<const uint4*>(u + QS + 32 * c + 16);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float2 S0[NC], S1[NC];
        zero2(S0);
        zero2(S1);
        const int kb = k0 + 64 * c;
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            uint32_t lo = w[wi] & 0x0F0F0F0Fu, hi = (w[wi] >> 4) & 0x0F0F0F0Fu;
            if constexpr (KIND == Q5_K) {
                lo |= ((qh[wi] >> (2 * c)) & 0x01010101u) << 4;
                hi |= ((qh[wi] >> (2 * c + 1)) & 0x01010101u) << 4;
            }
            dot4<NC>(lo, nb, xs + kb + 4 * wi, K, S0);
            dot4<NC>(hi, nb, xs + kb + 32 + 4 * wi, K, S1);
        }
        int sc0, m0, sc1, m1;
        k4_sm_words(h.y, h.z, h.w, 2 * c, sc0, m0);
        k4_sm_words(h.y, h.z, h.w, 2 * c + 1, sc1, m1);
        const float a0 = d * static_cast<float>(sc0), b0 = dmin * static_cast<float>(m0);
        const float a1 = d * static_cast<float>(sc1), b1 = dmin * static_cast<float>(m1);
        const int g = kb >> 4;   // first 16-element group of sub-block 2c
#pragma unroll
        for (int n = 0; n < NC; ++n) {
            const float* xsn = xsum + n * (K >> 4) + g;
            float t = fmaf(a0, S0[n].x + S0[n].y, acc[n]);
            t = fmaf(-b0, xsn[0] + xsn[1], t);
            t = fmaf(a1, S1[n].x + S1[n].y, t);
            acc[n] = fmaf(-b1, xsn[2] + xsn[3], t);
        }
    }
}

// Q6_K (210 B, 2-byte aligned): per 128-element half h and low-nibble run p,
// 32 code bytes and the shared 32 bytes of high bits; int8 scale per 16.
template <int NC>
__device__ __forceinline__ void unit_q6k(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    const float d = h2f(ld16(u, 208));
    const float2 nb = nbias(32.f);
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
        uint32_t qw[8];
        ld_words<8, 2>(u + 128 + 32 * h, qw);
#pragma unroll 1
        for (int p = 0; p < 2; ++p) {
            uint32_t w[8];
            ld_words<8, 2>(u + 64 * h + 32 * p, w);
            float2 SL[2][NC], SH[2][NC];   // [16-element half of the run][column]
            zero2(SL[0]);
            zero2(SL[1]);
            zero2(SH[0]);
            zero2(SH[1]);
            const int kl = k0 + 128 * h + 32 * p, kh = kl + 64;   // groups g = p and g = p + 2
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
                const uint32_t lo = (w[wi] & 0x0F0F0F0Fu) | (((qw[wi] >> (2 * p)) << 4) & 0x30303030u);
                const uint32_t hi = ((w[wi] >> 4) & 0x0F0F0F0Fu) | (((qw[wi] >> (2 * p + 4)) << 4) & 0x30303030u);
                dot4<NC>(lo, nb, xs + kl + 4 * wi, K, SL[wi >> 2]);
                dot4<NC>(hi, nb, xs + kh + 4 * wi, K, SH[wi >> 2]);
            }
            // scale index (element / 16): 8 h + 2 g + (l >= 16)
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const float sl = d * static_cast<float>(static_cast<int8_t>(u[192 + 8 * h + 2 * p + t]));
                const float shh = d * static_cast<float>(static_cast<int8_t>(u[192 + 8 * h + 2 * (p + 2) + t]));
#pragma unroll
                for (int n = 0; n < NC; ++n)
                    acc[n] = fmaf(shh, SH[t][n].x + SH[t][n].y, fmaf(sl, SL[t][n].x + SL[t][n].y, acc[n]));
            }
        }
    }
}

// Q2_K (84 B, 4-byte aligned): 2-bit codes, 4-bit scale and min per 16.
template <int NC>
__device__ __forceinline__ void unit_q2k(const uint8_t* u, const float* xs, const float* xsum, int K, int k0,
                                         float (&acc)[NC]) {
    const uint32_t dd = *reinterpret_cast<const uint32_t*>(u + 80);
    const float d = h2f(dd), dmin = h2f(dd >> 16);
    const float2 nb = nbias(0.f);
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = reinterpret_cast<const uint32_t*>(u + 16 + 32 * h)[i];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float2 S[2][NC];
            zero2(S[0]);
            zero2(S[1]);
            const int kb = k0 + 128 * h + 32 * g;
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) dot4<NC>((w[wi] >> (2 * g)) & 0x03030303u, nb, xs + kb + 4 * wi, K, S[wi >> 2]);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int idx = 8 * h + 2 * g + t;
                const uint32_t sb = u[idx];
                const float a = d * static_cast<float>(sb & 15), b = dmin * static_cast<float>(sb >> 4);
#pragma unroll
                for (int n = 0; n < NC; ++n)
                    acc[n] = fmaf(-b, xsum[n * (K >> 4) + ((kb >> 4) + t)], fmaf(a, S[t][n].x + S[t][n].y, acc[n]));
            }
        }
    }
}

// Q3_K (110 B, 2-byte aligned): 2-bit codes plus the hmask bit (clear = -4),
// 6-bit scale minus 32 per 16.
template <int NC>
__device__ __forceinline__ void unit_q3k(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    const float d = h2f(ld16(u, 108));
    const float2 nb = nbias(4.f);
    uint32_t hm[8];
    ld_words<8, 2>(u, hm);
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
        uint32_t w[8];
        ld_words<8, 2>(u + 32 + 32 * h, w);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int j = 4 * h + g;
            float2 S[2][NC];
            zero2(S[0]);
            zero2(S[1]);
            const int kb = k0 + 128 * h + 32 * g;
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
                const uint32_t c = ((w[wi] >> (2 * g)) & 0x03030303u) | (((hm[wi] >> j) & 0x01010101u) << 2);
                dot4<NC>(c, nb, xs + kb + 4 * wi, K, S[wi >> 2]);
            }
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const float a = d * static_cast<float>(q3_scale(u + 96, 2 * j + t) - 32);
#pragma unroll
                for (int n = 0; n < NC; ++n) acc[n] = fmaf(a, S[t][n].x + S[t][n].y, acc[n]);
            }
        }
    }
}

// IQ4_XS (136 B, 8-byte aligned): eight 32-element codebook groups, 6-bit
// group scale minus 32.
template <int NC>
__device__ __forceinline__ void unit_iq4xs(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    const uint2 hd = *reinterpret_cast<const uint2*>(u);
    const float d = h2f(hd.x);
    const uint32_t sh = hd.x >> 16, sl = hd.y;
#pragma unroll 1
    for (int ib = 0; ib < 8; ++ib) {
        const uint2 c0 = *reinterpret_cast<const uint2*>(u + 8 + 16 * ib);
        const uint2 c1 = *reinterpret_cast<const uint2*>(u + 16 + 16 * ib);
        const uint32_t q[4] = {c0.x, c0.y, c1.x, c1.y};
        float2 S[NC];
        zero2(S);
        cb_group<KvTable, NC>(q, xs + k0 + 32 * ib, K, S);
        const int ls = static_cast<int>(((sl >> (4 * ib)) & 15u) | (((sh >> (2 * ib)) & 3u) << 4));
        const float a = d * static_cast<float>(ls - 32);
#pragma unroll
        for (int n = 0; n < NC; ++n) acc[n] = fmaf(a, S[n].x + S[n].y, acc[n]);
    }
}

// Repacked Q4_0 (qrepack): a unit is the 16 code bytes of eight blocks, then
// their eight f16 scales; every code word is aligned, so each block decodes
// like the odd blocks of the native layout (same nibble-in-mantissa trick,
// activations staged in that order). Rolled over block pairs.
template <int NC>
__device__ __forceinline__ void unit_q4_0r(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    const uint32_t mask[5] = {0xFu, 0xF0u, 0xF00u, 0xF000u, 0xF0000u};
    const uint32_t kMagic = 0x43000000u;   // 128.0f
    const float2 nb0 = make_float2(-(128.f + 8.f * 0x1p-16f), -(128.f + 8.f * 0x1p-12f));
    const float2 nb1 = make_float2(-(128.f + 8.f * 0x1p-8f), -(128.f + 8.f * 0x1p-4f));
    const float2 nb2 = make_float2(-136.f, -(128.f + 8.f * 0x1p-8f));
    const float2 nb3 = make_float2(-(128.f + 8.f * 0x1p-4f), -136.f);
    const uint4 sv = *reinterpret_cast<const uint4*>(u + 128);
#pragma unroll 1
    for (int pr = 0; pr < 4; ++pr) {
        const uint32_t sp = pr == 0 ? sv.x : pr == 1 ? sv.y : pr == 2 ? sv.z : sv.w;
        const uint4 c0 = *reinterpret_cast<const uint4*>(u + 32 * pr);
        const uint4 c1 = *reinterpret_cast<const uint4*>(u + 32 * pr + 16);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t words[4] = {h ? c1.x : c0.x, h ? c1.y : c0.y, h ? c1.z : c0.z, h ? c1.w : c0.w};
            const float d = h2f(h ? (sp >> 16) : sp);
            const int kb = k0 + 32 * (2 * pr + h);
            float2 S[NC][2];
#pragma unroll
            for (int n = 0; n < NC; ++n) S[n][0] = S[n][1] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t v = words[j], sh = v >> 12;
                const float2 f01 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[0], kMagic)),
                                                          __uint_as_float(and_or(v, mask[1], kMagic))), nb0);
                const float2 f23 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[2], kMagic)),
                                                          __uint_as_float(and_or(v, mask[3], kMagic))), nb1);
                const float2 f45 = __fadd2_rn(make_float2(__uint_as_float(and_or(v, mask[4], kMagic)),
                                                          __uint_as_float(and_or(sh, mask[2], kMagic))), nb2);
                const float2 f67 = __fadd2_rn(make_float2(__uint_as_float(and_or(sh, mask[3], kMagic)),
                                                          __uint_as_float(and_or(sh, mask[4], kMagic))), nb3);
#pragma unroll
                for (int n = 0; n < NC; ++n) {
                    const float4 xl = *reinterpret_cast<const float4*>(xs + n * K + kb + 8 * j);
                    const float4 xh = *reinterpret_cast<const float4*>(xs + n * K + kb + 8 * j + 4);
                    S[n][0] = __ffma2_rn(f01, make_float2(xl.x, xl.y), S[n][0]);
                    S[n][1] = __ffma2_rn(f23, make_float2(xl.z, xl.w), S[n][1]);
                    S[n][0] = __ffma2_rn(f45, make_float2(xh.x, xh.y), S[n][0]);
                    S[n][1] = __ffma2_rn(f67, make_float2(xh.z, xh.w), S[n][1]);
                }
            }
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float2 t2 = __fadd2_rn(S[n][0], S[n][1]);
                acc[n] = fmaf(d, t2.x + t2.y, acc[n]);
            }
        }
    }
}

// Repacked Q8_0: the 32 code bytes of eight blocks, then their eight f16
// scales. Rolled over block pairs; codes in natural order.
template <int NC>
__device__ __forceinline__ void unit_q8_0r(const uint8_t* u, const float* xs, int K, int k0, float (&acc)[NC]) {
    const float2 nb = nbias(128.f);
    const uint4 sv = *reinterpret_cast<const uint4*>(u + 256);
#pragma unroll 1
    for (int pr = 0; pr < 4; ++pr) {
        const uint32_t sp = pr == 0 ? sv.x : pr == 1 ? sv.y : pr == 2 ? sv.z : sv.w;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 c0 = *reinterpret_cast<const uint4*>(u + 64 * pr + 32 * h);
            const uint4 c1 = *reinterpret_cast<const uint4*>(u + 64 * pr + 32 * h + 16);
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            const int kb = k0 + 32 * (2 * pr + h);
            float2 S[NC];
            zero2(S);
#pragma unroll
            for (int i = 0; i < 8; ++i) dot4<NC>(w[i] ^ 0x80808080u, nb, xs + kb + 4 * i, K, S);   // int8 + 128
            const float d = h2f(h ? (sp >> 16) : sp);
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[n] = fmaf(d, S[n].x + S[n].y, acc[n]);
        }
    }
}

template <int KIND, int NC>
__device__ __forceinline__ void unit(const uint8_t* u, const float* xs, const float* xsum, int K, int k0,
                                     float (&acc)[NC]) {
    if constexpr (KIND == Q4_0) {
        static_assert(SG<KIND>::UB == 8, "the Q4_0 decoder takes eight blocks");
        if constexpr (NC == 1) unit_q4_0_flat<NC>(u, xs, K, k0, acc);
        else unit_q4_0<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == Q8_0) {
        static_assert(SG<KIND>::UB == 8, "the Q8_0 decoder takes eight blocks");
        unit_q8_0<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == Q4_0R) {
        unit_q4_0r<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == Q8_0R) {
        unit_q8_0r<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == Q5_0) {
        static_assert(SG<KIND>::UB == 8, "the Q5_0 decoder takes eight blocks");
        unit_q5_0<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == IQ4_NL) {
        static_assert(SG<KIND>::UB == 8, "the IQ4_NL decoder takes eight blocks");
        unit_iq4nl<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == MXFP4) {
        static_assert(SG<KIND>::UB == 16, "the MXFP4 decoder takes sixteen blocks");
        unit_mxfp4<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == Q4_K || KIND == Q5_K) {
        unit_k45<KIND, NC>(u, xs, xsum, K, k0, acc);
    } else if constexpr (KIND == Q6_K) {
        unit_q6k<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == Q2_K) {
        unit_q2k<NC>(u, xs, xsum, K, k0, acc);
    } else if constexpr (KIND == Q3_K) {
        unit_q3k<NC>(u, xs, K, k0, acc);
    } else if constexpr (KIND == Q4_1 || KIND == Q5_1 || KIND == Q8_1) {
        static_assert(SG<KIND>::UB == 8, "the Q4_1 / Q5_1 / Q8_1 decoder takes eight blocks");
        unit_legacy1<KIND, NC>(u, xs, xsum, K, k0, acc);
    } else {
        static_assert(KIND == IQ4_XS, "every format has a unit decoder");
        unit_iq4xs<NC>(u, xs, K, k0, acc);
    }
}

// ---------------------------------------------------------------------------
// shared-memory layout
// ---------------------------------------------------------------------------
struct Lay {
    int xs, red, tbl, bars, total;
};

// Grouped tables (int32): ecnt[E + 1] (last = bad ids), eoff[E + 2],
// ioff[E + 2] (items before expert e), pos[A], order[A], misc[4].
__host__ __device__ __forceinline__ int tbl_ints(int E, int A) { return 3 * (E + 2) + 2 * A + 4; }

__host__ __device__ __forceinline__ Lay layout(int stage_b, int stages, int ncmax, int K, int nw, bool grouped, int E,
                                               int A, bool xsum) {
    Lay l;
    int off = stages * stage_b;
    l.xs = off;
    off += ncmax * K * 4;
    off += xsum ? ncmax * (K / 16) * 4 : 0;   // per-16 activation sums (formats with mins)
    l.red = off;
    off += 2 * ncmax * nw * 32 * 4;
    l.tbl = off;
    off += grouped ? tbl_ints(E, A) * 4 : 0;
    off = (off + 15) & ~15;
    l.bars = off;
    off += (2 * kMaxStages + 6) * 8 + 16;
    l.total = off + 128;   // + slack to align the base to 128 bytes
    return l;
}

struct Tables {
    int* ecnt;
    int* eoff;
    int* ioff;
    int* pos;
    int* order;
    int* misc;   // [0] total items, [1] bad count
};

__device__ __forceinline__ Tables tables(uint8_t* base, int E, int A) {
    Tables t;
    int* p = reinterpret_cast<int*>(base);
    t.ecnt = p;
    t.eoff = p + (E + 2);
    t.ioff = p + 2 * (E + 2);
    t.pos = p + 3 * (E + 2);
    t.order = t.pos + A;
    t.misc = t.order + A;
    return t;
}

// One work item: 32 rows (row group g) of expert e, columns [col0, col0 + ncol).
struct Item {
    int e, col0, ncol;
    int64_t g;
};

// Walks the CTA's contiguous item range in order (plain: one problem). The
// first lookup binary-searches the expert (a linear scan over up to a thousand
// experts in shared memory would delay the CTA's first weight copy by
// microseconds); later ones step forward.
struct ItemWalker {
    int e = -1;
    __device__ __forceinline__ Item at(int64_t i, const GemvArgs& a, const Tables& t, int64_t rg, int ncmax) {
        Item it;
        if (!a.x_row) {
            it.e = 0;
            it.col0 = 0;
            it.ncol = a.ncols;
            it.g = i;
            return it;
        }
        if (e < 0) {
            // last expert e with ioff[e] <= i (ioff is non-decreasing, ioff[0] = 0)
            int lo = 0, hi = a.n_experts;   // ioff[n_experts] = total > i
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (t.ioff[mid] <= i) lo = mid;
                else hi = mid;
            }
            e = lo;
        }
        while (t.ioff[e + 1] <= i) ++e;
        const int64_t local = i - t.ioff[e];
        const int b = static_cast<int>(local / rg);
        it.e = e;
        it.g = local - static_cast<int64_t>(b) * rg;
        it.col0 = t.eoff[e] + b * ncmax;
        it.ncol = min(ncmax, t.ecnt[e] - b * ncmax);
        return it;
    }
};

// Bucket the assignments by expert, in assignment order (deterministic: every
// CTA builds the same tables). Run by one warp after the CTA has written each
// assignment's bucket (expert id, or E for a bad id or activation row) to
// pos[]. On return pos[r] = bucket << 16 | rank of r within its bucket.
__device__ void build_tables(const GemvArgs& a, const Tables& t, int64_t rg, int ncmax, int lane) {
    const unsigned full = 0xffffffffu;
    const int E = a.n_experts, A = a.n_assign;
    for (int e = lane; e <= E; e += 32) t.ecnt[e] = 0;
    __syncwarp();
    for (int r0 = 0; r0 < A; r0 += 32) {
        const int r = r0 + lane;
        const bool act = r < A;
        const int key = act ? t.pos[r] : -1;
        const unsigned same = __match_any_sync(full, key);
        const int rank = __popc(same & ((1u << lane) - 1u));
        const int base = act ? t.ecnt[key] : 0;
        __syncwarp();
        if (act) {
            t.pos[r] = (key << 16) | (base + rank);
            if (rank == 0) t.ecnt[key] = base + __popc(same);
        }
        __syncwarp();
    }
    // exclusive scans over buckets 0..E of the assignment counts and of the
    // work items (row groups x column blocks), one run of buckets per lane
    const int per = (E + 1 + 31) / 32;
    const int e0 = min(E + 1, lane * per), e1 = min(E + 1, e0 + per);
    const int rgi = static_cast<int>(rg);
    int cs = 0, is = 0;
    for (int e = e0; e < e1; ++e) {
        cs += t.ecnt[e];
        if (e < E) is += ((t.ecnt[e] + ncmax - 1) / ncmax) * rgi;
    }
    int ci = cs, ii = is;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int c2 = __shfl_up_sync(full, ci, off), i2 = __shfl_up_sync(full, ii, off);
        if (lane >= off) {
            ci += c2;
            ii += i2;
        }
    }
    const int ctot = __shfl_sync(full, ci, 31), itot = __shfl_sync(full, ii, 31);
    int cx = ci - cs, ix = ii - is;
    for (int e = e0; e < e1; ++e) {
        t.eoff[e] = cx;
        t.ioff[e] = ix;
        cx += t.ecnt[e];
        if (e < E) ix += ((t.ecnt[e] + ncmax - 1) / ncmax) * rgi;
    }
    __syncwarp();
    if (lane == 0) {
        t.eoff[E + 1] = ctot;
        t.ioff[E + 1] = itot;
        t.misc[0] = itot;
        t.misc[1] = t.ecnt[E];
    }
    __syncwarp();
    for (int r = lane; r < A; r += 32) {
        const int v = t.pos[r];
        t.order[t.eoff[v >> 16] + (v & 0xFFFF)] = r;
    }
    __syncwarp();
}

__device__ __forceinline__ float silu(float v) { return v / (1.f + expf(-v)); }

__device__ __forceinline__ float load_x(const void* X, int xdt, int64_t i) {
    if (xdt == 1) return __half2float(reinterpret_cast<const __half*>(X)[i]);
    return reinterpret_cast<const float*>(X)[i];
}

// Stage the activations of columns [col0, col0 + ncol) (zeros up to NCMAX) in
// the format's layout. Consumers only. Each thread issues a batch of eight
// 16-byte loads before it stores any of them, so the staging costs one L2
// round trip per batch instead of one per load.
template <int KIND, int NCMAX, bool SWIGLU>
__device__ void stage_x_rows(const GemvArgs& a, const Tables& t, const Item& it, float* xs, int tid, int nthr) {
    constexpr int B = 8;
    const int K = a.K;
    const int kq = K / 4;
    const int total = NCMAX * kq;
    const bool vec = a.x_dtype == 0 && (reinterpret_cast<uintptr_t>(a.X) & 15) == 0;
    for (int base = tid; base < total; base += B * nthr) {
        float4 v[B];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int idx = base + j * nthr;
            v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < total) {
                const int n = idx / kq, k = 4 * (idx - n * kq);
                if (n < it.ncol) {
                    const int64_t row = a.x_row ? static_cast<int64_t>(a.x_row[t.order[it.col0 + n]]) : n;
                    const int64_t off = row * (SWIGLU ? a.x_stride : static_cast<int64_t>(K)) + k;
                    if constexpr (SWIGLU) {
                        // gate value k and up value K + k of a gate_up output row
                        const float* xr = reinterpret_cast<const float*>(a.X) + off;
                        const float4 g = *reinterpret_cast<const float4*>(xr);
                        const float4 u = *reinterpret_cast<const float4*>(xr + K);
                        v[j] = make_float4(silu(g.x) * u.x, silu(g.y) * u.y, silu(g.z) * u.z, silu(g.w) * u.w);
                    } else if (vec) {
                        v[j] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.X) + off);
                    } else {
                        v[j].x = load_x(a.X, a.x_dtype, off);
                        v[j].y = load_x(a.X, a.x_dtype, off + 1);
                        v[j].z = load_x(a.X, a.x_dtype, off + 2);
                        v[j].w = load_x(a.X, a.x_dtype, off + 3);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int idx = base + j * nthr;
            if (idx >= total) continue;   // (no break: the loop must unroll, v[] stays in registers)
            const int n = idx / kq, k = 4 * (idx - n * kq);
            if constexpr (KIND == Q4_0 || KIND == Q4_0R) {
                const float vv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int kk = k + c, b = kk >> 5, e = kk & 31;
                    // native even blocks start 2 bytes off a word; repacked codes are all aligned
                    const int slot = q4_slot(e, KIND == Q4_0 && (b & 1) == 0);
                    // times 2^-p, an exact power-of-two product
                    xs[n * K + 32 * b + slot] = vv[c] * __int_as_float((127 - q4_pow(slot & 7)) << 23);
                }
            } else if constexpr (CbOrder<KIND>::ON) {
                // MXFP4's table holds twice the E2M1 value: its activations are
                // staged halved (exact)
                const float sc = (KIND == MXFP4) ? 0.5f : 1.f;
                const float vv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int kk = k + c;
                    xs[n * K + (kk & ~31) + cb_slot(kk & 31)] = vv[c] * sc;
                }
            } else {
                *reinterpret_cast<float4*>(xs + n * K + k) = v[j];
            }
        }
    }
}


// Per-16 activation sums (sequential fp32 adds over the staged values, in
// natural order) for the formats with a minimum term: xsum[n * K / 16 + g].
template <int NCMAX>
__device__ void stage_xsum(const float* xs, float* xsum, int K, int tid, int nthr) {
    const int per = K / 16;
    for (int i = tid; i < NCMAX * per; i += nthr) {
        const int n = i / per, g = i - n * per;
        const float4* p = reinterpret_cast<const float4*>(xs + n * K + 16 * g);
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = p[q];
            t += v.x;
            t += v.y;
            t += v.z;
            t += v.w;
        }
        xsum[i] = t;
    }
}

template <int KIND, int NC, int NCMAX>
__device__ __forceinline__ void consume_item(const GemvArgs& a, const Tables& t, const Item& item, uint8_t* stage0,
                                             int stage_b, const float* xs, float* red, uint64_t* full,
                                             uint64_t* empty, uint64_t* red_full, uint64_t* red_empty,
                                             volatile int* abort_flag, int it_base, int gi, int warp, int lane) {
    using G = SGeo<KIND>;
    constexpr int NW = G::NW;
    const int nwu = a.nwu, ngroups = NW / nwu, grp = warp / nwu, u = warp - grp * nwu;
    const int S = a.stages, K = a.K;
    float acc[NC];
#pragma unroll
    for (int n = 0; n < NC; ++n) acc[n] = 0.f;
    // first chunk of this item handled by my group
    int c = (grp - it_base % ngroups + ngroups) % ngroups;
    for (; c < a.cpr; c += ngroups) {
        const int it = it_base + c;
        const int s = it % S, use = it / S;
        const bool ok = !*abort_flag && mbar_wait(&full[s], use & 1, abort_flag, a.err);
        const int units = min(nwu, a.upr - c * nwu);
        if (ok && u < units)
            unit<KIND, NC>(stage0 + s * stage_b + lane * a.stride + u * G::UNIT_B, xs, xs + NCMAX * K, K,
                           (c * nwu + u) * G::UNIT_E, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    // cross-warp sum through shared memory; the item's writer warp (rotating)
    // waits, adds and stores
    const int p = gi & 1, use = gi >> 1;
    float* rb = red + p * NCMAX * NW * 32;   // fixed stride: items may differ in NC
    if (use > 0 && !*abort_flag) mbar_wait(&red_empty[p], (use - 1) & 1, abort_flag, a.err);
#pragma unroll
    for (int n = 0; n < NC; ++n) rb[(n * NW + warp) * 32 + lane] = acc[n];
    __syncwarp();
    if (lane == 0) mbar_arrive(&red_full[p]);
    if (warp == gi % NW) {
        const bool ok = !*abort_flag && mbar_wait(&red_full[p], use & 1, abort_flag, a.err);
        const int64_t row = item.g * kRows + lane;
        if (ok && row < a.M) {
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                if (n < item.ncol) {
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < NW; ++w) v += rb[(n * NW + w) * 32 + lane];
                    const int64_t r = a.x_row ? static_cast<int64_t>(t.order[item.col0 + n]) : n;
                    store_y(a.Y, a.y_dtype, r * a.M + row, v);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[p]);
    }
}

// Q4_0 (17 warps) gets the registers of one CTA per SM: its decoder spills at
// the 60 registers two such CTAs would allow. The other formats keep room for
// a second CTA (the next kernel's, under programmatic dependent launch).
template <int KIND> struct MinBlocks { static constexpr int V = (KIND == Q4_0 || KIND == Q4_0R) ? 1 : 2; };

// SWI: the activations are SwiGLU of gate_up rows (the MoE down projection).
// A template parameter, not a runtime mode, so that the plain kernels carry
// none of its code: the single-column decode kernels are sensitive to their
// instruction footprint (measured: the unexecuted SwiGLU staging in them cost
// the two-GEMV decode step 2.7 us).
template <int KIND, int NCMAX, bool SWI>
__global__ void __launch_bounds__((SG<KIND>::NW + 1) * 32, MinBlocks<KIND>::V)
    k_gemv(const __grid_constant__ CUtensorMap tmW, GemvArgs a) {
    using G = SGeo<KIND>;
    constexpr int NW = G::NW;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // 128-byte aligned base (TMA tensor destinations), by arithmetic on the
    // shared array so that accesses stay shared-memory loads and stores
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const bool grouped = a.x_row != nullptr;
    const int K = a.K;
    const int stage_b = kRows * a.stride;
    const Lay L = layout(stage_b, a.stages, NCMAX, K, NW, grouped, a.n_experts, a.n_assign, XSum<KIND>::ON);
    uint8_t* stage0 = smem;
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    float* red = reinterpret_cast<float*>(smem + L.red);
    const Tables T = tables(smem + L.tbl, a.n_experts, a.n_assign);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + kMaxStages;
    uint64_t* red_full = empty + kMaxStages;
    uint64_t* red_empty = red_full + 2;
    uint64_t* tbl_ready = red_empty + 2;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tbl_ready + 1);

    // Let the next kernel on the stream start its set-up as soon as possible.
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], a.nwu);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(&red_full[p], NW);
            mbar_init(&red_empty[p], 1);
        }
        mbar_init(tbl_ready, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int64_t rg = (a.M + kRows - 1) / kRows;   // row groups per problem
    const int S = a.stages;
    if (grouped) {
        // the expert ids come from earlier kernels: wait for them, then every
        // thread files a share of the assignments into their buckets
        grid_dep_wait();
        for (int r = threadIdx.x; r < a.n_assign; r += blockDim.x) {
            const int e = a.expert_id[r];
            const int64_t xr = a.x_row[r];
            T.pos[r] = (e >= 0 && e < a.n_experts && xr >= 0 && xr < a.n_x_rows) ? e : a.n_experts;
        }
        __syncthreads();
    }

    if (warp == NW) {
        // ---------------- producer warp ----------------
        const uint64_t pol = l2_evict_first_policy();
        int64_t n_items = rg;
        bool waited = false;
        if (grouped || !(a.flags & kFlagPrefetchW)) {
            grid_dep_wait();
            waited = true;
        }
        if (grouped) {
            build_tables(a, T, rg, NCMAX, lane);
            n_items = T.misc[0];
            __syncwarp();
            if (lane == 0) mbar_arrive(tbl_ready);
        }
        const int64_t lo = static_cast<int64_t>(blockIdx.x) * n_items / gridDim.x;
        const int64_t hi = static_cast<int64_t>(blockIdx.x + 1) * n_items / gridDim.x;
        ItemWalker walk;
        int it = 0;
        const uint32_t box_bytes = static_cast<uint32_t>(stage_b);
        const int cg = a.nwu * G::UNIT_B / 16;   // granules per chunk
        for (int64_t i = lo; i < hi; ++i) {
            const Item item = walk.at(i, a, T, rg, NCMAX);
            for (int c = 0; c < a.cpr; ++c, ++it) {
                const int s = it % S, use = it / S;
                if (use > 0 && !waited) {
                    // every prefetch stage is issued: wait for the previous grid
                    grid_dep_wait();
                    waited = true;
                }
                if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, abort_flag, a.err)) goto drain;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[s], box_bytes);
                    // innermost coordinate in 8-byte words: a multiple of two (16-byte aligned)
                    tma3d(stage0 + s * stage_b, &tmW, 2 * c * cg, static_cast<int>(item.g * kRows), item.e, &full[s],
                          pol);
                }
                __syncwarp();
            }
        }
        if (!waited) grid_dep_wait();
    drain:
        // Before the CTA can retire, every issued copy must have landed: wait
        // (bounded, ignoring the abort flag) for the last phase of each stage.
        {
            const int issued = it;
            for (int s = 0; s < S && s < issued; ++s) {
                const int last_use = (issued - 1 - s) / S;   // uses of slot s: it = s + S * use
                const long long t0 = clock64();
                while (!mbar_try_wait(&full[s], last_use & 1)) {
                    if (clock64() - t0 > (1ll << 31)) {
                        atomicOr(a.err, DEV_ERR_TIMEOUT);
                        break;
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumer warps ----------------
    grid_dep_wait();
    int64_t n_items = rg;
    if (grouped) {
        if (!mbar_wait(tbl_ready, 0, abort_flag, a.err)) *abort_flag = 1;
        n_items = T.misc[0];
        // assignments with a bad expert id or activation row: NaN rows, flagged
        if (blockIdx.x == 0 && !*abort_flag && T.misc[1] > 0) {
            const int nb = T.misc[1], b0 = T.eoff[a.n_experts];
            for (int64_t idx = threadIdx.x; idx < static_cast<int64_t>(nb) * a.M; idx += NW * 32) {
                const int64_t j = idx / a.M;
                store_y(a.Y, a.y_dtype, static_cast<int64_t>(T.order[b0 + j]) * a.M + (idx - j * a.M),
                        __int_as_float(0x7fc00000));
            }
            if (threadIdx.x == 0) atomicOr(a.err, DEV_ERR_BAD_INDEX);
        }
    }
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * n_items / gridDim.x;
    const int64_t hi = static_cast<int64_t>(blockIdx.x + 1) * n_items / gridDim.x;
    ItemWalker walk;
    int cur_e = -1, cur_c = -1, it_base = 0, gi = 0;
    for (int64_t i = lo; i < hi; ++i, it_base += a.cpr, ++gi) {
        const Item item = walk.at(i, a, T, rg, NCMAX);
        if (item.e != cur_e || item.col0 != cur_c) {
            if (cur_e >= 0) named_bar_sync(1, NW * 32);   // everyone is done with the old activations
            stage_x_rows<KIND, NCMAX, SWI>(a, T, item, xs, threadIdx.x, NW * 32);
            named_bar_sync(1, NW * 32);
            if constexpr (XSum<KIND>::ON) {
                stage_xsum<NCMAX>(xs, xs + NCMAX * K, K, threadIdx.x, NW * 32);
                named_bar_sync(1, NW * 32);
            }
            cur_e = item.e;
            cur_c = item.col0;
        }
        const int nc = item.ncol;
        if (NCMAX == 1 || nc <= 1)
            consume_item<KIND, 1, NCMAX>(a, T, item, stage0, stage_b, xs, red, full, empty, red_full, red_empty,
                                         abort_flag, it_base, gi, warp, lane);
        else if (NCMAX == 2 || nc <= 2)
            consume_item<KIND, (NCMAX < 2 ? NCMAX : 2), NCMAX>(a, T, item, stage0, stage_b, xs, red, full, empty,
                                                               red_full, red_empty, abort_flag, it_base, gi, warp,
                                                               lane);
        else if (NCMAX == 4 || nc <= 4)
            consume_item<KIND, (NCMAX < 4 ? NCMAX : 4), NCMAX>(a, T, item, stage0, stage_b, xs, red, full, empty,
                                                               red_full, red_empty, abort_flag, it_base, gi, warp,
                                                               lane);
        else
            consume_item<KIND, NCMAX, NCMAX>(a, T, item, stage0, stage_b, xs, red, full, empty, red_full,
                                             red_empty, abort_flag, it_base, gi, warp, lane);
    }
}

// Launch tunables, overridable for sweeps: QMM_GEMV_NWU (warps per chunk),
// QMM_GEMV_STAGES, QMM_GEMV_SMEM (KB of shared memory per CTA), QMM_GEMV_CTAS.
// 0 = automatic.
int env_int(const char* name) {
    const char* v = getenv(name);
    return v ? atoi(v) : 0;
}
const int kEnvNwu = env_int("QMM_GEMV_NWU");
const int kEnvStages = env_int("QMM_GEMV_STAGES");
const int kEnvSmemKB = env_int("QMM_GEMV_SMEM");
const int kEnvCtas = env_int("QMM_GEMV_CTAS");   // CTAs per SM (1 or 2)

int pow2ceil(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

struct Plan {
    bool ok = false;
    int ncmax = 1, nwu = 0, stride = 0, stages = 0, upr = 0, cpr = 0;  // stride = box granules * 16
    size_t smem = 0;
};

template <int KIND>
Plan plan(const Problem& p) {
    using G = SGeo<KIND>;
    Plan pl;
    if (p.K > (1 << 24) || p.K % G::UNIT_E) return pl;
    if (p.row_bytes % 16 || p.row_stride % 16 || reinterpret_cast<uintptr_t>(p.W) % 16) return pl;
    const bool grouped = p.x_row != nullptr;
    if (p.x_mode == 1 && (!p.x_row || p.x_dtype != 0 || p.K % 4 || p.x_stride % 4 || p.x_stride < 2 * p.K ||
                          reinterpret_cast<uintptr_t>(p.X) % 16))
        return pl;
    if (grouped) {
        if (p.expert_stride % 16 || p.n_experts > kMaxGroupedExperts || p.N > kMaxGroupedAssign) return pl;
        // up to four columns per problem: measured on the 64-token MoE
        // projections, the 8-column decode (register-bound) lost more than
        // re-streaming the rows of the experts with over four tokens
        // (a split-K view has the same few columns in every slice: no more)
        const int want = p.cols_per_expert > 0
                             ? pow2ceil(p.cols_per_expert)
                             : pow2ceil(static_cast<int>((4 * p.N + p.n_experts - 1) / p.n_experts));
        pl.ncmax = want < 4 ? want : 4;
        // item counts are int32 on the device
        if ((p.N + p.n_experts) * ((p.M + kRows - 1) / kRows) >= (int64_t(1) << 31)) return pl;
    } else {
        if (p.N > 8) return pl;
        pl.ncmax = pow2ceil(static_cast<int>(p.N));
    }
    const int K = static_cast<int>(p.K);
    // Warps per chunk (nwu): a divisor of NW whose chunk is whole 16-byte
    // vectors, and whose last chunk of a row is too. The NW / nwu consumer
    // groups take the chunks round-robin, and the number of stages must be a
    // multiple of the number of groups: then every stage belongs to one group,
    // which consumes its chunks in order, so no waiter is ever two phases
    // ahead of a stage's barrier (a parity wait cannot tell those apart).
    const int E = grouped ? p.n_experts : 0, A = grouped ? static_cast<int>(p.N) : 0;
    // short rows: no more warps per chunk than the row has units (the rest
    // of a group would idle on every chunk)
    int pref = (kEnvNwu > 0) ? kEnvNwu : SG<KIND>::NWU;
    while (pref > 1 && pref > K / G::UNIT_E) pref >>= 1;
    int cands[16], ncand = 0;   // the preferred size, smaller ones, then larger ones
    for (int w = pref; w >= 1; w >>= 1) cands[ncand++] = w;
    for (int w = G::NW; w > pref && ncand < 16; w >>= 1) cands[ncand++] = w;
    for (int ci = 0; ci < ncand; ++ci) {
        const int w = cands[ci];
        if (w > G::NW || G::NW % w || (w * G::UNIT_B) % 16) continue;
        const int upr = K / G::UNIT_E;
        const int ngroups = G::NW / w;
        const int cg = w * G::UNIT_B / 16;          // granules per chunk
        const int bg = (cg % 2) ? cg : cg + 1;      // box granules: odd
        if (2 * bg > 256) continue;                 // TMA box dimension limit (256 8-byte words)
        const int stride = bg * 16;
        const int stage_b = kRows * stride;
        auto total = [&](int st) {
            return layout(stage_b, st, pl.ncmax, K, G::NW, grouped, E, A, XSum<KIND>::ON).total;
        };
        if (ngroups > kMaxStages || total(ngroups) > kSmemBudget) continue;
        // two CTAs per SM when the stages fit in half the SM, else one deep CTA
        const int want = ngroups >= 4 ? ngroups : 4;
        int budget = kEnvSmemKB > 0 ? kEnvSmemKB * 1024 : (total(want) <= kCoresident ? kCoresident : kSmemBudget);
        if (budget > kSmemBudget) budget = kSmemBudget;
        int st = kMaxStages;
        while (st > ngroups && total(st) > budget) --st;
        if (kEnvStages > 0 && kEnvStages <= kMaxStages && total(kEnvStages) <= kSmemBudget) st = kEnvStages;
        st = (st / ngroups) * ngroups;
        if (st < ngroups) st = ngroups;
        if (st < 2) st = 2;
        if (total(st) > kSmemBudget) continue;
        pl.upr = upr;
        pl.nwu = w;
        pl.cpr = (upr + w - 1) / w;
        pl.stride = stride;
        pl.stages = st;
        pl.smem = static_cast<size_t>(total(st));
        pl.ok = true;
        return pl;
    }
    return pl;
}

template <int KIND, int NCMAX>
cudaError_t launch_nc(const Problem& p, const Plan& pl, cudaStream_t s) {
    using G = SGeo<KIND>;
    // SwiGLU staging only for the grouped product (the MoE down projection),
    // which uses at most four columns per problem
    auto kern = k_gemv<KIND, NCMAX, false>;
    if constexpr (NCMAX <= 4) {
        if (p.x_mode == 1) kern = k_gemv<KIND, NCMAX, true>;
    }
    // weights as (8-byte word of the row, row, expert)
    CUtensorMap tm;
    const int E = p.x_row ? p.n_experts : 1;
    const uint64_t rstride = p.row_stride ? p.row_stride : p.row_bytes;
    const uint64_t estride = p.x_row ? p.expert_stride : static_cast<uint64_t>(p.M) * rstride;
    const uint64_t dims[3] = {p.row_bytes / 8, static_cast<uint64_t>(p.M), static_cast<uint64_t>(E)};
    const uint64_t strides[2] = {rstride, estride};
    const uint32_t box[3] = {static_cast<uint32_t>(pl.stride / 8), static_cast<uint32_t>(kRows), 1};
    if (!encode_tiled_map(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, p.W, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(pl.smem));
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t rg = (p.M + kRows - 1) / kRows;
    const int sms = sm_count(dev);
    // plain: at most one CTA per row group; grouped: the item count is known
    // only on the device, so one CTA per SM
    const int per_sm = (kEnvCtas == 2 && 2 * pl.smem <= 226 * 1024) ? 2 : 1;
    const int grid = p.x_row ? per_sm * sms : static_cast<int>(imin64(rg, static_cast<int64_t>(per_sm) * sms));
    GemvArgs a = {};
    a.W = p.W;
    a.row_bytes = p.row_bytes;
    a.M = p.M;
    a.K = static_cast<int>(p.K);
    a.X = p.X;
    a.x_dtype = p.x_dtype;
    a.Y = p.Y;
    a.y_dtype = p.y_dtype;
    a.x_mode = p.x_mode;
    a.x_stride = p.x_stride ? p.x_stride : p.K;
    a.ncols = static_cast<int>(p.N);
    a.x_row = p.x_row;
    a.expert_id = p.expert_id;
    a.expert_stride = p.expert_stride;
    a.n_experts = p.x_row ? p.n_experts : 0;
    a.n_assign = p.x_row ? static_cast<int>(p.N) : 0;
    a.n_x_rows = p.n_x_rows;
    a.stages = pl.stages;
    a.nwu = pl.nwu;
    a.stride = pl.stride;
    a.upr = pl.upr;
    a.cpr = pl.cpr;
    a.flags = (!p.x_row && (p.flags & QMM_FLAG_WEIGHTS_CONST)) ? kFlagPrefetchW : 0;
    a.err = p.err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((G::NW + 1) * 32);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tm, a);
    count_launch(1);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int KIND>
void run(const Problem& p, cudaStream_t s, cudaError_t* e) {
    const Plan pl = plan<KIND>(p);
    if (!pl.ok) {
        *e = cudaErrorInvalidValue;
        return;
    }
    switch (pl.ncmax) {
    case 1: *e = launch_nc<KIND, 1>(p, pl, s); break;
    case 2: *e = launch_nc<KIND, 2>(p, pl, s); break;
    case 4: *e = launch_nc<KIND, 4>(p, pl, s); break;
    default: *e = launch_nc<KIND, 8>(p, pl, s); break;
    }
}

template <int KIND>
void ok_dispatch(const Problem& p, bool* out) { *out = plan<KIND>(p).ok; }

}  // namespace

bool gemv_stream_ok(const Problem& p) {
    bool ok = false;
    QMM_DISPATCH_GEMV_KIND(p.kind, ok_dispatch, p, &ok);
    return ok;
}

cudaError_t launch_gemv_stream(const Problem& p, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    QMM_DISPATCH_GEMV_KIND(p.kind, run, p, s, &e);
    return e;
}

}  // namespace qmm
