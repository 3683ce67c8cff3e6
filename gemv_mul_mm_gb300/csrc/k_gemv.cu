// k_gemv.cu -- weight-streaming quantized GEMV for small N (decode).
//
// y[n, m] = sum_k W[m, k] * x[n, k], N <= 8. Decode is bound by streaming the
// weights from HBM once (inferencelayer 0.2.8 src/cublas_prefill.rs: "decode's
// whole cost is streaming weights"), so the design is about bytes in flight
// and coalescing, not arithmetic:
//
//   * A CTA owns groups of 32 weight rows (one row per lane) and walks them in
//     K-chunks. One producer warp moves each chunk of the 32 rows from HBM into
//     a shared-memory stage with 1-D bulk copies (`cp.async.bulk`, one 16-byte
//     aligned copy per row, completing on an mbarrier, L2 evict-first); up to
//     4 stages are in flight per SM (~100 KB), enough to cover HBM latency.
//   * NW consumer warps split each chunk along K: warp w decodes its unit of
//     the chunk for all 32 rows (lane = row), reading the row's bytes with
//     16-byte shared loads (row stride padded to an odd number of 16-byte
//     words, so the 32 lanes hit distinct banks) and the activations with
//     broadcast loads. No cross-lane reduction; the NW partial sums per row
//     are added through shared memory at the end of the row group.
//   * Activations are staged once per CTA (one bulk copy when they are fp32 and
//     16-byte aligned) in a per-format layout: for Q4_0 each block's 32 values
//     are permuted to match the order in which two nibbles at a time are OR-ed
//     into the mantissa of 128.0f (no int->float convert), plus one offset per
//     block; they feed packed fp32x2 FMAs (sm_100 FFMA2), and the scale d
//     multiplies the block's partial sum in fp32.
//   * Persistent grid (one or two CTAs per SM) over the row groups, launched
//     with programmatic dependent launch: the next kernel's set-up (and, when
//     the caller declares the weights constant, its first weight stages)
//     overlaps the tail of the previous kernel on the stream.
//
// The P4 page's v3 lesson (stage x in shared, keep lanes on distinct banks,
// keep loads in flight) is kept; its f16x2 accumulation is not (too lossy for
// the 1e-3 relative bar over K = 4096), nor its structure-of-arrays layout.
#include <cstdlib>

#include <cuda_fp16.h>

#include "decode.cuh"
#include "qmm_internal.cuh"
#include "sm100_async.cuh"

namespace qmm {
namespace {

constexpr int kRows = 32;
constexpr int kMaxStages = 6;
constexpr int kSmemBudget = 220 * 1024;

// Per format: blocks per warp unit (UB) and consumer warps (NW). A unit's bytes
// times NW (one chunk row) is a multiple of 16 for every format. Measured on
// the decode workload (M = 14336, K = 4096): Q8_0 runs best with one CTA of 8
// consumer warps per SM (half a row per stage), Q4_0 with 16 consumer warps
// (a whole row per stage) -- the extra warps hide its decode latency.
template <int KIND> struct SG;
template <> struct SG<Q8_0>   { static constexpr int UB = 8,  NW = 8; };
template <> struct SG<Q4_0>   { static constexpr int UB = 8,  NW = 16; };
template <> struct SG<Q5_0>   { static constexpr int UB = 8,  NW = 8; };
template <> struct SG<IQ4_NL> { static constexpr int UB = 8,  NW = 8; };
template <> struct SG<MXFP4>  { static constexpr int UB = 16, NW = 4; };
template <> struct SG<Q4_K>   { static constexpr int UB = 1,  NW = 8; };
template <> struct SG<Q5_K>   { static constexpr int UB = 1,  NW = 8; };
template <> struct SG<Q6_K>   { static constexpr int UB = 1,  NW = 8; };
template <> struct SG<Q2_K>   { static constexpr int UB = 1,  NW = 8; };
template <> struct SG<Q3_K>   { static constexpr int UB = 1,  NW = 8; };
template <> struct SG<IQ4_XS> { static constexpr int UB = 1,  NW = 8; };

template <int KIND> struct SGeo {
    static constexpr int NW = SG<KIND>::NW;
    static constexpr int UNIT_B = SG<KIND>::UB * Geo<KIND>::BB;
    static constexpr int UNIT_E = SG<KIND>::UB * Geo<KIND>::BE;
    static constexpr int CHUNK_B = NW * UNIT_B;
    static constexpr int CHUNK_E = NW * UNIT_E;
    static constexpr int STRIDE = CHUNK_B + (((CHUNK_B / 16) % 2 == 0) ? 16 : 32);
    static constexpr int STAGE_B = kRows * STRIDE;
    static constexpr bool PARTIAL_OK = (UNIT_B % 16) == 0;  // a partial chunk is whole 16-byte rows
    static_assert(CHUNK_B % 16 == 0, "a chunk row must be whole 16-byte vectors");
    static_assert(STRIDE % 16 == 0 && (STRIDE / 16) % 2 == 1, "padded row stride");
};

struct GemvArgs {
    const uint8_t* W;
    size_t row_bytes;
    int64_t M;
    int K;
    const void* X;
    int x_dtype;
    int ncols;      // valid columns (<= NCOL)
    float* Y;
    int stages;
    int flags;      // kFlagPrefetchW | kFlagBulkX
    unsigned* err;
};

constexpr int kFlagPrefetchW = 1;  // weights may be read before the previous grid completes
constexpr int kFlagBulkX = 2;      // activations are fp32, 16-byte aligned: one bulk copy

__device__ __forceinline__ float load_x(const void* X, int xdt, int64_t i) {
    if (xdt == 1) return __half2float(reinterpret_cast<const __half*>(X)[i]);
    return reinterpret_cast<const float*>(X)[i];
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------------------
// unit decoders: acc[n] += sum over the unit's elements of W * x[n]
// ---------------------------------------------------------------------------

// Any format, from shared bytes (scale applied per element).
template <int KIND, int NCOL>
__device__ __forceinline__ void unit_generic(const uint8_t* u, const float* xs, const float*, int K, int k0,
                                             float (&acc)[NCOL]) {
    constexpr int BB = Geo<KIND>::BB, BE = Geo<KIND>::BE, UB = SG<KIND>::UB;
#pragma unroll 1
    for (int blk = 0; blk < UB; ++blk) {
        const uint8_t* b = u + blk * BB;
#pragma unroll 1
        for (int j = 0; j < BE / 32; ++j) {
            const int kb = k0 + blk * BE + 32 * j;
            float s[NCOL];
#pragma unroll
            for (int n = 0; n < NCOL; ++n) s[n] = 0.f;
#pragma unroll 8
            for (int i = 0; i < 32; ++i) {
                const float v = elem32<KIND>(b, j, i);
#pragma unroll
                for (int n = 0; n < NCOL; ++n) s[n] = fmaf(v, xs[n * K + kb + i], s[n]);
            }
#pragma unroll
            for (int n = 0; n < NCOL; ++n) acc[n] += s[n];
        }
    }
}

// (a & b) | c in one LOP3 with all three operands in registers (an immediate
// mask plus an immediate constant would otherwise take two instructions).
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Q4_0 staged-activation order. Within a block the decoder walks four 32-bit
// words of code bytes; a word holding code bytes (b0, b1, b2, b3) yields the
// low nibbles of (b0, b2), then of (b1, b3), then the high nibbles of (b0, b2)
// and of (b1, b3). Odd blocks start 4-byte aligned (word j = bytes 4j..4j+3);
// even blocks start 2 bytes off, so their words are [14, 15, 0, 1] and then
// bytes 4j-2..4j+1. q4_slot(e, even) is the staged position of element e.
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
    // word j's 8 slots: lo (b0, b2, b1, b3), then hi (b0, b2, b1, b3)
    const int within = (k & 1) * 2 + (k >> 1);
    return 8 * j + 4 * hi + within;
}

// Q4_0: 8 blocks of 18 bytes (144 B, 16-byte aligned in shared memory).
// One LOP3 turns the low nibbles of bytes 0 and 2 of a word into 0x430q_000p:
// read as fp32 it is 128 + q (+ p / 65536, far below the 1e-3 bar), and one
// IMAD (x 65536 + 0x43000000, on the FMA pipe) turns its low half into exactly
// 128 + p. So S = sum (128 + q) x and sum (q - 8) x = S - 136 * sum x = S - cb.
template <int NCOL>
__device__ __forceinline__ void unit_q4_0(const uint8_t* u, const float* xs, const float* cb, int K, int k0,
                                          float (&acc)[NCOL]) {
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(u)[i];
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    const int nb32 = K / 32;
    const uint32_t kMask = 0x000F000Fu, kMagic = 0x43000000u;
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
        float2 S[NCOL][2];
#pragma unroll
        for (int n = 0; n < NCOL; ++n) S[n][0] = S[n][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t v = words[j];
            const uint32_t t0 = and_or(v, kMask, kMagic);
            const uint32_t t1 = and_or(v >> 8, kMask, kMagic);
            const uint32_t t2 = and_or(v >> 4, kMask, kMagic);
            const uint32_t t3 = and_or(v >> 12, kMask, kMagic);
            const float2 f0 = make_float2(__uint_as_float(t0 * 65536u + kMagic), __uint_as_float(t0));
            const float2 f1 = make_float2(__uint_as_float(t1 * 65536u + kMagic), __uint_as_float(t1));
            const float2 f2 = make_float2(__uint_as_float(t2 * 65536u + kMagic), __uint_as_float(t2));
            const float2 f3 = make_float2(__uint_as_float(t3 * 65536u + kMagic), __uint_as_float(t3));
#pragma unroll
            for (int n = 0; n < NCOL; ++n) {
                const float4 xl = *reinterpret_cast<const float4*>(xs + n * K + kb + 8 * j);
                const float4 xh = *reinterpret_cast<const float4*>(xs + n * K + kb + 8 * j + 4);
                S[n][0] = __ffma2_rn(f0, make_float2(xl.x, xl.y), S[n][0]);
                S[n][1] = __ffma2_rn(f1, make_float2(xl.z, xl.w), S[n][1]);
                S[n][0] = __ffma2_rn(f2, make_float2(xh.x, xh.y), S[n][0]);
                S[n][1] = __ffma2_rn(f3, make_float2(xh.z, xh.w), S[n][1]);
            }
        }
#pragma unroll
        for (int n = 0; n < NCOL; ++n) {
            const float2 t2 = __fadd2_rn(S[n][0], S[n][1]);
            acc[n] = fmaf(d, (t2.x + t2.y) - cb[n * nb32 + (kb >> 5)], acc[n]);
        }
    }
}

// Q8_0: 8 blocks of 34 bytes (272 B). Code byte c (two's complement) XOR 0x80
// is c + 128; placed in the low byte under 0x4B000000 it reads 2^23 + c + 128,
// and one packed subtract of (2^23 + 128) leaves c exactly.
template <int NCOL>
__device__ __forceinline__ void unit_q8_0(const uint8_t* u, const float* xs, const float*, int K, int k0,
                                          float (&acc)[NCOL]) {
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
        float2 S[NCOL][2];
#pragma unroll
        for (int n = 0; n < NCOL; ++n) S[n][0] = S[n][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            float4 xv[NCOL];
#pragma unroll
            for (int n = 0; n < NCOL; ++n) xv[n] = *reinterpret_cast<const float4*>(xs + n * K + kb + i);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int b0 = o + 2 + i + 2 * h, b1 = b0 + 1;
                const float f0 = __int_as_float(static_cast<int>(
                    __byte_perm(w[b0 >> 2] ^ 0x80808080u, 0x4B000000u, 0x7650u | static_cast<unsigned>(b0 & 3))));
                const float f1 = __int_as_float(static_cast<int>(
                    __byte_perm(w[b1 >> 2] ^ 0x80808080u, 0x4B000000u, 0x7650u | static_cast<unsigned>(b1 & 3))));
                const float2 q = __fadd2_rn(make_float2(f0, f1), off);
#pragma unroll
                for (int n = 0; n < NCOL; ++n) {
                    const float2 xp = h ? make_float2(xv[n].z, xv[n].w) : make_float2(xv[n].x, xv[n].y);
                    S[n][h] = __ffma2_rn(q, xp, S[n][h]);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < NCOL; ++n) {
            const float2 t2 = __fadd2_rn(S[n][0], S[n][1]);
            acc[n] = fmaf(d, t2.x + t2.y, acc[n]);
        }
    }
}

template <int KIND, int NCOL>
__device__ __forceinline__ void unit(const uint8_t* u, const float* xs, const float* cb, int K, int k0,
                                     float (&acc)[NCOL]) {
    // the Q4_0 / Q8_0 decoders take eight blocks (a 16-byte multiple) at a time
    if constexpr (KIND == Q4_0 || KIND == Q8_0) {
        static_assert(SG<KIND>::UB % 8 == 0, "Q4_0 / Q8_0 units are whole groups of eight blocks");
#pragma unroll
        for (int h = 0; h < SG<KIND>::UB / 8; ++h) {
            if constexpr (KIND == Q4_0) unit_q4_0<NCOL>(u + h * 8 * 18, xs, cb, K, k0 + h * 256, acc);
            else unit_q8_0<NCOL>(u + h * 8 * 34, xs, cb, K, k0 + h * 256, acc);
        }
    } else {
        unit_generic<KIND, NCOL>(u, xs, cb, K, k0, acc);
    }
}

template <int KIND> __host__ __device__ constexpr int cb_floats(int K, int ncol) { return KIND == Q4_0 ? ncol * (K / 32) : 0; }
// Q4_0 stages the raw activations apart from the permuted copy.
template <int KIND> __host__ __device__ constexpr int raw_floats(int K, int ncol) { return KIND == Q4_0 ? ncol * K : 0; }

// Activation staging by the consumer threads, after the raw fp32 activations
// are in `raw` (bulk copy; nullptr = read them from global memory). Q4_0
// permutes each block into decode order (a permutation within 32 words, so a
// warp's stores hit 32 distinct banks) and stores 136 * (sum of the block) in
// cb, one block per thread with a lane-rotated walk (conflict-free); the other
// formats keep the natural order.
template <int KIND, int NCOL>
__device__ void stage_x(const GemvArgs& a, float* xs, float* cb, const float* raw, int tid, int nthr) {
    const int K = a.K;
    auto xval = [&](int n, int k) -> float {
        if (n >= a.ncols) return 0.f;
        return raw ? raw[n * K + k] : load_x(a.X, a.x_dtype, static_cast<int64_t>(n) * K + k);
    };
    if constexpr (KIND == Q4_0) {
        for (int n = 0; n < NCOL; ++n)
            for (int k = tid; k < K; k += nthr) {
                const int b = k >> 5, e = k & 31;
                xs[n * K + 32 * b + q4_slot(e, (b & 1) == 0)] = xval(n, k);
            }
        const int nb = K / 32;
        for (int i = tid; i < NCOL * nb; i += nthr) {
            const int n = i / nb, b = i - n * nb;
            float sum = 0.f;
            for (int e = 0; e < 32; ++e) sum += xval(n, 32 * b + ((e + tid) & 31));
            cb[i] = 136.f * sum;
        }
    } else {
        for (int n = 0; n < NCOL; ++n)
            for (int k = tid; k < K; k += nthr) {
                if (raw && n < a.ncols) continue;   // already in place
                xs[n * K + k] = xval(n, k);
            }
    }
}

// Shared-memory layout of one CTA.
template <int KIND, int NCOL>
struct Smem {
    uint8_t* stage0;
    float* xs;
    float* cb;
    float* raw;        // bulk-copy target of the activations
    float* red;        // [2][NCOL][NW][32]
    uint64_t* full;    // [kMaxStages]
    uint64_t* empty;   // [kMaxStages]
    uint64_t* red_full;   // [2]
    uint64_t* red_empty;  // [2]
    uint64_t* x_full;
    int* abort_flag;

    __host__ __device__ static size_t bytes(int K, int stages) {
        using G = SGeo<KIND>;
        size_t b = static_cast<size_t>(stages) * G::STAGE_B;
        b += sizeof(float) * (static_cast<size_t>(NCOL) * K + cb_floats<KIND>(K, NCOL) + raw_floats<KIND>(K, NCOL) +
                              2 * NCOL * G::NW * 32);
        b = (b + 7) & ~size_t(7);
        b += (2 * kMaxStages + 5) * sizeof(uint64_t) + 16;
        return b;
    }

    __device__ Smem(uint8_t* base, int K, int stages) {
        using G = SGeo<KIND>;
        stage0 = base;
        xs = reinterpret_cast<float*>(base + stages * G::STAGE_B);
        cb = xs + NCOL * K;
        raw = raw_floats<KIND>(K, NCOL) ? cb + cb_floats<KIND>(K, NCOL) : xs;
        red = cb + cb_floats<KIND>(K, NCOL) + raw_floats<KIND>(K, NCOL);
        full = reinterpret_cast<uint64_t*>(
            (reinterpret_cast<uintptr_t>(red + 2 * NCOL * G::NW * 32) + 7) & ~static_cast<uintptr_t>(7));
        empty = full + kMaxStages;
        red_full = empty + kMaxStages;
        red_empty = red_full + 2;
        x_full = red_empty + 2;
        abort_flag = reinterpret_cast<int*>(x_full + 1);
    }
};

template <int KIND, int NCOL>
__global__ void __launch_bounds__((SG<KIND>::NW + 1) * 32) k_gemv(GemvArgs a) {
    using G = SGeo<KIND>;
    constexpr int NW = G::NW;
    extern __shared__ __align__(128) uint8_t smem[];
    const int K = a.K;
    Smem<KIND, NCOL> sm(smem, K, a.stages);
    volatile int* abort_flag = sm.abort_flag;

    // Let the next kernel on the stream start its set-up as our CTAs retire.
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], NW);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(&sm.red_full[p], NW);
            mbar_init(&sm.red_empty[p], 1);
        }
        mbar_init(sm.x_full, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int64_t ngroups = (a.M + kRows - 1) / kRows;
    const int nchunks = (K + G::CHUNK_E - 1) / G::CHUNK_E;
    const int ST = a.stages;
    const bool bulk_x = (a.flags & kFlagBulkX) != 0;

    if (warp == NW) {
        // ---------------- producer warp ----------------
        const uint64_t pol = l2_evict_first_policy();
        int it = 0;
        bool waited = false;
        if (!(a.flags & kFlagPrefetchW)) {
            grid_dep_wait();
            waited = true;
        }
        for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
            const int rows = static_cast<int>(imin64(kRows, a.M - g * kRows));
            const uint8_t* wg = a.W + static_cast<size_t>(g * kRows) * a.row_bytes;
            for (int kc = 0; kc < nchunks; ++kc, ++it) {
                const int s = it % ST, use = it / ST;
                if (use > 0 && !waited) {
                    // all prefetched stages are issued: now the activations
                    grid_dep_wait();
                    waited = true;
                    if (bulk_x && lane == 0) {
                        const uint32_t xb = static_cast<uint32_t>(a.ncols) * K * 4u;
                        mbar_arrive_expect_tx(sm.x_full, xb);
                        bulk_g2s(sm.raw, a.X, xb, sm.x_full);
                    }
                }
                if (use > 0 && !mbar_wait(&sm.empty[s], (use - 1) & 1, abort_flag, a.err)) goto drain;
                const int units = min(NW, (K - kc * G::CHUNK_E) / G::UNIT_E);
                const uint32_t bytes = static_cast<uint32_t>(units * G::UNIT_B);
                if (lane == 0) mbar_arrive_expect_tx(&sm.full[s], static_cast<uint32_t>(rows) * bytes);
                __syncwarp();
                if (lane < rows)
                    bulk_g2s_hint(sm.stage0 + s * G::STAGE_B + lane * G::STRIDE,
                                  wg + static_cast<size_t>(lane) * a.row_bytes + static_cast<size_t>(kc) * G::CHUNK_B,
                                  bytes, &sm.full[s], pol);
                if (waited && it == 0 && bulk_x && lane == 0) {
                    const uint32_t xb = static_cast<uint32_t>(a.ncols) * K * 4u;
                    mbar_arrive_expect_tx(sm.x_full, xb);
                    bulk_g2s(sm.raw, a.X, xb, sm.x_full);
                }
            }
        }
        if (!waited) {
            // every stage fit in the prefetch window
            grid_dep_wait();
            waited = true;
            if (bulk_x && lane == 0) {
                const uint32_t xb = static_cast<uint32_t>(a.ncols) * K * 4u;
                mbar_arrive_expect_tx(sm.x_full, xb);
                bulk_g2s(sm.raw, a.X, xb, sm.x_full);
            }
        }
    drain:
        // Before the CTA can retire, every issued copy must have landed: wait
        // (bounded, ignoring the abort flag) for the last phase of each stage
        // and for the activation copy.
        {
            const int issued = it;
            for (int s = 0; s < ST && s < issued; ++s) {
                const int last_use = (issued - 1 - s) / ST;  // uses of slot s: it = s + ST*use
                const long long t0 = clock64();
                while (!mbar_try_wait(&sm.full[s], last_use & 1)) {
                    if (clock64() - t0 > (1ll << 31)) {
                        atomicOr(a.err, DEV_ERR_TIMEOUT);
                        break;
                    }
                }
            }
            if (bulk_x && waited) {
                const long long t0 = clock64();
                while (!mbar_try_wait(sm.x_full, 0)) {
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
    if (bulk_x) {
        if (!mbar_wait(sm.x_full, 0, abort_flag, a.err)) *abort_flag = 1;
    }
    stage_x<KIND, NCOL>(a, sm.xs, sm.cb, bulk_x ? sm.raw : nullptr, threadIdx.x, NW * 32);
    named_bar_sync(1, NW * 32);

    int it = 0, gi = 0;
    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x, ++gi) {
        float acc[NCOL];
#pragma unroll
        for (int n = 0; n < NCOL; ++n) acc[n] = 0.f;
        for (int kc = 0; kc < nchunks; ++kc, ++it) {
            const int s = it % ST, use = it / ST;
            const bool ok = !*abort_flag && mbar_wait(&sm.full[s], use & 1, abort_flag, a.err);
            const int units = min(NW, (K - kc * G::CHUNK_E) / G::UNIT_E);
            if (ok && warp < units)
                unit<KIND, NCOL>(sm.stage0 + s * G::STAGE_B + lane * G::STRIDE + warp * G::UNIT_B, sm.xs, sm.cb, K,
                                 kc * G::CHUNK_E + warp * G::UNIT_E, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
        // Cross-warp sum through shared memory: every warp deposits its partial
        // sums and arrives; the group's writer warp (rotating) waits, adds and
        // stores, then frees the buffer. Only the writer waits.
        const int p = gi & 1, use = gi >> 1;
        float* rb = sm.red + p * NCOL * NW * 32;
        if (use > 0 && !*abort_flag) mbar_wait(&sm.red_empty[p], (use - 1) & 1, abort_flag, a.err);
#pragma unroll
        for (int n = 0; n < NCOL; ++n) rb[(n * NW + warp) * 32 + lane] = acc[n];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.red_full[p]);
        if (warp == gi % NW) {
            const bool ok = !*abort_flag && mbar_wait(&sm.red_full[p], use & 1, abort_flag, a.err);
            const int64_t row = g * kRows + lane;
            if (ok && row < a.M) {
#pragma unroll
                for (int n = 0; n < NCOL; ++n) {
                    if (n < a.ncols) {
                        float v = 0.f;
#pragma unroll
                        for (int w = 0; w < NW; ++w) v += rb[(n * NW + w) * 32 + lane];
                        a.Y[static_cast<int64_t>(n) * a.M + row] = v;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.red_empty[p]);
        }
    }
}

// Two CTAs per SM: each CTA gets up to half of the SM's shared memory.
constexpr int kCtaSmem = 113 * 1024;

// Launch tunables, overridable for sweeps: QMM_GEMV_STAGES (2..4) and
// QMM_GEMV_CTAS (CTAs per SM, 1 or 2). 0 = automatic.
int env_int(const char* name) {
    const char* v = getenv(name);
    return v ? atoi(v) : 0;
}
const int kEnvStages = env_int("QMM_GEMV_STAGES");
const int kEnvCtas = env_int("QMM_GEMV_CTAS");

template <int KIND>
bool ok_kind(const Problem& p) {
    using G = SGeo<KIND>;
    if (p.x_row) return false;
    if (p.N > 8 || p.K > (1 << 24)) return false;
    if (p.row_bytes % 16 || reinterpret_cast<uintptr_t>(p.W) % 16) return false;
    if (p.K % G::UNIT_E) return false;
    if (!G::PARTIAL_OK && p.K % G::CHUNK_E) return false;
    const int K = static_cast<int>(p.K);
    if (p.N <= 1) return Smem<KIND, 1>::bytes(K, 2) <= kSmemBudget;
    if (p.N <= 2) return Smem<KIND, 2>::bytes(K, 2) <= kSmemBudget;
    if (p.N <= 4) return Smem<KIND, 4>::bytes(K, 2) <= kSmemBudget;
    return Smem<KIND, 8>::bytes(K, 2) <= kSmemBudget;
}

template <int KIND, int NCOL>
cudaError_t launch_ncol(const Problem& p, cudaStream_t s) {
    using G = SGeo<KIND>;
    const int K = static_cast<int>(p.K);
    // Prefer two CTAs per SM (more warps to hide latency); otherwise one CTA
    // with as many stages as fit.
    // Formats with 8 consumer warps fill an SM with one deep CTA; 4-warp
    // formats run two CTAs per SM (measured on the decode workload).
    int stages = kMaxStages, per_sm = 2;
    while (stages > 2 && Smem<KIND, NCOL>::bytes(K, stages) > kCtaSmem) --stages;
    const bool one_cta = kEnvCtas == 1 || (kEnvCtas != 2 && G::NW >= 8);
    if (one_cta || Smem<KIND, NCOL>::bytes(K, stages) > kCtaSmem) {
        per_sm = 1;
        stages = kMaxStages;
        while (stages > 2 && Smem<KIND, NCOL>::bytes(K, stages) > kSmemBudget) --stages;
    }
    if (kEnvStages >= 2 && kEnvStages <= kMaxStages &&
        Smem<KIND, NCOL>::bytes(K, kEnvStages) <= (per_sm == 2 ? kCtaSmem : kSmemBudget))
        stages = kEnvStages;
    const size_t smem = Smem<KIND, NCOL>::bytes(K, stages);
    auto kern = k_gemv<KIND, NCOL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t ngroups = (p.M + kRows - 1) / kRows;
    const int grid = static_cast<int>(imin64(ngroups, static_cast<int64_t>(per_sm) * sm_count(dev)));
    GemvArgs a;
    a.W = p.W;
    a.row_bytes = p.row_bytes;
    a.M = p.M;
    a.K = K;
    a.X = p.X;
    a.x_dtype = p.x_dtype;
    a.ncols = static_cast<int>(p.N);
    a.Y = p.Y;
    a.stages = stages;
    a.err = p.err;
    a.flags = (weight_prefetch() ? kFlagPrefetchW : 0) |
              ((p.x_dtype == 0 && reinterpret_cast<uintptr_t>(p.X) % 16 == 0) ? kFlagBulkX : 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((G::NW + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    count_launch(1);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int KIND>
void run(const Problem& p, cudaStream_t s, cudaError_t* e) {
    if (p.N <= 1) *e = launch_ncol<KIND, 1>(p, s);
    else if (p.N <= 2) *e = launch_ncol<KIND, 2>(p, s);
    else if (p.N <= 4) *e = launch_ncol<KIND, 4>(p, s);
    else *e = launch_ncol<KIND, 8>(p, s);
}

template <int KIND>
void ok_dispatch(const Problem& p, bool* out) { *out = ok_kind<KIND>(p); }

}  // namespace

bool gemv_stream_ok(const Problem& p) {
    bool ok = false;
    QMM_DISPATCH_KIND(p.kind, ok_dispatch, p, &ok);
    return ok;
}

cudaError_t launch_gemv_stream(const Problem& p, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    QMM_DISPATCH_KIND(p.kind, run, p, s, &e);
    return e;
}

}  // namespace qmm
