// k_gemm_tc.cu -- quantized prefill GEMM on the 5th-generation tensor cores.
//
// Y[n * M + m] = sum_k W[m, k] * X[n * K + k]   (ferrox-cuda 0.21.0
// src/mul_mm.rs, `BODY_SRC`: the batched product whose K-loop that page runs
// as an fp32 FMA over shared tiles; here the contraction runs on tcgen05).
//
// One CTA computes a 128 (weight rows) x 128 (tokens) tile of Y:
//   * warp 0 (one thread) issues the TMA loads of the raw quantized bytes of
//     the tile's 128 rows for one 256-element super-step (a 2-D tensor map over
//     W, 16-byte aligned box) and, for the formats with mins, of the per-group
//     activation sums; warp 14 (one thread) loads the f16 activation sub-tiles
//     (128 tokens x 64 k, 128-byte swizzled, the K-major layout the MMA reads);
//   * warps 2-5 (one thread per weight row) decode the raw bytes in registers
//     into f16 INTEGER CODES -- the stored code times its integer sub-scale, or
//     the codebook value -- and store them straight into tensor memory (the
//     row's TMEM lane), plus the fp32 scales of the row into shared memory; in
//     the super-block kernel most formats add warps 16-19, a second decoder
//     set that takes every other super-step;
//   * warp 1 (one elected thread) issues tcgen05.mma kind::f16 with A = codes
//     from TMEM and B = activations from shared memory into fp32 TMEM
//     accumulators, one fresh accumulator per promotion unit;
//   * warps 6-13 read each finished unit from TMEM (tcgen05.ld) and apply the
//     fp32 scales to the PARTIAL SUMS: acc += d * D1 - dmin * D2 per 256-element
//     super-block (K-quants, IQ4_XS, and MXFP4 with its block exponents folded
//     into the operands) or acc += d * D per 32-element block (Q8_0, Q4_0,
//     Q5_0, IQ4_NL, Q4_1, Q5_1, Q8_1), then store Y.
// Keeping A in TMEM halves the shared-memory traffic per MMA (only B is read
// from shared memory) and spares the decoders the swizzled stores.
// The K-quant mins (-dmin * sum_s m_s * sum_{k in s} x_k) come out of a second,
// K = 16 (or 32) MMA per super-block: A = the integer mins, B = the per-group
// activation sums split hi + lo in f16 (a pre-pass kernel), into accumulator D2.
// Tile schedule: when the 128 x 128 tiles fill the SMs in whole waves, each
// CTA owns one tile. Otherwise (fewer tiles than SMs, or a ragged last wave)
// one CTA per SM takes an equal share of the flattened (tile, super-step)
// sequence: a CTA may end one tile's K range and begin the next one's; whole
// tiles go straight to Y, parts to a partial-tile workspace that a second
// kernel (k_tile_fixup) adds up in CTA order -- deterministic, and no CTA
// ever waits for another.
// Every wait is bounded (about a second); a timeout latches DEV_ERR_TIMEOUT and
// the CTA unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <mutex>

#include "decode.cuh"
#include "qmm.h"
#include "qmm_internal.cuh"
#include "sm100_async.cuh"
#include "tc_fastdec.cuh"

namespace qmm {
namespace {

constexpr int BM = 128, BN = 128, KSUP = 256, KSUB = 64;
static_assert(KSUB == 64, "a sub-step is four K = 16 MMAs: two 32-element blocks");
constexpr int kProdWarp = 0, kMmaWarp = 1, kNumDec = 4, kEpi0 = 6, kNumEpi = 8;   // decoders: warps 2-5
constexpr int kXWarp = kEpi0 + kNumEpi;           // activation-tile producer
constexpr int kWaitWarp = kXWarp + 1;             // waits on behalf of the MMA issuer
constexpr int kThreads = (kWaitWarp + 1) * 32;    // 512
// The super-block kernel decodes with one or two sets of four decoder warps
// (the second set, warps 16-19, takes the odd super-steps). Measured on the
// prefill workloads: two sets 10-19 % faster for Q5_K, Q6_K, Q3_K, IQ4_XS
// and MXFP4, 4 % for Q2_K, 5 % slower for Q4_K.
template <int KIND> struct DecSets { static constexpr int N = KIND == Q4_K ? 1 : 2; };
template <int KIND> struct SBThreads { static constexpr int V = kThreads + (DecSets<KIND>::N - 1) * 128; };
constexpr int kBarHand = 1;                       // named barriers 1, 2: waiter -> issuer hand-over
constexpr int X_SUB = BN * KSUB * 2;              // 16 KB: one 64-wide activation sub-tile
constexpr int X_TILE = 2 * X_SUB;                 // an activation stage holds two sub-steps
constexpr int MIN_TILE = 128 * 32;                // 4 KB, 32B-swizzled K-major (K = 16)
constexpr int kTmemCols = 512;
// Tensor memory (512 columns x 128 lanes, lane = weight row of the tile):
//   [0, 128)    A operand: four stages of 64 f16 codes per row (32 columns each)
//   [128, 512)  fp32 accumulators: three 128-column units, one per 32-element
//               block, for the per-32 formats (two, and the min term D2 of the
//               super-step at 384, for Q4_1 / Q5_1); otherwise D1 of two
//               super-blocks (double buffered) at 128 and 256, and the min
//               term D2 at 384.
constexpr int kAStages = 4;
constexpr int kACols = KSUB / 2;
constexpr int kDCol0 = kAStages * kACols;
// (per-32 formats with mins: two units, the min term D2 at column 384)
template <int KIND> struct NDBuf { static constexpr int N = TcGeo<KIND>::PER32 && !TcGeo<KIND>::MINS ? 3 : 2; };
// instruction descriptor: D f32, A/B f16, both K-major, N = 128, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((BN >> 3) << 17) | ((BM >> 4) << 24);

constexpr int gcd16(int v) { return (v % 16 == 0) ? 16 : (v % 8 == 0) ? 8 : (v % 4 == 0) ? 4 : (v % 2 == 0) ? 2 : 1; }

template <int KIND> struct Raw {
    static constexpr int SBB = (KSUP / Geo<KIND>::BE) * Geo<KIND>::BB;  // bytes of one super-step of a row
    static constexpr int MIS = (SBB % 16 == 0) ? 0 : 16 - gcd16(SBB);   // largest start offset in a 16-B line
    static constexpr int B0 = ((SBB + MIS + 15) / 16) * 16;
    static constexpr int BOXB = ((B0 / 16) % 2 == 1) ? B0 : B0 + 16;    // odd number of 16-B lines per row
    static constexpr int STAGE = BM * BOXB;
    static_assert(BOXB / 2 <= 256, "TMA box inner dimension");
};

template <int KIND> struct Mins;

// Shared-memory pipeline depths per format: X stages (activation sub-tiles) and
// raw stages (quantized bytes per super-step), as deep as the 227 KB allow --
// TMA latency must be covered by the stages in flight. (The decoded A stages
// live in tensor memory.)
template <int KIND> struct Stages {
    static constexpr int RAWB = 128 * Raw<KIND>::BOXB;
    static constexpr int MINS = Mins<KIND>::TILES * 4096 * 4;   // amin + bmin, double buffered
    static constexpr int FIXED = MINS + 2 * 128 * 8 * 4 + 2048 + 1024;
    static constexpr int BUDGET = 226 * 1024 - FIXED;
    static constexpr int AS = kAStages;
    static constexpr int RS = (BUDGET - 3 * X_TILE) >= 4 * RAWB ? 4 : (BUDGET - 3 * X_TILE) >= 3 * RAWB ? 3 : 2;
    static constexpr int XS0 = (BUDGET - RS * RAWB) / X_TILE;
    static constexpr int XS = XS0 > 4 ? 4 : XS0;
    static_assert(XS >= 3, "shared memory for at least three activation stages");
};

template <int KIND> struct Mins {
    static constexpr bool ON = TcGeo<KIND>::MINS;
    static constexpr int G = TcGeo<KIND>::MIN_GROUPS;       // groups per super-block
    static constexpr int KMW = 2 * G;                        // hi + lo activation sums per super-block
    static constexpr int TILES = ON ? KMW / 16 : 0;          // K = 16 MMAs per super-block
};

struct TcArgs {
    int M, N, K, nsup;   // N: activation rows the MMAs see (2 per token in pair mode)
    int tiles_m;      // tiles along M; tile t is (t % tiles_m, t / tiles_m)
    int wq, wr;       // shared super-steps: work = tiles * nsup = wq * G + wr (work < 2^31)
    float* Y;
    int y_dtype;      // 0 fp32, 1 f16, 2 bf16
    // pair mode (fp32 activations): activation rows 2n and 2n + 1 are the f16
    // high and low parts of token n scaled by 2^s_n; Y[n] = (column 2n +
    // column 2n + 1) * inv_scale[n]. Only with one tile per CTA.
    int pair;
    int ntok;
    const float* inv_scale;
    float* part;      // shared tiles: [CTA][2][BN][BM] fp32 partial tiles, or null (one tile per CTA)
    unsigned* err;
};

// The CTA's share of the flattened (tile, super-step) sequence. Without a
// partial-tile workspace the grid is (tiles_m, tiles_n) and each CTA takes
// its own tile's super-steps; with one, the grid is one-dimensional and CTA b
// takes steps [b * work / G, (b + 1) * work / G), so that every SM gets the
// same number of super-steps whatever the tile count (a tile's steps may be
// shared by consecutive CTAs, whose partial sums a second kernel adds up).
// 32-bit arithmetic only: a 64-bit division is a subroutine call whose
// register saves spill in this kernel.
struct Span {
    int t0, s0, n;    // first tile (-1: the CTA's own tile), its first super-step, steps
};
__device__ __forceinline__ Span cta_span(const TcArgs& a) {
    if (!a.part) return {-1, 0, a.nsup};
    const int b = blockIdx.x, G = gridDim.x;
    const int lo = b * a.wq + (b * a.wr) / G;               // floor(b * work / G)
    const int hi = (b + 1) * a.wq + ((b + 1) * a.wr) / G;
    return {lo / a.nsup, lo % a.nsup, hi - lo};
}

// The end of the CTA's part of tile t: a whole tile goes to Y (token-major,
// ragged edges clipped), a part to the CTA's partial slot -- 0 for the tile
// it began in, 1 for the tile it ends in. The epilogue thread holds row r,
// columns half * 64 + [0, 64).
__device__ __forceinline__ void store_tile(const TcArgs& a, const Span& sp, int t, bool whole, int half, int r,
                                           const float2 (&acc)[32]) {
    float* dst;
    int64_t stride;
    int lim;
    if (whole) {
        const int m0 = sp.t0 < 0 ? static_cast<int>(blockIdx.x) * BM : (t % a.tiles_m) * BM;
        const int n0 = (sp.t0 < 0 ? static_cast<int>(blockIdx.y) : t / a.tiles_m) * BN + half * 64;
        const int m = m0 + r;
        if (a.pair) {
            // columns 2i, 2i + 1 of this thread are the two parts of token n0 / 2 + i
            const int tok0 = n0 >> 1;
            const int tl = m < a.M ? min(32, a.ntok - tok0) : 0;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < tl)
                    store_y(a.Y, a.y_dtype, static_cast<int64_t>(tok0 + i) * a.M + m,
                            (acc[i].x + acc[i].y) * a.inv_scale[tok0 + i]);
            return;
        }
        lim = m < a.M ? min(64, a.N - n0) : 0;
        if (a.y_dtype != 0) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
                if (i < lim)
                    store_y(a.Y, a.y_dtype, static_cast<int64_t>(n0 + i) * a.M + m,
                            (i & 1) ? acc[i >> 1].y : acc[i >> 1].x);
            return;
        }
        dst = a.Y + static_cast<int64_t>(n0) * a.M + m;
        stride = a.M;
    } else {
        const int slot = (t == sp.t0) ? 0 : 1;
        dst = a.part + (static_cast<int64_t>(blockIdx.x * 2 + slot) * BN + half * 64) * BM + r;
        stride = BM;
        lim = 64;
    }
#pragma unroll
    for (int i = 0; i < 64; ++i)
        if (i < lim) dst[i * stride] = (i & 1) ? acc[i >> 1].y : acc[i >> 1].x;
}

// Walks the CTA's steps in order: tile t (rows m0.., tokens n0..) and the
// super-step s within the tile's K (divisions only when the tile changes).
struct Step {
    int t, s, m0, n0;
    __device__ __forceinline__ Step(const TcArgs& a, const Span& sp) {
        if (sp.t0 < 0) {
            t = 0;
            s = 0;
            m0 = blockIdx.x * BM;
            n0 = blockIdx.y * BN;
        } else {
            t = sp.t0;
            s = sp.s0;
            corner(a);
        }
    }
    __device__ __forceinline__ void corner(const TcArgs& a) {
        m0 = (t % a.tiles_m) * BM;
        n0 = (t / a.tiles_m) * BN;
    }
    __device__ __forceinline__ void next(const TcArgs& a) {
        if (++s == a.nsup) {
            s = 0;
            ++t;
            corner(a);
        }
    }
};

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// shared-memory matrix descriptors (sm_100 format, version 1), K-major
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFF) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ uint64_t desc_sw32(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFF) >> 4) | (1ull << 16) | (static_cast<uint64_t>(256 >> 4) << 32) |
           (1ull << 46) | (6ull << 61);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// A operand from tensor memory, B from shared memory
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// 32 consecutive 32-bit columns of this thread's lane
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
        "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
        "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
// Named-barrier rendezvous of `nthreads` threads (whole warps) that also
// returns the AND of every participant's `v`.
__device__ __forceinline__ bool bar_red_and(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %2, 0;\n\t"
        "bar.red.and.pred q, %1, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(static_cast<uint32_t>(v)), "r"(nthreads)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }


// Bounded wait that also honours the CTA's abort flag; false = give up.
// A phase that has already completed is taken without touching the flag.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
    if (mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    return mbar_wait(bar, parity, abort, err);
}

// Polling variant for the waits on the critical path of the pipeline.
__device__ __forceinline__ bool spin_bar(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
    if (mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    // no nap between probes: the hand-over to the MMA issuer is on the
    // critical path (measured: the per-32 formats ran 10 % slower with a
    // 32 ns nap)
    return mbar_wait_poll(bar, parity, abort, err, 0u);
}

// The same for a whole warp: lane 0 alone polls the barrier (hundreds of
// polling lanes slow down every other barrier operation of the CTA, among
// them the MMA issuer's), __syncwarp orders the other lanes after its
// acquire, and the outcome is broadcast. All 32 lanes must call it.
template <bool SPIN = false>
__device__ __forceinline__ bool warp_wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
        ok = (SPIN ? spin_bar(bar, parity, abort, err) : wait_bar(bar, parity, abort, err)) ? 1 : 0;
    __syncwarp();
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Waits (bounded, ignoring abort) for the phase with `parity` of a barrier.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, unsigned* err) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > (1ll << 31)) {
            atomicOr(err, DEV_ERR_TIMEOUT);
            return;
        }
    }
}

// The 16 f16 min codes of one A_min tile row as eight f16x2 words, extracted
// with word-wide masks and shifts and made exact f16 by the 0x64 magic byte
// (1024 + m, minus 1024): Q4_K / Q5_K -- the 8 mins of the 12-byte scale field
// (bytes 4..7 low 6 bits; bytes 8..11 high nibble with the top 2 bits of bytes
// 4..7), twice; Q2_K -- the high nibbles of its 16 scale bytes; Q4_1 / Q5_1
// -- the f16 mins of the super-step's eight blocks themselves (bytes 2..3 of
// each block), twice. The fields are 4-byte aligned in the staged tile.
template <int KIND>
__device__ __forceinline__ void min_words(const uint8_t* row, uint32_t (&w)[8]) {
    const uint32_t m1024 = h2int(-1024);
    if constexpr (KIND == Q4_1 || KIND == Q5_1) {
        constexpr int BW = Geo<KIND>::BB / 4;
        const uint32_t* f = reinterpret_cast<const uint32_t*>(row);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w[i] = prmt(f[BW * 2 * i], f[BW * (2 * i + 1)], 0x7632u);
            w[4 + i] = w[i];
        }
    } else if constexpr (KIND == Q2_K) {
        const uint32_t* f = reinterpret_cast<const uint32_t*>(row);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t m4 = (f[i] >> 4) & 0x0F0F0F0Fu;
            w[2 * i] = hadd2_u(prmt(m4, kMagB, 0x4140u), m1024);
            w[2 * i + 1] = hadd2_u(prmt(m4, kMagB, 0x4342u), m1024);
        }
    } else {
        const uint32_t* f = reinterpret_cast<const uint32_t*>(row + 4);
        const uint32_t s1 = f[1], s2 = f[2];
        const uint32_t lo4 = s1 & 0x3F3F3F3Fu;
        const uint32_t hi4 = ((s2 >> 4) & 0x0F0F0F0Fu) | (((s1 >> 6) & 0x03030303u) << 4);
        w[0] = hadd2_u(prmt(lo4, kMagB, 0x4140u), m1024);
        w[1] = hadd2_u(prmt(lo4, kMagB, 0x4342u), m1024);
        w[2] = hadd2_u(prmt(hi4, kMagB, 0x4140u), m1024);
        w[3] = hadd2_u(prmt(hi4, kMagB, 0x4342u), m1024);
        w[4] = w[0];
        w[5] = w[1];
        w[6] = w[2];
        w[7] = w[3];
    }
}

template <int KIND>
struct Layout {
    using R = Raw<KIND>;
    using MN = Mins<KIND>;
    static constexpr int AS = Stages<KIND>::AS, XS = Stages<KIND>::XS, RS = Stages<KIND>::RS;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_RAW = OFF_X + XS * X_TILE;
    static constexpr int OFF_AMIN = (OFF_RAW + RS * R::STAGE + 1023) & ~1023;
    static constexpr int MINB = MN::TILES * MIN_TILE;
    static constexpr int OFF_BMIN = OFF_AMIN + 2 * MINB;
    static constexpr int OFF_SC = OFF_BMIN + 2 * MINB;               // [2][128][8] floats
    static constexpr int OFF_BAR = OFF_SC + 2 * BM * 8 * 4;
    // barriers: raw_full/empty[RS], a_full/empty[AS], x_full/empty[XS], amin_full/empty[2],
    // bmin_full/empty[2], d_full/empty[ND], sc_full/empty[2], done
    static constexpr int NBAR = 2 * RS + 2 * AS + 2 * XS + 4 + 4 + 2 * NDBuf<KIND>::N + 4 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16 + 1024;               // + alignment slack
};

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const __grid_constant__ CUtensorMap tmB, TcArgs a) {
    using R = Raw<KIND>;
    using MN = Mins<KIND>;
    using L = Layout<KIND>;
    constexpr bool PER32 = TcGeo<KIND>::PER32;
    constexpr int BB = Geo<KIND>::BB;
    constexpr int AS = L::AS, XS = L::XS, RS = L::RS;
    constexpr int ND = NDBuf<KIND>::N;

    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic on the shared array
    // so that every access below compiles to shared (not generic) loads/stores
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* x_tiles = smem + L::OFF_X;
    uint8_t* raw = smem + L::OFF_RAW;
    uint8_t* amin = smem + L::OFF_AMIN;
    uint8_t* bmin = smem + L::OFF_BMIN;
    float* sbuf = reinterpret_cast<float*>(smem + L::OFF_SC);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + RS;
    uint64_t* a_full = raw_empty + RS;
    uint64_t* a_empty = a_full + AS;
    uint64_t* x_full = a_empty + AS;
    uint64_t* x_empty = x_full + XS;
    uint64_t* amin_full = x_empty + XS;
    uint64_t* amin_empty = amin_full + 2;
    uint64_t* bmin_full = amin_empty + 2;
    uint64_t* bmin_empty = bmin_full + 2;
    uint64_t* d_full = bmin_empty + 2;
    uint64_t* d_empty = d_full + ND;
    uint64_t* sc_full = d_empty + ND;
    uint64_t* sc_empty = sc_full + 2;
    uint64_t* done = sc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the partial-tile fix-up that follows may be scheduled now; it waits for
    // this grid to finish before reading anything
    asm volatile("griddepcontrol.launch_dependents;" :::);

    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kNumDec);
        }
        for (int i = 0; i < AS; ++i) {
            mbar_init(&a_full[i], kNumDec);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < XS; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        for (int i = 0; i < ND; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kNumEpi);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&amin_full[i], kNumDec);
            mbar_init(&amin_empty[i], 1);
            mbar_init(&bmin_full[i], 1);
            mbar_init(&bmin_empty[i], 1);
            mbar_init(&sc_full[i], kNumDec);
            mbar_init(&sc_empty[i], kNumEpi);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // each role works out the CTA's span itself (kept out of the registers
    // live across the roles)
    if (warp == kProdWarp) {
        // ------------------------------------------------ TMA producer: weights (+ group sums)
        if (lane == 0) {
            const Span span = cta_span(a);
            const int nloc = span.n;
            int s_issued = 0;
            Step st(a, span);
            for (int s = 0; s < nloc; ++s, st.next(a)) {
                const int rs = s % RS;
                if (s >= RS && !wait_bar(&raw_empty[rs], ((s / RS) - 1) & 1, abort_flag, a.err)) break;
                mbar_arrive_expect_tx(&raw_full[rs], R::STAGE);
                tma2d(raw + rs * R::STAGE, &tmW, ((st.s * R::SBB) & ~15) / 2, st.m0, &raw_full[rs]);
                if constexpr (MN::ON) {
                    const int b = s & 1;
                    if (s >= 2 && !wait_bar(&bmin_empty[b], ((s >> 1) - 1) & 1, abort_flag, a.err)) {
                        s_issued = s + 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&bmin_full[b], L::MINB);
#pragma unroll
                    for (int t = 0; t < MN::TILES; ++t)
                        tma2d(bmin + b * L::MINB + t * MIN_TILE, &tmB, st.s * MN::KMW + 16 * t, st.n0,
                              &bmin_full[b]);
                }
                s_issued = s + 1;
            }
            // every issued copy must land before the CTA retires
            for (int s = (s_issued > RS ? s_issued - RS : 0); s < s_issued; ++s)
                drain_bar(&raw_full[s % RS], (s / RS) & 1, a.err);
            if constexpr (MN::ON)
                for (int s = (s_issued > 2 ? s_issued - 2 : 0); s < s_issued; ++s)
                    drain_bar(&bmin_full[s & 1], (s >> 1) & 1, a.err);
        }
    } else if (warp == kXWarp) {
        // ------------------------------------------------ TMA producer: activation sub-tiles
        if (lane == 0) {
            const Span span = cta_span(a);
            const int nloc = span.n;
            int sx = 0;
            constexpr int XPS = KSUP / KSUB / 2;         // stages of two sub-steps per super-step
            const int nx = nloc * XPS;
            Step st(a, span);
            for (; sx < nx; ++sx) {
                if (sx > 0 && sx % XPS == 0) st.next(a);
                const int k0 = (st.s * XPS + sx % XPS) * 2 * KSUB;
                const int xs = sx % XS;
                if (sx >= XS && !wait_bar(&x_empty[xs], ((sx / XS) - 1) & 1, abort_flag, a.err)) break;
                mbar_arrive_expect_tx(&x_full[xs], X_TILE);
                tma2d(x_tiles + xs * X_TILE, &tmX, k0, st.n0, &x_full[xs]);
                tma2d(x_tiles + xs * X_TILE + X_SUB, &tmX, k0 + KSUB, st.n0, &x_full[xs]);
            }
            for (int i = (sx > XS ? sx - XS : 0); i < sx; ++i) drain_bar(&x_full[i % XS], (i / XS) & 1, a.err);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The warp follows the schedule converged and lane 0 issues. It never
        // touches shared memory between MMAs (a shared-memory access queued
        // behind MMAs stalls for ~100 cycles): the waits are done by the
        // waiter warp, which hands each ready sub-step over through a named
        // barrier (bar.red also carries whether to go on).
        const int nloc = cta_span(a).n;
        // Shared-memory descriptors are built once: the activation stages are
        // 1024-byte aligned and end below 2^18, so the descriptor of base + o
        // is the base's plus o / 16 in its address field (no carry). Building
        // one in front of every MMA measured 94-118 cycles per MMA against
        // the 64 of one issued back to back.
        const uint64_t xdesc0 = desc_sw128(smem_u32(x_tiles));
        int sub = 0;
        int ub = 0;   // per-32 formats: accumulator of the sub-step's first 32-element block
        for (int s = 0; s < nloc; ++s) {
            for (int q = 0; q < KSUP / KSUB; ++q, ++sub) {
                const bool go = bar_red_and(kBarHand + (sub & 1), 64, true);
                if (go && lane == 0) {
                    tc_fence_after();
                    const int as = sub % AS, xs = (sub >> 1) % XS;
                    const uint32_t a_tm = tmem + as * kACols;
                    const uint64_t xd = xdesc0 + static_cast<uint32_t>((xs * X_TILE + (sub & 1) * X_SUB) >> 4);
                    if constexpr (PER32) {
                        const int b1 = (ub + 1 == ND) ? 0 : ub + 1;
                        const uint32_t d0 = tmem + kDCol0 + ub * BN, d1 = tmem + kDCol0 + b1 * BN;
                        tc_mma_ts(d0, a_tm, xd, kIdesc, 0u);
                        tc_mma_ts(d0, a_tm + 8, xd + 2, kIdesc, 1u);
                        tc_commit(&d_full[ub]);
                        tc_mma_ts(d1, a_tm + 16, xd + 4, kIdesc, 0u);
                        tc_mma_ts(d1, a_tm + 24, xd + 6, kIdesc, 1u);
                        if constexpr (MN::ON) {
                            // the super-step's min term, published with its last block
                            if (q == KSUP / KSUB - 1) {
                                const int b = s & 1;
#pragma unroll
                                for (int t = 0; t < MN::TILES; ++t)
                                    tc_mma(tmem + kDCol0 + 2 * BN,
                                           desc_sw32(smem_u32(amin + b * L::MINB + t * MIN_TILE)),
                                           desc_sw32(smem_u32(bmin + b * L::MINB + t * MIN_TILE)), kIdesc, t);
                                tc_commit(&amin_empty[b]);
                                tc_commit(&bmin_empty[b]);
                            }
                        }
                        tc_commit(&d_full[b1]);
                    } else {
                        const uint32_t d = tmem + kDCol0 + (s & 1) * BN;
#pragma unroll
                        for (int kk = 0; kk < KSUB / 16; ++kk)
                            tc_mma_ts(d, a_tm + 8 * kk, xd + 2 * kk, kIdesc, (q | kk) != 0);
                    }
                    tc_commit(&a_empty[as]);
                    if (sub & 1) tc_commit(&x_empty[xs]);
                    if constexpr (!PER32) {
                        if (q == KSUP / KSUB - 1) {
                            const int b = s & 1;
                            if constexpr (MN::ON) {
#pragma unroll
                                for (int t = 0; t < MN::TILES; ++t)
                                    tc_mma(tmem + kDCol0 + 2 * BN,
                                           desc_sw32(smem_u32(amin + b * L::MINB + t * MIN_TILE)),
                                           desc_sw32(smem_u32(bmin + b * L::MINB + t * MIN_TILE)), kIdesc, t);
                                tc_commit(&amin_empty[b]);
                                tc_commit(&bmin_empty[b]);
                            }
                            tc_commit(&d_full[b]);
                        }
                    }
                }
                if constexpr (PER32) ub = (ub + 2) % ND;
                __syncwarp();
            }
        }
        if (lane == 0) {
            // all MMAs issued by this thread are complete before TMEM is freed
            tc_commit(done);
            drain_bar(done, 0, a.err);
        }
        __syncwarp();
    } else if (warp == kWaitWarp) {
        // ------------------------------------------------------------ MMA waiter
        // Waits (lane 0, bounded) for everything sub-step `sub` needs -- its A
        // stage, its activation stage, free accumulators and, at the end of a
        // super-block, the mins tiles -- then releases it to the issuer. After
        // a failure it keeps handing over "stop" so both sides stay in step.
        const int nloc = cta_span(a).n;
        int sub = 0;
        bool ok = true;
        for (int s = 0; s < nloc; ++s) {
            for (int q = 0; q < KSUP / KSUB; ++q, ++sub) {
                if (lane == 0 && ok) {
                    const int as = sub % AS, xi = sub >> 1, xs = xi % XS;
                    ok = spin_bar(&a_full[as], (sub / AS) & 1, abort_flag, a.err);
                    if (ok && (sub & 1) == 0) ok = spin_bar(&x_full[xs], (xi / XS) & 1, abort_flag, a.err);
                    if constexpr (PER32) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int u = 8 * s + 2 * q + h;
                            if (ok && u >= ND) ok = spin_bar(&d_empty[u % ND], ((u / ND) - 1) & 1, abort_flag, a.err);
                        }
                        if constexpr (MN::ON) {
                            // D2 is free here: the epilogue reads it with the previous
                            // super-step's last block, which it has finished before
                            // the blocks waited for above
                            if (q == KSUP / KSUB - 1) {
                                const int b = s & 1;
                                if (ok) ok = spin_bar(&amin_full[b], (s >> 1) & 1, abort_flag, a.err);
                                if (ok) ok = spin_bar(&bmin_full[b], (s >> 1) & 1, abort_flag, a.err);
                            }
                        }
                    } else {
                        if (ok && q == 0 && s >= 2) ok = spin_bar(&d_empty[s & 1], ((s >> 1) - 1) & 1, abort_flag, a.err);
                        if constexpr (MN::ON) {
                            if (q == KSUP / KSUB - 1) {
                                const int b = s & 1;
                                if (ok) ok = spin_bar(&amin_full[b], (s >> 1) & 1, abort_flag, a.err);
                                if (ok) ok = spin_bar(&bmin_full[b], (s >> 1) & 1, abort_flag, a.err);
                                // D2 is single-buffered: the epilogue must be done with super-block s - 1
                                if (ok && s >= 1) ok = spin_bar(&d_empty[(s - 1) & 1], ((s - 1) >> 1) & 1, abort_flag, a.err);
                            }
                        }
                    }
                }
                bar_red_and(kBarHand + (sub & 1), 64, lane != 0 || ok);
            }
        }
    } else if (warp < kEpi0) {
        // ------------------------------------------------------------ decoders
        // weight row within the tile = the TMEM lane this warp may access
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const Span span = cta_span(a);
        const int nloc = span.n;
        int sub = 0;
        int ks = span.s0;   // super-step within the row
        for (int s = 0; s < nloc; ++s, ks = (ks + 1 == a.nsup) ? 0 : ks + 1) {
            const int rs = s % RS;
            bool ok = warp_wait_bar(&raw_full[rs], (s / RS) & 1, abort_flag, a.err);
            const uint8_t* row = raw + rs * R::STAGE + r * R::BOXB + ((ks * R::SBB) & 15);
            // scales for the epilogue
            if (ok && s >= 2) ok = warp_wait_bar(&sc_empty[s & 1], ((s >> 1) - 1) & 1, abort_flag, a.err);
            float* sc = sbuf + ((s & 1) * BM + r) * 8;
            if (ok) {
                if constexpr (PER32) {
#pragma unroll
                    for (int blk = 0; blk < 8; ++blk) sc[blk] = scale32<KIND>(row + blk * BB);
                } else {
                    const float2 dd = scale256<KIND>(row);
                    sc[0] = dd.x;
                    sc[1] = dd.y;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sc_full[s & 1]);
            if constexpr (MN::ON) {
                const int b = s & 1;
                if (ok && s >= 2) ok = warp_wait_bar(&amin_empty[b], ((s >> 1) - 1) & 1, abort_flag, a.err);
                if (ok) {
                    // A_min tile(s): 32B-swizzled K-major, 16 f16 per row per tile
                    // (every tile holds the same min codes: they meet the hi
                    // and the lo halves of the activation sums)
                    uint32_t w[8];
                    min_words<KIND>(row, w);
#pragma unroll
                    for (int t = 0; t < MN::TILES; ++t) {
                        uint8_t* tb = amin + b * L::MINB + t * MIN_TILE + (r >> 3) * 256 + (r & 7) * 32;
                        const int sw = (r >> 2) & 1;
                        *reinterpret_cast<uint4*>(tb + ((0 ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4*>(tb + ((1 ^ sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                    fence_proxy_async();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&amin_full[b]);
            }
            // Two sub-steps per pass: their decodes are independent instruction
            // streams the compiler interleaves (one decoder warp per scheduler
            // is latency-bound on a single stream); then each is stored and
            // published in order. Decode first, then wait for the stage to be
            // free, so the decode stays off the stage's round trip (ok is
            // warp-uniform: tcgen05.st is warp-collective).
            static_assert((KSUP / KSUB) % 2 == 0, "sub-steps are decoded in pairs");
            // K-quants: the super-block's integer sub-scales as f16, once
            uint32_t scw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if constexpr (FastDecPre<KIND>::ON) {
                if (ok) FastDec<KIND>::pre(row, scw);
            }
#pragma unroll 1
            for (int q = 0; q < KSUP / KSUB; q += 2) {
                uint32_t o[2][32];
                if (ok) {
                    if constexpr (FastDecPre<KIND>::ON) {
                        FastDec<KIND>::sub_pre(row, q, o[0], scw);
                        FastDec<KIND>::sub_pre(row, q + 1, o[1], scw);
                    } else {
                        FastDec<KIND>::sub(row, q, o[0]);
                        FastDec<KIND>::sub(row, q + 1, o[1]);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h, ++sub) {
                    const int as = sub % AS;
                    if (ok && sub >= AS)
                        ok = warp_wait_bar<true>(&a_empty[as], ((sub / AS) - 1) & 1, abort_flag, a.err);
                    if (ok) {
                        tc_fence_after();
                        tmem_st32(tmem + lane_addr + as * kACols, o[h]);
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[as]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[rs]);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kEpi0;
        const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
        const int half = ew >> 2;                  // column half: 64 columns each
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        float2 acc[32];   // columns 2i, 2i + 1 of this thread's 64, updated with packed FMAs
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.f, 0.f);
        const Span span = cta_span(a);
        const int nloc = span.n;
        // one segment per tile the CTA works on; the tile is stored after
        // its last super-step (the store sits outside the per-step loop: the
        // accumulators stay in registers)
        int et = span.t0, es = span.s0;   // the segment's tile and first super-step
        for (int s = 0; s < nloc;) {
            const int seg_end = min(nloc, s + a.nsup - es);
            const bool whole = es == 0 && seg_end - s == a.nsup;
            for (; s < seg_end; ++s) {
                const float* sc = sbuf + ((s & 1) * BM + r) * 8;
                warp_wait_bar(&sc_full[s & 1], (s >> 1) & 1, abort_flag, a.err);
                if constexpr (PER32) {
                    for (int j = 0; j < 8; ++j) {
                        const int u = 8 * s + j, b = u % ND;
                        const bool ok = warp_wait_bar(&d_full[b], (u / ND) & 1, abort_flag, a.err);
                        tc_fence_after();
                        const float2 d2 = make_float2(sc[j], sc[j]);
                        if (ok) {
#pragma unroll
                            for (int c = 0; c < 4; c += 2) {
                                float v[32];
                                tmem_ld16(tmem + lane_addr + kDCol0 + b * BN + half * 64 + c * 16,
                                          *reinterpret_cast<float(*)[16]>(v));
                                tmem_ld16(tmem + lane_addr + kDCol0 + b * BN + half * 64 + c * 16 + 16,
                                          *reinterpret_cast<float(*)[16]>(v + 16));
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    acc[c * 8 + i] = __ffma2_rn(d2, make_float2(v[2 * i], v[2 * i + 1]), acc[c * 8 + i]);
                                if constexpr (MN::ON) {
                                    // Q4_1 / Q5_1, with the super-step's last block: + the
                                    // min term sum_b m_b * (activation sum of block b)
                                    if (j == 7) {
                                        tmem_ld16(tmem + lane_addr + kDCol0 + 2 * BN + half * 64 + c * 16,
                                                  *reinterpret_cast<float(*)[16]>(v));
                                        tmem_ld16(tmem + lane_addr + kDCol0 + 2 * BN + half * 64 + c * 16 + 16,
                                                  *reinterpret_cast<float(*)[16]>(v + 16));
                                        tmem_wait_ld();
#pragma unroll
                                        for (int i = 0; i < 16; ++i)
                                            acc[c * 8 + i] = __fadd2_rn(acc[c * 8 + i], make_float2(v[2 * i], v[2 * i + 1]));
                                    }
                                }
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&d_empty[b]);
                    }
                } else {
                    const int b = s & 1;
                    const bool ok = warp_wait_bar(&d_full[b], (s >> 1) & 1, abort_flag, a.err);
                    tc_fence_after();
                    const float2 d2 = make_float2(sc[0], sc[0]), ndm2 = make_float2(-sc[1], -sc[1]);
                    if (ok) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            float v[16];
                            tmem_ld16(tmem + lane_addr + kDCol0 + b * BN + half * 64 + c * 16, v);
                            if constexpr (MN::ON) {
                                float w2[16];
                                tmem_ld16(tmem + lane_addr + kDCol0 + 2 * BN + half * 64 + c * 16, w2);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    acc[c * 8 + i] = __ffma2_rn(ndm2, make_float2(w2[2 * i], w2[2 * i + 1]),
                                                                __ffma2_rn(d2, make_float2(v[2 * i], v[2 * i + 1]),
                                                                           acc[c * 8 + i]));
                            } else {
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    acc[c * 8 + i] = __ffma2_rn(d2, make_float2(v[2 * i], v[2 * i + 1]), acc[c * 8 + i]);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&d_empty[b]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sc_empty[s & 1]);
            }
            if (!*abort_flag) store_tile(a, span, et, whole, half, r, acc);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.f, 0.f);
            es = 0;
            ++et;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// The formats with one fp32 scale per 256-element super-block (Q4_K, Q5_K,
// Q6_K, Q2_K, Q3_K, IQ4_XS, and MXFP4 through its exponent fold) run a leaner
// pipeline, k_gemm_sb. Its unit is a half-step: two sub-steps (K = 128, eight
// MMAs). Each half-step's MMAs end
// with ONE tcgen05.commit on the stage's `done` barrier, which releases at
// once everything the half-step read -- its A stage in tensor memory, its
// activation stage (and, on the second half of a super-step, the min-term
// tiles) -- and, on the second half, tells the epilogue that the super-step's
// accumulators are complete. Measured on a lone issuing thread, every commit
// costs the tensor pipe about 80 cycles (a group of four N = 128 MMAs takes
// 256); the per-sub-step kernel above commits seven to nine times per
// super-step, this one twice.
//
// Tensor memory (512 columns):
//   formats with mins: A stages [0, 128) (two of 64 columns), D1 double
//                      buffered at 128 and 256, the min term D2 at 384;
//   the others:        A stages [0, 256) (four), D1 at 256 and 384.
// A waiter on a barrier never falls two phases behind: the decoders and the
// activation producer refill a stage only after its previous use completed;
// the epilogue reads super-step s before the waiter lets the second half of
// super-step s + 1 issue (that half waits for the epilogue's d_empty of s).
// Half-step h's completion is signalled on done[h % 4] whatever the number of
// stages: with two A stages and two decoder sets, a stage's previous user is
// the other set, and a barrier per stage could then be two phases ahead of a
// set's last wait on it; with four barriers, every waiter for half-step h has
// itself seen h - 4 complete. Likewise, where the raw stages are odd in
// number, a decoder first waits until the other set has released its stage
// (raw_empty) before it waits for the stage's next load.
// ---------------------------------------------------------------------------
constexpr int kHalfSubs = 2;                   // sub-steps per half-step
constexpr int kACols2 = kHalfSubs * kACols;    // 64 TMEM columns per A stage
constexpr int X_HALF = kHalfSubs * X_SUB;      // 32 KB activation stage

template <int KIND> struct PipeSB {
    static constexpr bool MINS = Mins<KIND>::ON;
    static constexpr int NS = MINS ? 2 : 4;                   // stages (A in TMEM, X in SMEM)
    static constexpr int D1COL = NS * kACols2;                // 128 or 256
    static constexpr int D2COL = D1COL + 2 * BN;              // 384 (formats with mins)
    static constexpr int MINB = Mins<KIND>::TILES * MIN_TILE;
    static constexpr int RAWB = BM * Raw<KIND>::BOXB;
    static constexpr int SCD = 4;                             // scale buffers (super-steps in flight)
    static constexpr int NDONE = 4;                           // completion barriers, done[h % 4]
    static constexpr int FIXED = NS * X_HALF + 2 * MINB + SCD * BM * 2 * 4 + 2048;
    static constexpr int FREE = 226 * 1024 - FIXED;
    static constexpr int RS = FREE >= 4 * RAWB ? 4 : FREE >= 3 * RAWB ? 3 : 2;
    static_assert(FIXED + RS * RAWB <= 226 * 1024, "shared memory");
    static_assert(D1COL + 2 * BN <= kTmemCols && (!MINS || D2COL + BN <= kTmemCols), "tensor memory");
};

template <int KIND>
struct LayoutSB {
    using P = PipeSB<KIND>;
    static constexpr int OFF_X = 0;                                      // 1024-aligned stages
    static constexpr int OFF_RAW = OFF_X + P::NS * X_HALF;
    static constexpr int OFF_AMIN = (OFF_RAW + P::RS * P::RAWB + 1023) & ~1023;
    static constexpr int OFF_BMIN = OFF_AMIN + P::MINB;
    static constexpr int OFF_SC = OFF_BMIN + P::MINB;                    // [SCD][128][2] floats
    static constexpr int OFF_BAR = OFF_SC + P::SCD * BM * 2 * 4;
    // raw_full/empty[RS], a_full[NS], x_full[NS], done[NDONE], d_empty[2], sc_full/empty[SCD], fin
    static constexpr int NBAR = 2 * P::RS + 2 * P::NS + P::NDONE + 2 + 2 * P::SCD + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16 + 1024;                   // + alignment slack
};

template <int KIND>
__global__ void __launch_bounds__(SBThreads<KIND>::V, 1)
    k_gemm_sb(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const __grid_constant__ CUtensorMap tmB, TcArgs a) {
    using R = Raw<KIND>;
    using MN = Mins<KIND>;
    using P = PipeSB<KIND>;
    using L = LayoutSB<KIND>;
    static_assert(!TcGeo<KIND>::PER32, "super-block formats only");
    constexpr int NS = P::NS, RS = P::RS, SCD = P::SCD, NDONE = P::NDONE;
    static_assert(NDONE == 4 && NDONE % NS == 0, "done[h % 4]: each barrier belongs to one stage");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* x_tiles = smem + L::OFF_X;
    uint8_t* raw = smem + L::OFF_RAW;
    uint8_t* amin = smem + L::OFF_AMIN;
    uint8_t* bmin = smem + L::OFF_BMIN;
    float* sbuf = reinterpret_cast<float*>(smem + L::OFF_SC);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + RS;
    uint64_t* a_full = raw_empty + RS;
    uint64_t* x_full = a_full + NS;
    uint64_t* done = x_full + NS;
    uint64_t* d_empty = done + NDONE;   // [2]: the epilogue is done with super-step s (index s & 1)
    uint64_t* sc_full = d_empty + 2;
    uint64_t* sc_empty = sc_full + SCD;
    uint64_t* fin = sc_empty + SCD;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.launch_dependents;" :::);

    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kNumDec);
        }
        for (int i = 0; i < NS; ++i) {
            mbar_init(&a_full[i], kNumDec);
            mbar_init(&x_full[i], 1);
        }
        for (int i = 0; i < NDONE; ++i) mbar_init(&done[i], 1);
        for (int i = 0; i < 2; ++i) mbar_init(&d_empty[i], kNumEpi);
        for (int i = 0; i < SCD; ++i) {
            mbar_init(&sc_full[i], kNumDec);
            mbar_init(&sc_empty[i], kNumEpi);
        }
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProdWarp) {
        // ------------------------------------------------ TMA producer: raw weights
        if (lane == 0) {
            const Span span = cta_span(a);
            const int nloc = span.n;
            int s_issued = 0;
            Step st(a, span);
            for (int s = 0; s < nloc; ++s, st.next(a)) {
                const int rs = s % RS;
                if (s >= RS && !wait_bar(&raw_empty[rs], ((s / RS) - 1) & 1, abort_flag, a.err)) break;
                mbar_arrive_expect_tx(&raw_full[rs], R::STAGE);
                tma2d(raw + rs * R::STAGE, &tmW, ((st.s * R::SBB) & ~15) / 2, st.m0, &raw_full[rs]);
                s_issued = s + 1;
            }
            for (int s = (s_issued > RS ? s_issued - RS : 0); s < s_issued; ++s)
                drain_bar(&raw_full[s % RS], (s / RS) & 1, a.err);
        }
    } else if (warp == kXWarp) {
        // ------------------------------------------------ TMA producer: activations (+ their group sums)
        if (lane == 0) {
            const Span span = cta_span(a);
            const int nh = 2 * span.n;
            int h = 0;
            Step st(a, span);
            for (; h < nh; ++h) {
                const int half = h & 1, i = h % NS;
                if (h > 0 && half == 0) st.next(a);
                if (h >= NS && !wait_bar(&done[(h - NS) % NDONE], ((h - NS) / NDONE) & 1, abort_flag, a.err)) break;
                const int k0 = st.s * KSUP + half * kHalfSubs * KSUB;
                mbar_arrive_expect_tx(&x_full[i], X_HALF + ((MN::ON && half) ? P::MINB : 0));
                tma2d(x_tiles + i * X_HALF, &tmX, k0, st.n0, &x_full[i]);
                tma2d(x_tiles + i * X_HALF + X_SUB, &tmX, k0 + KSUB, st.n0, &x_full[i]);
                if constexpr (MN::ON) {
                    // the min term's activation sums ride with the super-step's
                    // second half (single buffer: the previous super-step's min
                    // MMA completed with the stage's previous use)
                    if (half) {
#pragma unroll
                        for (int t = 0; t < MN::TILES; ++t)
                            tma2d(bmin + t * MIN_TILE, &tmB, st.s * MN::KMW + 16 * t, st.n0, &x_full[i]);
                    }
                }
            }
            for (int j = (h > NS ? h - NS : 0); j < h; ++j) drain_bar(&x_full[j % NS], (j / NS) & 1, a.err);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Never touches shared memory between MMAs: the waiter warp hands each
        // ready half-step over through a named barrier.
        const int nh = 2 * cta_span(a).n;
        const uint64_t xdesc0 = desc_sw128(smem_u32(x_tiles));
        uint64_t adesc[MN::TILES > 0 ? MN::TILES : 1], bdesc[MN::TILES > 0 ? MN::TILES : 1];
#pragma unroll
        for (int t = 0; t < MN::TILES; ++t) {
            adesc[t] = desc_sw32(smem_u32(amin + t * MIN_TILE));
            bdesc[t] = desc_sw32(smem_u32(bmin + t * MIN_TILE));
        }
        for (int h = 0; h < nh; ++h) {
            const bool go = bar_red_and(kBarHand + (h & 1), 64, true);
            if (go && lane == 0) {
                tc_fence_after();
                const int i = h % NS, half = h & 1;
                const uint32_t a_tm = tmem + i * kACols2;
                const uint64_t xd = xdesc0 + static_cast<uint32_t>((i * X_HALF) >> 4);
                const uint32_t d = tmem + P::D1COL + ((h >> 1) & 1) * BN;
#pragma unroll
                for (int sub = 0; sub < kHalfSubs; ++sub)
#pragma unroll
                    for (int kk = 0; kk < KSUB / 16; ++kk)
                        tc_mma_ts(d, a_tm + sub * kACols + 8 * kk, xd + sub * (X_SUB >> 4) + 2 * kk, kIdesc,
                                  (half | sub | kk) != 0);
                if constexpr (MN::ON) {
                    if (half) {
#pragma unroll
                        for (int t = 0; t < MN::TILES; ++t) tc_mma(tmem + P::D2COL, adesc[t], bdesc[t], kIdesc, t);
                    }
                }
                tc_commit(&done[h % NDONE]);
            }
            __syncwarp();
        }
        if (lane == 0) {
            tc_commit(fin);
            drain_bar(fin, 0, a.err);
        }
        __syncwarp();
    } else if (warp == kWaitWarp) {
        // ------------------------------------------------------------ MMA waiter
        const int nh = 2 * cta_span(a).n;
        bool ok = true;
        for (int h = 0; h < nh; ++h) {
            if (lane == 0 && ok) {
                const int i = h % NS, u = h / NS, s = h >> 1;
                ok = spin_bar(&a_full[i], u & 1, abort_flag, a.err);
                if (ok) ok = spin_bar(&x_full[i], u & 1, abort_flag, a.err);
                if constexpr (MN::ON) {
                    // the second half of super-step s rewrites the (single) min
                    // term: the epilogue must be done with s - 1
                    if (ok && (h & 1) && s >= 1)
                        ok = spin_bar(&d_empty[(s - 1) & 1], ((s - 1) >> 1) & 1, abort_flag, a.err);
                } else {
                    // super-step s overwrites D1[s & 1]: the epilogue must be
                    // done with s - 2 (one super-step of slack for the epilogue)
                    if (ok && !(h & 1) && s >= 2)
                        ok = spin_bar(&d_empty[s & 1], ((s - 2) >> 1) & 1, abort_flag, a.err);
                }
            }
            bar_red_and(kBarHand + (h & 1), 64, lane != 0 || ok);
        }
    } else if (warp < kEpi0 || warp > kWaitWarp) {
        // ------------------------------------------------------------ decoders
        // set 0 (warps 2-5) and, with two sets, set 1 (warps 16-19) take
        // alternate super-steps; every barrier of a super-step still counts
        // the four warps of the one set that decodes it
        const int dset = warp > kWaitWarp ? 1 : 0, dstep = DecSets<KIND>::N;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const Span span = cta_span(a);
        const int nloc = span.n;
        for (int s = dset; s < nloc; s += dstep) {
            const int ks = static_cast<int>((static_cast<int64_t>(span.s0) + s) % a.nsup);   // super-step within the row
            const int rs = s % RS;
            bool ok = true;
            // the stage's previous load was decoded by the other set: its
            // release bounds raw_full's phase (see above)
            if (RS % dstep != 0 && s >= RS) ok = warp_wait_bar(&raw_empty[rs], ((s / RS) - 1) & 1, abort_flag, a.err);
            if (ok) ok = warp_wait_bar(&raw_full[rs], (s / RS) & 1, abort_flag, a.err);
            const uint8_t* row = raw + rs * R::STAGE + r * R::BOXB + ((ks * R::SBB) & 15);
            if (ok && s >= SCD) ok = warp_wait_bar(&sc_empty[s % SCD], ((s / SCD) - 1) & 1, abort_flag, a.err);
            if (ok) {
                const float2 dd = scale256<KIND>(row);
                float* sc = sbuf + ((s % SCD) * BM + r) * 2;
                sc[0] = dd.x;
                sc[1] = dd.y;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sc_full[s % SCD]);
            uint32_t scw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (ok) FastDec<KIND>::pre(row, scw);
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                const int h = 2 * s + half, i = h % NS;
                uint32_t o[kHalfSubs][32];
                if (ok) {
                    FastDec<KIND>::sub_pre(row, 2 * half, o[0], scw);
                    FastDec<KIND>::sub_pre(row, 2 * half + 1, o[1], scw);
                }
                // decode first, then wait for the stage, so the decode stays off
                // the stage's round trip (ok is warp-uniform: tcgen05.st is
                // warp-collective)
                if (ok && h >= NS) ok = warp_wait_bar<true>(&done[(h - NS) % NDONE], ((h - NS) / NDONE) & 1, abort_flag, a.err);
                if constexpr (MN::ON) {
                    if (half && ok) {
                        // A_min tile(s) of super-step s: 32B-swizzled K-major, 16 f16
                        // per row per tile (every tile holds the same min codes: they
                        // meet the hi and the lo halves of the activation sums)
                        uint32_t w[8];
                        min_words<KIND>(row, w);
#pragma unroll
                        for (int t = 0; t < MN::TILES; ++t) {
                            uint8_t* tb = amin + t * MIN_TILE + (r >> 3) * 256 + (r & 7) * 32;
                            const int sw = (r >> 2) & 1;
                            *reinterpret_cast<uint4*>(tb + ((0 ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4*>(tb + ((1 ^ sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                        fence_proxy_async();
                    }
                }
                if (ok) {
                    tc_fence_after();
                    tmem_st32(tmem + lane_addr + i * kACols2, o[0]);
                    tmem_st32(tmem + lane_addr + i * kACols2 + kACols, o[1]);
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[i]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[rs]);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kEpi0;
        const int quad = warp & 3;
        const int half = ew >> 2;                  // column half: 64 columns each
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        float2 acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.f, 0.f);
        const Span span = cta_span(a);
        const int nloc = span.n;
        int et = span.t0, es = span.s0;
        for (int s = 0; s < nloc;) {
            const int seg_end = min(nloc, s + a.nsup - es);
            const bool whole = es == 0 && seg_end - s == a.nsup;
            for (; s < seg_end; ++s) {
                const float* sc = sbuf + ((s % SCD) * BM + r) * 2;
                warp_wait_bar(&sc_full[s % SCD], (s / SCD) & 1, abort_flag, a.err);
                const int h = 2 * s + 1;
                const bool ok = warp_wait_bar(&done[h % NDONE], (h / NDONE) & 1, abort_flag, a.err);
                tc_fence_after();
                const float2 d2 = make_float2(sc[0], sc[0]), ndm2 = make_float2(-sc[1], -sc[1]);
                const uint32_t dcol = P::D1COL + (s & 1) * BN + half * 64;
                if (ok) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[16];
                        tmem_ld16(tmem + lane_addr + dcol + c * 16, v);
                        if constexpr (MN::ON) {
                            float w2[16];
                            tmem_ld16(tmem + lane_addr + P::D2COL + half * 64 + c * 16, w2);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                acc[c * 8 + i] = __ffma2_rn(ndm2, make_float2(w2[2 * i], w2[2 * i + 1]),
                                                            __ffma2_rn(d2, make_float2(v[2 * i], v[2 * i + 1]),
                                                                       acc[c * 8 + i]));
                        } else {
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                acc[c * 8 + i] = __ffma2_rn(d2, make_float2(v[2 * i], v[2 * i + 1]), acc[c * 8 + i]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&d_empty[s & 1]);
                    mbar_arrive(&sc_empty[s % SCD]);
                }
            }
            if (!*abort_flag) store_tile(a, span, et, whole, half, r, acc);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.f, 0.f);
            es = 0;
            ++et;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// The kernel for a format and its dynamic shared memory: the super-block
// pipeline for formats with one scale per 256 elements, the per-sub-step one
// for the per-32 formats.
using TcKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, TcArgs);
template <int KIND>
constexpr int tc_threads() {
    if constexpr (TcGeo<KIND>::PER32) return kThreads;
    else return SBThreads<KIND>::V;
}
template <int KIND>
TcKernel tc_kernel(int* smem_bytes) {
    if constexpr (TcGeo<KIND>::PER32) {
        *smem_bytes = Layout<KIND>::BYTES;
        return k_gemm_tc<KIND>;
    } else {
        *smem_bytes = LayoutSB<KIND>::BYTES;
        return k_gemm_sb<KIND>;
    }
}

// Per-group activation sums for the min term: out[n][s][0..G) = hi, [G..2G) = lo
// with hi = f16(sum), lo = f16(sum - hi); groups of 32 (Q4_K, Q5_K, Q4_1, Q5_1) or 16 (Q2_K).
// One thread per group, reading its 16 or 32 halves with 16-byte loads (the
// rows of X are 16-byte aligned and K is a multiple of 256).
__global__ void k_xsums(const __half* __restrict__ X, int N, int K, int gsize, int G, __half* __restrict__ out) {
    const int ngroups = K / gsize;
    const int64_t total = static_cast<int64_t>(N) * ngroups;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(i / ngroups), g = static_cast<int>(i % ngroups);
        const uint4* x = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(n) * K + static_cast<int64_t>(g) * gsize);
        uint4 v[4];
        const int nv = gsize / 8;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (j < nv) v[j] = __ldg(x + j);
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < nv) {
                const __half2* h = reinterpret_cast<const __half2*>(&v[j]);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 f = __half22float2(h[t]);
                    sum += f.x;
                    sum += f.y;
                }
            }
        }
        const __half hi = __float2half_rn(sum);
        const __half lo = __float2half_rn(sum - __half2float(hi));
        const int s = g / G, gi = g % G;
        __half* o = out + (static_cast<int64_t>(n) * (K / KSUP) + s) * (2 * G);
        o[gi] = hi;
        o[G + gi] = lo;
    }
}

// Adds up the partial tiles of the tiles whose super-steps were shared by
// several CTAs, in CTA order, and writes them to Y (the CTA that covers a
// whole tile has already written it). Grid (tiles, kFixSplit): each thread
// takes four consecutive rows of one token of the tile, a float4 of every
// partial that covers it.
constexpr int kFixThreads = 256;
constexpr int kFixSplit = BM * BN / 4 / kFixThreads;
__global__ void __launch_bounds__(kFixThreads) k_tile_fixup(const float* __restrict__ part, float* __restrict__ Y,
                                                            int M, int N, int tiles_m, int nsup, int64_t work,
                                                            int G, int y_dtype) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int t = blockIdx.x;
    // CTA b covers steps [b * work / G, (b + 1) * work / G): step g lies in CTA ((g + 1) * G - 1) / work
    const int64_t g0 = static_cast<int64_t>(t) * nsup, g1 = g0 + nsup - 1;
    const int b0 = static_cast<int>(((g0 + 1) * G - 1) / work), b1 = static_cast<int>(((g1 + 1) * G - 1) / work);
    if (b0 == b1) return;
    // the first CTA holds the tile in slot 0 if it began at the tile's first
    // step, else in slot 1 (its last tile); every later one began inside it
    const int slot0 = (static_cast<int64_t>(b0) * work / G == g0) ? 0 : 1;
    const int q = blockIdx.y * kFixThreads + threadIdx.x;   // float4 index within the tile
    const int nl = q / (BM / 4), ml = (q % (BM / 4)) * 4;
    const int m0 = (t % tiles_m) * BM + ml, n = (t / tiles_m) * BN + nl;
    if (n >= N || m0 >= M) return;
    const float4* p4 = reinterpret_cast<const float4*>(part) + q;
    float4 v = p4[(static_cast<int64_t>(b0) * 2 + slot0) * (BM * BN / 4)];
    for (int b = b0 + 1; b <= b1; ++b) {
        const float4 u = p4[static_cast<int64_t>(b) * 2 * (BM * BN / 4)];
        v.x += u.x;
        v.y += u.y;
        v.z += u.z;
        v.w += u.w;
    }
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (m0 + i < M) store_y(Y, y_dtype, static_cast<int64_t>(n) * M + m0 + i, vv[i]);
}

// fp32 activations for the tensor cores: token row n, scaled by the power of
// two 2^s_n that puts its largest magnitude in [2^9, 2^10), is split into
// f16 parts hi = f16(x 2^s_n) and lo = f16(x 2^s_n - hi), written as rows
// 2n and 2n + 1 of X2; inv_scale[n] = 2^-s_n. hi + lo equals x 2^s_n to about
// 2^-22 relative, far inside the 1e-3 bar. The scale keeps every finite fp32
// row inside f16's range, with room for the 32-element activation sums of
// the min term (< 2^15), which are carried in f16 too. One CTA per token row.
constexpr int kSplitThreads = 256;
__global__ void __launch_bounds__(kSplitThreads) k_xsplit(const float* __restrict__ X, int K,
                                                          __half* __restrict__ X2, float* __restrict__ inv_scale) {
    __shared__ float red[kSplitThreads / 32];
    const int64_t n = blockIdx.x;
    const float* x = X + n * K;
    float mx = 0.f;
    for (int k = threadIdx.x; k < K; k += kSplitThreads) mx = fmaxf(mx, fabsf(x[k]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int i = 1; i < kSplitThreads / 32; ++i) mx = fmaxf(mx, red[i]);
    // exponent of the largest magnitude (subnormal or zero rows count as 2^-127;
    // a non-finite row keeps scale 1 and stays non-finite)
    int se = 0;
    if (mx < INFINITY) {
        const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127;
        se = min(126, max(-126, 9 - e));
    }
    const float sc = __uint_as_float(static_cast<uint32_t>(se + 127) << 23);
    if (threadIdx.x == 0) inv_scale[n] = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);
    __half* hi = X2 + (2 * n) * K;
    __half* lo = hi + K;
    for (int k = threadIdx.x; k < K; k += kSplitThreads) {
        const float v = x[k] * sc;
        const __half h = __float2half_rn(v);
        hi[k] = h;
        lo[k] = __float2half_rn(v - __half2float(h));
    }
}

// ------------------------------------------------------------ host side
bool make_map(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
              uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
    const uint64_t dims[2] = {dim0, dim1};
    const uint64_t strides[1] = {stride1_bytes};
    const uint32_t box[2] = {box0, box1};
    return encode_tiled_map(tm, dt, 2, base, dims, strides, box, sw);
}

// Library-owned per-device workspace for the activation sums (grown on demand;
// the first call at a given size must not be inside stream capture).
struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
Workspace g_ws[64];
std::mutex g_ws_mu;

void* workspace(size_t bytes, cudaStream_t s, bool* capturing) {
    int dev = 0;
    *capturing = false;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& w = g_ws[dev];
    if (w.bytes < bytes) {
        // growing would allocate: not allowed while the stream is being captured
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
            *capturing = true;
            return nullptr;
        }
        if (w.ptr) cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
        if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) return nullptr;
        w.bytes = bytes;
    }
    return w.ptr;
}

bool release_workspaces() {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return false;
    bool ok = true;
    for (int dev = 0; dev < 64; ++dev) {
        Workspace& w = g_ws[dev];
        if (!w.ptr) continue;
        if (cudaSetDevice(dev) != cudaSuccess || cudaFree(w.ptr) != cudaSuccess) ok = false;
        w.ptr = nullptr;
        w.bytes = 0;
    }
    if (cudaSetDevice(cur) != cudaSuccess) ok = false;
    return ok;
}

template <int KIND>
void ok_kind(const Problem& p, bool* out) {
    // one CTA per tile puts the token tiles on grid.y (at most 65535 of them)
    // fp32 activations run as two f16 rows per token (pair mode)
    const int64_t rows = p.x_dtype == 1 ? p.N : 2 * p.N;
    const bool x_ok = p.x_dtype == 1 ? reinterpret_cast<uintptr_t>(p.X) % 16 == 0 : p.x_dtype == 0;
    *out = !p.x_row && x_ok && p.K % KSUP == 0 && p.row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(p.W) % 16 == 0 &&
           p.M <= (int64_t(1) << 30) && (rows + BN - 1) / BN <= 65535 && p.K <= (int64_t(1) << 30);
}

// QMM_TC_SPLIT: 0 = automatic, 1 = one tile per CTA always, 2 = shared
// super-steps whenever possible (for measurements).
const int kEnvSplit = [] {
    const char* v = getenv("QMM_TC_SPLIT");
    return v ? atoi(v) : 0;
}();
// Estimated cost, in super-steps, of sharing tiles: the partial-tile stores
// and the fix-up kernel. Measured on 4096 x 4096 x 512 (128 tiles, 16 steps
// each): sharing (14 steps per CTA) ran 8 % slower than one tile per CTA, so
// the fix-up costs about 3 of that workload's super-steps; 11008 x 4096 x 128
// (86 tiles) ran 22 - 28 % faster shared (10 steps per CTA instead of 16).
constexpr int kSplitCost = 3;

// Grid size when the CTAs share the tiles' super-steps, or 0 for one CTA per
// tile. One tile per CTA takes ceil(tiles / SMs) waves of nsup super-steps;
// sharing takes ceil(tiles * nsup / SMs) super-steps per CTA plus the fix-up.
int split_grid(int64_t tiles, int nsup, int sms) {
    const int64_t work = tiles * nsup;
    if (kEnvSplit == 1 || sms <= 0 || work >= (int64_t(1) << 31)) return 0;
    const int G = static_cast<int>(imin64(sms, work));
    if (kEnvSplit == 2) return G;
    const int64_t waves = (tiles + sms - 1) / sms;
    const int64_t per = (work + G - 1) / G;
    return (per + kSplitCost < waves * nsup) ? G : 0;
}

template <int KIND>
void run(const Problem& p, cudaStream_t s, cudaError_t* e) {
    using R = Raw<KIND>;
    using MN = Mins<KIND>;
    const int M = static_cast<int>(p.M), K = static_cast<int>(p.K);
    const int ntok = static_cast<int>(p.N);
    // fp32 activations run as f16 (hi, lo) pairs: two MMA rows per token
    const bool pair = p.x_dtype == 0;
    const int N = pair ? 2 * ntok : ntok;
    const int nsup = K / KSUP;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int64_t tiles = static_cast<int64_t>(tiles_m) * tiles_n;
    int dev = 0;
    if ((*e = cudaGetDevice(&dev)) != cudaSuccess) return;
    const int G = pair ? 0 : split_grid(tiles, nsup, sm_count(dev));
    // one workspace: the (hi, lo) activations and their scales (fp32 input),
    // the activation sums (formats with mins), then the partial tiles
    const size_t x2_bytes = pair ? ((static_cast<size_t>(N) * K * 2 + 255) & ~size_t(255)) : 0;
    const size_t inv_bytes = pair ? ((static_cast<size_t>(ntok) * 4 + 255) & ~size_t(255)) : 0;
    const size_t xs_bytes = MN::ON ? ((static_cast<size_t>(N) * nsup * MN::KMW * 2 + 255) & ~size_t(255)) : 0;
    const size_t part_bytes = static_cast<size_t>(G) * 2 * BM * BN * sizeof(float);
    uint8_t* ws = nullptr;
    if (x2_bytes + inv_bytes + xs_bytes + part_bytes) {
        bool capturing = false;
        ws = static_cast<uint8_t*>(workspace(x2_bytes + inv_bytes + xs_bytes + part_bytes, s, &capturing));
        if (!ws) {
            *e = capturing ? cudaErrorStreamCaptureUnsupported : cudaErrorMemoryAllocation;
            return;
        }
    }
    const __half* X = static_cast<const __half*>(p.X);
    float* inv_scale = nullptr;
    if (pair) {
        __half* X2 = reinterpret_cast<__half*>(ws);
        inv_scale = reinterpret_cast<float*>(ws + x2_bytes);
        k_xsplit<<<static_cast<unsigned>(ntok), kSplitThreads, 0, s>>>(static_cast<const float*>(p.X), K, X2,
                                                                          inv_scale);
        count_launch(1);
        if ((*e = cudaGetLastError()) != cudaSuccess) return;
        X = X2;
    }
    uint8_t* xs_ws = ws ? ws + x2_bytes + inv_bytes : nullptr;
    CUtensorMap tmW, tmX, tmB;
    if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT16, p.W, p.row_bytes / 2, M, p.row_bytes, R::BOXB / 2, BM,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, K, N, static_cast<uint64_t>(K) * 2, KSUB, BN,
                  CU_TENSOR_MAP_SWIZZLE_128B)) {
        *e = cudaErrorInvalidValue;
        return;
    }
    tmB = tmX;
    if constexpr (MN::ON) {
        const int threads = 256;
        const int64_t total = static_cast<int64_t>(N) * (K / (KSUP / MN::G));
        const int blocks = static_cast<int>(imin64((total + threads - 1) / threads, 4096));
        k_xsums<<<blocks, threads, 0, s>>>(X, N, K, KSUP / MN::G, MN::G, reinterpret_cast<__half*>(xs_ws));
        count_launch(1);
        if ((*e = cudaGetLastError()) != cudaSuccess) return;
        if (!make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xs_ws, static_cast<uint64_t>(nsup) * MN::KMW, N,
                      static_cast<uint64_t>(nsup) * MN::KMW * 2, 16, BN, CU_TENSOR_MAP_SWIZZLE_32B)) {
            *e = cudaErrorInvalidValue;
            return;
        }
    }
    int smem_bytes = 0;
    const TcKernel kern = tc_kernel<KIND>(&smem_bytes);
    if ((*e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes)) != cudaSuccess) return;
    TcArgs a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.nsup = nsup;
    a.tiles_m = tiles_m;
    a.wq = G ? static_cast<int>(tiles * nsup / G) : 0;
    a.wr = G ? static_cast<int>(tiles * nsup % G) : 0;
    a.Y = p.Y;
    a.y_dtype = p.y_dtype;
    a.pair = pair ? 1 : 0;
    a.ntok = ntok;
    a.inv_scale = inv_scale;
    a.part = G ? reinterpret_cast<float*>(xs_ws + xs_bytes) : nullptr;
    a.err = p.err;
    const dim3 grid = G ? dim3(G) : dim3(tiles_m, tiles_n);
    kern<<<grid, tc_threads<KIND>(), smem_bytes, s>>>(tmW, tmX, tmB, a);
    count_launch(1);
    if ((*e = cudaGetLastError()) != cudaSuccess || !G) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles), kFixSplit);
    cfg.blockDim = dim3(kFixThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *e = cudaLaunchKernelEx(&cfg, k_tile_fixup, static_cast<const float*>(a.part), a.Y, M, N, tiles_m, nsup,
                            tiles * nsup, G, p.y_dtype);
    count_launch(1);
    if (*e == cudaSuccess) *e = cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free variant (qgemm_noalloc). Its scratch -- the per-group
// activation sums of the formats with mins -- lives in this fixed device
// array instead of the library's cudaMalloc-grown workspace. The array is
// reserved on every GPU that loads the library until the process exits, and
// every call shares it, so calls that overlap on the GPU race on it.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code cannot use the array's name as a device address) and
// forgotten by qmm_shutdown.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

template <int KIND>
void run_noalloc(const Problem& p, cudaStream_t s, int* status) {
    using R = Raw<KIND>;
    using MN = Mins<KIND>;
    using L = Layout<KIND>;
    const int M = static_cast<int>(p.M), N = static_cast<int>(p.N), K = static_cast<int>(p.K);
    const int nsup = K / KSUP;
    *status = 0;
    CUtensorMap tmW, tmX, tmB;
    if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT16, p.W, p.row_bytes / 2, M, p.row_bytes, R::BOXB / 2, BM,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.X, K, N, static_cast<uint64_t>(K) * 2, KSUB, BN,
                  CU_TENSOR_MAP_SWIZZLE_128B)) {
        *status = QMM_ERR_CUDA;
        return;
    }
    tmB = tmX;
    if constexpr (MN::ON) {
        const size_t need = static_cast<size_t>(N) * nsup * MN::KMW * 2;
        if (need > kNoAllocScratchBytes) {
            *status = QMM_ERR_NOALLOC_LIMIT;
            return;
        }
        void* ws = nullptr;
        if (noalloc_scratch(&ws) != cudaSuccess) {
            *status = QMM_ERR_CUDA;
            return;
        }
        // k_xsums writes every entry of the region this call reads, so nothing
        // left by an earlier call is ever used.
        const int threads = 256;
        const int64_t total = static_cast<int64_t>(N) * (K / (KSUP / MN::G));
        const int blocks = static_cast<int>(imin64((total + threads - 1) / threads, 4096));
        k_xsums<<<blocks, threads, 0, s>>>(static_cast<const __half*>(p.X), N, K, KSUP / MN::G, MN::G,
                                           static_cast<__half*>(ws));
        count_launch(1);
        if (cudaGetLastError() != cudaSuccess ||
            !make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ws, static_cast<uint64_t>(nsup) * MN::KMW, N,
                      static_cast<uint64_t>(nsup) * MN::KMW * 2, 16, BN, CU_TENSOR_MAP_SWIZZLE_32B)) {
            *status = QMM_ERR_CUDA;
            return;
        }
    }
    int smem_bytes = 0;
    const TcKernel kern = tc_kernel<KIND>(&smem_bytes);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess) {
        *status = QMM_ERR_CUDA;
        return;
    }
    TcArgs a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.nsup = nsup;
    a.tiles_m = (M + BM - 1) / BM;
    a.wq = 0;
    a.wr = 0;
    a.Y = p.Y;
    a.y_dtype = p.y_dtype;
    a.pair = 0;
    a.ntok = N;
    a.inv_scale = nullptr;
    a.part = nullptr;   // one tile per CTA: no partial-tile scratch
    a.err = p.err;
    const dim3 grid((M + BM - 1) / BM, (N + BN - 1) / BN);
    kern<<<grid, tc_threads<KIND>(), smem_bytes, s>>>(tmW, tmX, tmB, a);
    count_launch(1);
    if (cudaGetLastError() != cudaSuccess) *status = QMM_ERR_CUDA;
}

}  // namespace

bool release_gemm_workspaces() { return release_workspaces(); }

void forget_symbol_addresses() {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    for (auto& p : g_noalloc_ptr) p = nullptr;
}

int launch_gemm_tc_noalloc(const Problem& p, cudaStream_t s) {
    int status = 0;
    QMM_DISPATCH_KIND(p.kind, run_noalloc, p, s, &status);
    return status;
}

bool gemm_tc_ok(const Problem& p) {
    bool ok = false;
    QMM_DISPATCH_KIND(p.kind, ok_kind, p, &ok);
    return ok;
}

cudaError_t launch_gemm_tc(const Problem& p, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    QMM_DISPATCH_KIND(p.kind, run, p, s, &e);
    return e;
}

}  // namespace qmm
