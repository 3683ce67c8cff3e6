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
//   * Activations are staged once per CTA in a per-format layout: for Q4_0 the
//     pairs (2 x[e], x[e+16] / 8) of every block, plus one offset per block, so
//     that a nibble OR-ed into the mantissa of 128.0f (no int->float convert)
//     feeds a packed fp32x2 FMA (sm_100 FFMA2), and the scale d multiplies the
//     block's partial sum in fp32.
//   * Persistent grid (one CTA per SM) over the row groups.
//
// The P4 page's v3 lesson (stage x in shared, keep lanes on distinct banks,
// keep loads in flight) is kept; its f16x2 accumulation is not (too lossy for
// the 1e-3 relative bar over K = 4096), nor its structure-of-arrays layout.
#include <cuda_fp16.h>

#include "decode.cuh"
#include "qmm_internal.cuh"
#include "sm100_async.cuh"

namespace qmm {
namespace {

constexpr int kRows = 32;
constexpr int kMaxStages = 4;
constexpr int kSmemBudget = 220 * 1024;

// Per format: blocks per warp unit (UB) and consumer warps (NW). A unit's bytes
// times NW (one chunk row) is a multiple of 16 for every format.
template <int KIND> struct SG;
template <> struct SG<Q8_0>   { static constexpr int UB = 8,  NW = 4; };
template <> struct SG<Q4_0>   { static constexpr int UB = 8,  NW = 8; };
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
    int ncols;      // valid columns in this pass (<= NCOL)
    float* Y;       // already offset to the pass's first column
    int stages;
    unsigned* err;
};

__device__ __forceinline__ float load_x(const void* X, int xdt, int64_t i) {
    if (xdt == 1) return __half2float(reinterpret_cast<const __half*>(X)[i]);
    return reinterpret_cast<const float*>(X)[i];
}

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

// Q4_0: 8 blocks of 18 bytes (144 B, 16-byte aligned in shared memory).
// Code byte e is shifted to bits 15..22 (the top of the fp32 mantissa), so
// OR-ing 0x43000000 (128.0f) onto its low nibble gives 128 + q/2 and onto its
// high nibble 128 + 8 q, exactly (bit 23 is the exponent's LSB and must stay
// clear). Against the staged pairs (2 x[e], x[e+16] / 8) the block sum is
// S = sum q x + 256 X_lo + 16 X_hi, so sum (q - 8) x = S - (264 X_lo + 24 X_hi)
// = S - cb[block].
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
#pragma unroll
    for (int blk = 0; blk < 8; ++blk) {
        const int o = 18 * blk;
        const uint32_t dw = w[o >> 2];
        const float d = h2f((o & 3) ? (dw >> 16) : dw);
        const int kb = k0 + 32 * blk;
        float2 S[NCOL];
#pragma unroll
        for (int n = 0; n < NCOL; ++n) S[n] = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            float4 xv[NCOL];
#pragma unroll
            for (int n = 0; n < NCOL; ++n) xv[n] = *reinterpret_cast<const float4*>(xs + n * K + kb + 2 * e);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int bp = o + 2 + e + h;
                const uint32_t word = w[bp >> 2];
                const int pos = bp & 3;
                const uint32_t t = pos == 0 ? (word << 15) : pos == 1 ? (word << 7) : pos == 2 ? (word >> 1) : (word >> 9);
                const float2 f = make_float2(__int_as_float(0x43000000 | (t & 0x00078000u)),
                                             __int_as_float(0x43000000 | (t & 0x00780000u)));
#pragma unroll
                for (int n = 0; n < NCOL; ++n) {
                    const float2 xp = h ? make_float2(xv[n].z, xv[n].w) : make_float2(xv[n].x, xv[n].y);
                    S[n] = __ffma2_rn(f, xp, S[n]);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < NCOL; ++n) acc[n] = fmaf(d, (S[n].x + S[n].y) - cb[n * nb32 + (kb >> 5)], acc[n]);
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
        float2 S[NCOL];
#pragma unroll
        for (int n = 0; n < NCOL; ++n) S[n] = make_float2(0.f, 0.f);
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
                    S[n] = __ffma2_rn(q, xp, S[n]);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < NCOL; ++n) acc[n] = fmaf(d, S[n].x + S[n].y, acc[n]);
    }
}

template <int KIND, int NCOL>
__device__ __forceinline__ void unit(const uint8_t* u, const float* xs, const float* cb, int K, int k0,
                                     float (&acc)[NCOL]) {
    if constexpr (KIND == Q4_0) unit_q4_0<NCOL>(u, xs, cb, K, k0, acc);
    else if constexpr (KIND == Q8_0) unit_q8_0<NCOL>(u, xs, cb, K, k0, acc);
    else unit_generic<KIND, NCOL>(u, xs, cb, K, k0, acc);
}

// Activation staging (consumer threads): plain fp32, or the Q4_0 pair layout.
template <int KIND, int NCOL>
__device__ void stage_x(const GemvArgs& a, float* xs, float* cb, int tid, int nthr) {
    const int K = a.K;
    if constexpr (KIND == Q4_0) {
        const int nb = K / 32;
        for (int i = tid; i < NCOL * nb; i += nthr) {
            const int n = i / nb, b = i % nb;
            float lo = 0.f, hi = 0.f;
            float* dst = xs + n * K + 32 * b;
            for (int e = 0; e < 16; ++e) {
                const float xl = n < a.ncols ? load_x(a.X, a.x_dtype, static_cast<int64_t>(n) * K + 32 * b + e) : 0.f;
                const float xh =
                    n < a.ncols ? load_x(a.X, a.x_dtype, static_cast<int64_t>(n) * K + 32 * b + 16 + e) : 0.f;
                dst[2 * e] = 2.f * xl;
                dst[2 * e + 1] = xh * 0.125f;
                lo += xl;
                hi += xh;
            }
            cb[n * nb + b] = 264.f * lo + 24.f * hi;
        }
    } else {
        for (int i = tid; i < NCOL * K; i += nthr) {
            const int n = i / K;
            xs[i] = n < a.ncols ? load_x(a.X, a.x_dtype, i) : 0.f;
        }
    }
}

template <int KIND> __host__ __device__ constexpr int cb_floats(int K, int ncol) { return KIND == Q4_0 ? ncol * (K / 32) : 0; }

template <int KIND, int NCOL>
__global__ void __launch_bounds__((SG<KIND>::NW + 1) * 32, 1) k_gemv(GemvArgs a) {
    using G = SGeo<KIND>;
    constexpr int NW = G::NW;
    extern __shared__ __align__(128) uint8_t smem[];
    const int K = a.K;
    uint8_t* stage0 = smem;
    float* xs = reinterpret_cast<float*>(smem + a.stages * G::STAGE_B);
    float* cb = xs + NCOL * K;
    float* red = cb + cb_floats<KIND>(K, NCOL);
    uint64_t* full = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(red + 2 * NCOL * NW * 32) + 7) & ~static_cast<uintptr_t>(7));
    uint64_t* empty = full + kMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kMaxStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int64_t ngroups = (a.M + kRows - 1) / kRows;
    const int nchunks = (K + G::CHUNK_E - 1) / G::CHUNK_E;
    const int ST = a.stages;

    if (warp == NW) {
        // ---------------- producer warp ----------------
        const uint64_t pol = l2_evict_first_policy();
        int it = 0;
        for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
            const int rows = static_cast<int>(imin64(kRows, a.M - g * kRows));
            const uint8_t* wg = a.W + static_cast<size_t>(g * kRows) * a.row_bytes;
            for (int kc = 0; kc < nchunks; ++kc, ++it) {
                const int s = it % ST, use = it / ST;
                if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, abort_flag, a.err)) goto drain;
                const int units = min(NW, (K - kc * G::CHUNK_E) / G::UNIT_E);
                const uint32_t bytes = static_cast<uint32_t>(units * G::UNIT_B);
                if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(rows) * bytes);
                __syncwarp();
                if (lane < rows)
                    bulk_g2s_hint(stage0 + s * G::STAGE_B + lane * G::STRIDE,
                                  wg + static_cast<size_t>(lane) * a.row_bytes + static_cast<size_t>(kc) * G::CHUNK_B,
                                  bytes, &full[s], pol);
            }
        }
    drain:
        // Before the CTA can retire, every issued copy must have landed: wait
        // (bounded, ignoring the abort flag) for the last phase of each stage.
        {
            const int issued = it;
            for (int s = 0; s < ST && s < issued; ++s) {
                const int last_use = (issued - 1 - s) / ST;  // uses of slot s: it = s + ST*use
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
    stage_x<KIND, NCOL>(a, xs, cb, threadIdx.x, NW * 32);
    named_bar_sync(1, NW * 32);

    int it = 0, gi = 0;
    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x, ++gi) {
        float acc[NCOL];
#pragma unroll
        for (int n = 0; n < NCOL; ++n) acc[n] = 0.f;
        for (int kc = 0; kc < nchunks; ++kc, ++it) {
            const int s = it % ST, use = it / ST;
            const bool ok = !*abort_flag && mbar_wait(&full[s], use & 1, abort_flag, a.err);
            const int units = min(NW, (K - kc * G::CHUNK_E) / G::UNIT_E);
            if (ok && warp < units)
                unit<KIND, NCOL>(stage0 + s * G::STAGE_B + lane * G::STRIDE + warp * G::UNIT_B, xs, cb, K,
                                 kc * G::CHUNK_E + warp * G::UNIT_E, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        float* rb = red + (gi & 1) * NCOL * NW * 32;
#pragma unroll
        for (int n = 0; n < NCOL; ++n) rb[(n * NW + warp) * 32 + lane] = acc[n];
        named_bar_sync(1, NW * 32);
        if (warp == 0) {
            const int64_t row = g * kRows + lane;
            if (row < a.M) {
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
        }
    }
}

template <int KIND>
size_t smem_bytes(int K, int ncol, int stages) {
    using G = SGeo<KIND>;
    size_t b = static_cast<size_t>(stages) * G::STAGE_B;
    b += sizeof(float) * (static_cast<size_t>(ncol) * K + cb_floats<KIND>(K, ncol) + 2 * ncol * G::NW * 32);
    b = (b + 7) & ~size_t(7);
    b += 2 * kMaxStages * sizeof(uint64_t) + 16;
    return b;
}

template <int KIND>
bool ok_kind(const Problem& p) {
    using G = SGeo<KIND>;
    if (p.x_row) return false;
    if (p.N > 8 || p.K > (1 << 24)) return false;
    if (p.row_bytes % 16 || reinterpret_cast<uintptr_t>(p.W) % 16) return false;
    if (p.K % G::UNIT_E) return false;
    if (!G::PARTIAL_OK && p.K % G::CHUNK_E) return false;
    const int ncol = p.N <= 1 ? 1 : p.N <= 2 ? 2 : p.N <= 4 ? 4 : 8;
    return smem_bytes<KIND>(static_cast<int>(p.K), ncol, 2) <= kSmemBudget;
}

template <int KIND, int NCOL>
cudaError_t launch_ncol(const Problem& p, cudaStream_t s) {
    using G = SGeo<KIND>;
    const int K = static_cast<int>(p.K);
    int stages = kMaxStages;
    while (stages > 2 && smem_bytes<KIND>(K, NCOL, stages) > kSmemBudget) --stages;
    const size_t smem = smem_bytes<KIND>(K, NCOL, stages);
    auto kern = k_gemv<KIND, NCOL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t ngroups = (p.M + kRows - 1) / kRows;
    const int grid = static_cast<int>(imin64(ngroups, sm_count(dev)));
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
    kern<<<grid, (G::NW + 1) * 32, smem, s>>>(a);
    count_launch(1);
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
