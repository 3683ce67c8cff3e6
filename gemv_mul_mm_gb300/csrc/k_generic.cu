// k_generic.cu -- CUDA-core quantized GEMM for any shape and alignment.
//
// Y[n * M + m] = sum_k W[m, k] * X[n * K + k]   (ferrox-cuda 0.21.0
// src/mul_mm.rs, `BODY_SRC`), and the expert-indexed variant where column r
// reads expert expert_id[r]'s weights and activation row x_row[r].
//
// This is the path for shapes the specialised kernels do not take (rows that
// are not 16-byte multiples, unaligned pointers, K not a whole number of
// streaming groups). One CTA = 32 weight rows x NT columns; warp w owns 4 rows;
// lane l walks the row's 32-element chunks l, l+32, ...; each chunk is decoded
// once and multiplied into all NT columns; warps finish with a shuffle
// reduction. Accumulation is fp32 with the scale applied per element.
#include <cuda_fp16.h>

#include "decode.cuh"
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 8;
constexpr int kRowsPerCta = kRowsPerWarp * kWarps;

__device__ __forceinline__ float ldx(const void* X, int xdt, int64_t i) {
    if (xdt == 1) return __half2float(reinterpret_cast<const __half*>(X)[i]);
    return reinterpret_cast<const float*>(X)[i];
}

template <int KIND, int NT>
__global__ void __launch_bounds__(kWarps * 32) k_generic(Problem p) {
    constexpr int BB = Geo<KIND>::BB, BE = Geo<KIND>::BE;
    constexpr int CPB = BE / 32;  // 32-element chunks per block
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + warp * kRowsPerWarp;
    const bool grouped = p.x_row != nullptr;

    // Columns handled by this CTA and where their activations / weights live.
    const uint8_t* Wb = p.W;
    int64_t xrow[NT];
    int ncols;
    bool bad = false;
    if (grouped) {
        const int64_t r = blockIdx.y;
        const int e = p.expert_id[r];
        const int xr = p.x_row[r];
        if (e < 0 || e >= p.n_experts || xr < 0 || xr >= p.n_x_rows) {
            bad = true;
        } else {
            Wb = p.W + static_cast<size_t>(e) * p.expert_stride;
        }
        xrow[0] = bad ? 0 : xr;
        ncols = 1;
    } else {
        const int64_t n0 = static_cast<int64_t>(blockIdx.y) * NT;
        ncols = static_cast<int>(imin64(NT, p.N - n0));
#pragma unroll
        for (int c = 0; c < NT; ++c) xrow[c] = n0 + (c < ncols ? c : 0);
    }

    float acc[kRowsPerWarp][NT];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int c = 0; c < NT; ++c) acc[r][c] = 0.f;

    const int64_t nchunks = p.K / 32;
    if (!bad) {
        for (int64_t ch = lane; ch < nchunks; ch += 32) {
            const int64_t blk = ch / CPB;
            const int j = static_cast<int>(ch % CPB);
            const int64_t k0 = ch * 32;
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int64_t m = m0 + r;
                if (m >= p.M) break;
                const uint8_t* b = Wb + static_cast<size_t>(m) * p.row_bytes + static_cast<size_t>(blk) * BB;
#pragma unroll 4
                for (int i = 0; i < 32; ++i) {
                    const float v = elem32<KIND>(b, j, i);
#pragma unroll
                    for (int c = 0; c < NT; ++c)
                        acc[r][c] = fmaf(v, ldx(p.X, p.x_dtype, xrow[c] * p.K + k0 + i), acc[r][c]);
                }
            }
        }
    }

#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
#pragma unroll
        for (int c = 0; c < NT; ++c) {
            float v = acc[r][c];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            acc[r][c] = v;
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int64_t m = m0 + r;
            if (m >= p.M) break;
            if (grouped) {
                store_y(p.Y, p.y_dtype, static_cast<int64_t>(blockIdx.y) * p.M + m,
                        bad ? __int_as_float(0x7fc00000) : acc[r][0]);
            } else {
#pragma unroll
                for (int c = 0; c < NT; ++c)
                    if (c < ncols) store_y(p.Y, p.y_dtype, xrow[c] * p.M + m, acc[r][c]);
            }
        }
        if (bad && warp == 0 && blockIdx.x == 0) atomicOr(p.err, DEV_ERR_BAD_INDEX);
    }
}

template <int KIND>
void run(const Problem& p, cudaStream_t s, cudaError_t* err) {
    const unsigned gx = static_cast<unsigned>((p.M + kRowsPerCta - 1) / kRowsPerCta);
    *err = cudaSuccess;
    if (p.x_row) {
        // one column (assignment) per CTA row of the grid; gridDim.y <= 65535
        for (int64_t r0 = 0; r0 < p.N; r0 += 65535) {
            Problem q = p;
            const int64_t nr = imin64(65535, p.N - r0);
            q.x_row = p.x_row + r0;
            q.expert_id = p.expert_id + r0;
            q.Y = y_at(p.Y, r0 * p.M, p.y_dtype);
            q.N = nr;
            k_generic<KIND, 1><<<dim3(gx, static_cast<unsigned>(nr)), kWarps * 32, 0, s>>>(q);
            count_launch(1);
            if ((*err = cudaGetLastError()) != cudaSuccess) return;
        }
        return;
    }
    constexpr int NT = 8;
    const int64_t ny = (p.N + NT - 1) / NT;
    for (int64_t y0 = 0; y0 < ny; y0 += 65535) {
        Problem q = p;
        const int64_t nyy = imin64(65535, ny - y0);
        q.X = static_cast<const uint8_t*>(p.X) + y0 * NT * p.K * (p.x_dtype == 1 ? 2 : 4);
        q.Y = y_at(p.Y, y0 * NT * p.M, p.y_dtype);
        q.N = imin64(p.N - y0 * NT, nyy * NT);
        k_generic<KIND, NT><<<dim3(gx, static_cast<unsigned>(nyy)), kWarps * 32, 0, s>>>(q);
        count_launch(1);
        if ((*err = cudaGetLastError()) != cudaSuccess) return;
    }
}

}  // namespace

cudaError_t launch_generic(const Problem& p, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    QMM_DISPATCH_KIND(p.kind, run, p, s, &e);
    return e;
}

}  // namespace qmm
