// k_dequant.cu -- qdequant: expand quantized blocks to fp32, bit-exactly.
//
// The weight matrix is a flat run of blocks (rows are contiguous runs of whole
// blocks), so the kernel works on 2048-element tiles of that run: the tile's
// bytes (a multiple of 16 for every format) are staged into shared memory with
// coalesced 16-byte loads, then each thread decodes two float4 of output and
// writes them with coalesced 16-byte stores (256 threads x 16 B = 4 KB per
// store wave). Each float4 is one call of elem4, which derives the group's
// scale factors once for its four elements; codebooks are read from a copy in
// shared memory. The write of 4 bytes per element dominates the traffic, so
// the roofline is HBM: bytes = blocks + 4 * elements.
//
// Element values: Vulkore examples/llm/quant_test.cpp (the `ref::` CPU
// references, element-indexed) and ferrox-cuda 0.20.0 codebook.rs.
#include "decode.cuh"
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kTileElems = 2048;
constexpr int kThreads = 256;

template <int KIND>
__global__ void __launch_bounds__(kThreads) k_dequant(const uint8_t* __restrict__ w, int64_t nblocks,
                                                       float* __restrict__ out, int vec_in, int vec_out) {
    constexpr int BB = Geo<KIND>::BB, BE = Geo<KIND>::BE;
    constexpr int TB = kTileElems / BE;        // blocks per tile
    constexpr int TBYTES = TB * BB;            // multiple of 16 for every format
    static_assert(TBYTES % 16 == 0, "tile bytes must be whole 16-byte vectors");
    __shared__ __align__(16) uint8_t sbuf[TBYTES];
    __shared__ float tbl[16];   // codebook (IQ4_NL / IQ4_XS / MXFP4), one entry per bank
    if (threadIdx.x < 16) tbl[threadIdx.x] = codebook_entry<KIND>(threadIdx.x);

    const int64_t ntiles = (nblocks + TB - 1) / TB;
    const int64_t total_elems = nblocks * BE;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t b0 = t * TB;
        const int nb = static_cast<int>(imin64(TB, nblocks - b0));
        const uint8_t* src = w + b0 * BB;
        if (vec_in && nb == TB) {
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
            for (int i = threadIdx.x; i < TBYTES / 16; i += kThreads)
                reinterpret_cast<uint4*>(sbuf)[i] = __ldcs(s4 + i);
        } else {
            for (int i = threadIdx.x; i < nb * BB; i += kThreads) sbuf[i] = src[i];
        }
        __syncthreads();
        const int64_t e_base = t * kTileElems;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int e = 4 * threadIdx.x + half * (kTileElems / 2);
            const int blk = e / BE, eb = e % BE;
            if (blk < nb) {
                const float4 v = elem4<KIND>(sbuf + blk * BB, eb, tbl);
                float* dst = out + e_base + e;
                if (vec_out) {
                    __stcs(reinterpret_cast<float4*>(dst), v);
                } else if (e_base + e + 3 < total_elems) {
                    dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
                }
            }
        }
        __syncthreads();
    }
}

template <int KIND>
void run(const uint8_t* w, int64_t nblocks, float* out, cudaStream_t s, cudaError_t* err) {
    constexpr int TB = kTileElems / Geo<KIND>::BE;
    const int64_t ntiles = (nblocks + TB - 1) / TB;
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t grid = imin64(ntiles, static_cast<int64_t>(sm_count(dev)) * 8);
    const int vec_in = (reinterpret_cast<uintptr_t>(w) % 16) == 0;
    const int vec_out = (reinterpret_cast<uintptr_t>(out) % 16) == 0;
    k_dequant<KIND><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(w, nblocks, out, vec_in, vec_out);
    *err = cudaGetLastError();
    count_launch(1);
}

}  // namespace

cudaError_t launch_dequant(int kind, const uint8_t* w, int64_t nblocks, float* out, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    QMM_DISPATCH_KIND(kind, run, w, nblocks, out, s, &e);
    return e;
}

}  // namespace qmm
