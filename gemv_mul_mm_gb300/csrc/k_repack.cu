// k_repack.cu -- load-time repack of Q8_0 / Q4_0 rows into a structure-of-
// arrays layout, and the split-K streaming GEMV with an ordered reduce.
//
// The Vulkore examples/llm/quant_test.cpp page validates a load-time repack
// ("the native-layout kernels are correct and slow") whose layout splits the
// scales from the codes, checks that the repacked tensor reconstructs every
// element bit-exactly, and times a matvec on it plain and split over K with a
// reduce pass. Here:
//
//   * Layout. Rows stay contiguous and keep their byte count (18 per 32
//     elements for Q4_0, 34 for Q8_0). A row is a run of units of eight
//     blocks (256 elements): the eight code fields back to back (16 / 32 bytes
//     each, element order within a block as in the block), then the eight f16
//     scales. Every code vector and the scale vector are 16-byte aligned, so
//     the streaming GEMV loads them without realigning blocks.
//   * Split-K. K-slice e of every row is treated as "expert" e of the expert-
//     grouped streaming kernel (expert stride = the slice's bytes, row stride
//     = the whole row): each (slice, row group) is an independent work item,
//     so a product with few rows still covers every SM. Slice e of activation
//     row n is row n * split + e of the activations seen as split * N rows of
//     K / split values. The partial products of the slices are added by a
//     reduce kernel in slice order (deterministic).
#include <mutex>

#include "decode.cuh"
#include "qmm.h"
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kUnitElems = 256;   // elements per unit of eight blocks
static_assert(Q8_0R == kRepackedQ8_0 && Q4_0R == kRepackedQ4_0, "repacked layout ids");

// One unit per thread: native blocks [8 x BB] -> codes [8 x (BB - 2)], scales [8 x 2].
template <int BB>
__global__ void k_repack(const uint8_t* __restrict__ w, int64_t units, uint8_t* __restrict__ out) {
    constexpr int CB = BB - 2;   // code bytes per block
    for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t* src = w + u * 8 * BB;
        uint8_t* dst = out + u * 8 * BB;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            dst[8 * CB + 2 * b] = src[b * BB];
            dst[8 * CB + 2 * b + 1] = src[b * BB + 1];
#pragma unroll
            for (int i = 0; i < CB; ++i) dst[b * CB + i] = src[b * BB + 2 + i];
        }
    }
}

__global__ void k_split_rows(int32_t* __restrict__ x_row, int32_t* __restrict__ slice, int64_t A, int split) {
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < A;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        x_row[r] = static_cast<int32_t>(r);
        slice[r] = static_cast<int32_t>(r % split);
    }
}

// Y[n * M + m] = sum_e part[(n * split + e) * M + m], in slice order.
// A programmatic dependent of the GEMV: reads the partials after the wait.
__global__ void k_split_reduce(const float* __restrict__ part, float* __restrict__ Y, int y_dtype, int64_t N,
                               int64_t M, int split) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t total = N * M;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / M, m = i - n * M;
        const float* p = part + n * split * M + m;
        float acc = p[0];
        for (int e = 1; e < split; ++e) acc += p[e * M];
        store_y(Y, y_dtype, i, acc);
    }
}

// Library-owned per-device scratch of the split-K path (grown on demand; the
// growth is refused during stream capture, like the GEMM's workspace).
struct SplitWs {
    void* ptr = nullptr;
    size_t bytes = 0;
};
SplitWs g_split_ws[64];
std::mutex g_split_mu;

void* split_workspace(size_t bytes, cudaStream_t s, bool* capturing) {
    int dev = 0;
    *capturing = false;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_split_mu);
    SplitWs& w = g_split_ws[dev];
    if (w.bytes < bytes) {
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

size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

int block_bytes_of(int kind) { return kind == Q8_0 || kind == Q8_0R ? 34 : 18; }

}  // namespace

bool release_split_workspaces() {
    std::lock_guard<std::mutex> lk(g_split_mu);
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return false;
    bool ok = true;
    for (int dev = 0; dev < 64; ++dev) {
        SplitWs& w = g_split_ws[dev];
        if (!w.ptr) continue;
        if (cudaSetDevice(dev) != cudaSuccess || cudaFree(w.ptr) != cudaSuccess) ok = false;
        w.ptr = nullptr;
        w.bytes = 0;
    }
    if (cudaSetDevice(cur) != cudaSuccess) ok = false;
    return ok;
}

size_t repack_bytes(int kind, int64_t rows, int64_t cols) {
    if ((kind != Q8_0 && kind != Q4_0) || rows <= 0 || cols <= 0 || cols % kUnitElems) return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(cols / 32) * block_bytes_of(kind);
}

cudaError_t launch_repack(int kind, const uint8_t* w, int64_t rows, int64_t cols, uint8_t* out, cudaStream_t s) {
    const int64_t units = rows * (cols / kUnitElems);
    const int threads = 256;
    const int blocks = static_cast<int>(imin64((units + threads - 1) / threads, 8192));
    if (kind == Q8_0) k_repack<34><<<blocks, threads, 0, s>>>(w, units, out);
    else k_repack<18><<<blocks, threads, 0, s>>>(w, units, out);
    count_launch(1);
    return cudaGetLastError();
}

int launch_gemv_split(const Problem& p, int split, cudaStream_t s) {
    const int64_t units = p.K / kUnitElems;
    if (p.K % kUnitElems || p.N > 8) return QMM_ERR_UNIMPLEMENTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ERR_CUDA;
    if (split == 0) {
        // the smallest split (a divisor of the unit count) that gives every SM
        // two row-group items, within 64 ways
        const int64_t rg = (p.M + 31) / 32, want = 2 * static_cast<int64_t>(sm_count(dev));
        split = 1;
        for (int64_t d = 1; d <= imin64(units, 64); ++d) {
            if (units % d) continue;
            split = static_cast<int>(d);
            if (rg * d >= want) break;
        }
    }
    if (split < 1 || units % split) return QMM_ERR_BAD_ARGUMENT;
    if (split == 1) {
        if (!gemv_stream_ok(p)) return QMM_ERR_UNIMPLEMENTED;
        return launch_gemv_stream(p, s) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
    }
    const int64_t A = static_cast<int64_t>(split) * p.N;
    const size_t slice_bytes = p.row_bytes / static_cast<size_t>(split);
    Problem q = p;
    q.row_bytes = slice_bytes;
    q.row_stride = p.row_bytes;
    q.K = p.K / split;
    q.N = A;
    q.expert_stride = slice_bytes;
    q.n_experts = split;
    q.n_x_rows = A;
    q.cols_per_expert = static_cast<int>(p.N);
    q.y_dtype = 0;
    const size_t part_bytes = up256(static_cast<size_t>(A) * p.M * 4);
    const size_t idx_bytes = up256(static_cast<size_t>(A) * 4);
    bool capturing = false;
    uint8_t* ws = static_cast<uint8_t*>(split_workspace(part_bytes + 2 * idx_bytes, s, &capturing));
    if (!ws) return capturing ? QMM_ERR_WORKSPACE_IN_CAPTURE : QMM_ERR_CUDA;
    float* part = reinterpret_cast<float*>(ws);
    int32_t* x_row = reinterpret_cast<int32_t*>(ws + part_bytes);
    int32_t* slice = reinterpret_cast<int32_t*>(ws + part_bytes + idx_bytes);
    q.Y = part;
    q.x_row = x_row;
    q.expert_id = slice;
    if (!gemv_stream_ok(q)) return QMM_ERR_UNIMPLEMENTED;
    const int threads = 256;
    k_split_rows<<<static_cast<int>(imin64((A + threads - 1) / threads, 64)), threads, 0, s>>>(x_row, slice, A,
                                                                                               split);
    count_launch(1);
    if (cudaGetLastError() != cudaSuccess) return QMM_ERR_CUDA;
    if (launch_gemv_stream(q, s) != cudaSuccess) return QMM_ERR_CUDA;
    const int64_t total = p.N * p.M;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(imin64((total + threads - 1) / threads, 4096)));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_split_reduce, static_cast<const float*>(part), p.Y, p.y_dtype,
                                             p.N, p.M, split);
    count_launch(1);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace qmm
