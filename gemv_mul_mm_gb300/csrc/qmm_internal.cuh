// qmm_internal.cuh -- launchers shared between the entry points (api.cu) and
// the kernel translation units. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qmm {

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// Device-side error latch bits (OR-ed by kernels, read by qmm_check_device_error).
enum : unsigned {
    DEV_ERR_TIMEOUT = 1u,      // a bounded mbarrier wait ran out
    DEV_ERR_BAD_INDEX = 2u,    // an expert id or activation row out of range
};

// Number of streaming multiprocessors of `device` (cached).
int sm_count(int device);

// Records `n` kernel launches in the process-wide counter.
void count_launch(int n);

// Encodes a tiled TMA tensor map of `rank` dimensions (dims / box innermost
// first; strides[i] is the byte stride of dimension i + 1). False when the
// driver entry point is missing or rejects the description.
bool encode_tiled_map(CUtensorMap* tm, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw,
                      CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

// Problem description shared by the product kernels.
struct Problem {
    int kind;
    const uint8_t* W;        // weights (expert 0 for grouped)
    size_t row_bytes;        // bytes of the K elements a row contributes
    size_t row_stride = 0;   // bytes between rows (0: row_bytes; a K-slice view is shorter)
    int64_t M, K, N;         // N = columns (plain) or assignments (grouped)
    const void* X;
    int x_dtype;             // 0 f32, 1 f16
    float* Y;
    // grouped only
    const int32_t* x_row = nullptr;
    const int32_t* expert_id = nullptr;
    size_t expert_stride = 0;
    int n_experts = 0;
    int64_t n_x_rows = 0;
    unsigned flags = 0;      // QMM_FLAG_* of the call
    int y_dtype = 0;         // output element: 0 fp32, 1 f16, 2 bf16
    // activation rows: x_mode 0 reads X[row * K + k]; 1 (SwiGLU, fp32 X with
    // rows of x_stride >= 2 K values) reads silu(X[row * x_stride + k]) *
    // X[row * x_stride + K + k]
    int x_mode = 0;
    int64_t x_stride = 0;
    // grouped: every expert has exactly this many assignments (a split-K view),
    // or 0 (unknown, routed tokens)
    int cols_per_expert = 0;
    unsigned* err = nullptr; // device latch
};

// Bytes of one output element.
__host__ __device__ __forceinline__ int y_size(int y_dtype) { return y_dtype == 0 ? 4 : 2; }

// Output element i (of the call's output type) = v, rounded to nearest even
// for the 16-bit types.
__device__ __forceinline__ void store_y(float* Y, int y_dtype, int64_t i, float v) {
    if (y_dtype == 0) Y[i] = v;
    else if (y_dtype == 1) reinterpret_cast<__half*>(Y)[i] = __float2half_rn(v);
    else reinterpret_cast<__nv_bfloat16*>(Y)[i] = __float2bfloat16_rn(v);
}

// Y advanced by `elems` output elements.
__host__ __device__ __forceinline__ float* y_at(float* Y, int64_t elems, int y_dtype) {
    return reinterpret_cast<float*>(reinterpret_cast<char*>(Y) + elems * y_size(y_dtype));
}

// k_selftest.cu : a kernel whose bounded wait runs out (failure-path test)
cudaError_t launch_wait_never(unsigned* err, long long cycles, cudaStream_t s);

// k_dequant.cu
cudaError_t launch_dequant(int kind, const uint8_t* w, int64_t nblocks, float* out, cudaStream_t s);

// k_generic.cu : CUDA-core kernels for any shape and alignment
cudaError_t launch_generic(const Problem& p, cudaStream_t s);

// k_gemv.cu : weight-streaming GEMV (bulk-copy staged rows): N <= 8 columns, or
// the expert-grouped product (p.x_row set). p.kind may be a repacked layout.
bool gemv_stream_ok(const Problem& p);
cudaError_t launch_gemv_stream(const Problem& p, cudaStream_t s);

// k_repack.cu : the repacked layouts (qrepack) and the split-K GEMV. Problem
// kind ids of the repacked layouts (decode.cuh Q8_0R / Q4_0R).
constexpr int kRepackedQ8_0 = 32, kRepackedQ4_0 = 33;
size_t repack_bytes(int kind, int64_t rows, int64_t cols);
cudaError_t launch_repack(int kind, const uint8_t* w, int64_t rows, int64_t cols, uint8_t* out, cudaStream_t s);
// qgemm_repacked: the streaming GEMV over K-slices of a (repacked or native)
// layout, split ways, with an ordered reduce; split 0 = automatic. Returns a
// qmm_status.
int launch_gemv_split(const Problem& p, int split, cudaStream_t s);
// Frees the split-K path's grown workspaces on every device.
bool release_split_workspaces();

// k_moe.cu : the mixture-of-experts layer (qmoe_ffn)
size_t moe_workspace_bytes(int64_t T, int top_k, int64_t d_model, int64_t d_ff);
int launch_moe_ffn(int kind, const uint8_t* W_gu, size_t gu_stride, size_t gu_row_bytes, const uint8_t* W_down,
                   size_t down_stride, size_t down_row_bytes, int n_experts, const float* X, int64_t T,
                   int64_t d_model, int64_t d_ff, const int32_t* ids, const float* w, int top_k, float* Y,
                   void* workspace, unsigned* err, cudaStream_t s);

// k_gemm_tc.cu : tcgen05 tensor-core GEMM
bool gemm_tc_ok(const Problem& p);
cudaError_t launch_gemm_tc(const Problem& p, cudaStream_t s);
// Same GEMM with its scratch in a fixed device array (no allocation);
// returns a qmm_status code.
int launch_gemm_tc_noalloc(const Problem& p, cudaStream_t s);
// Frees the GEMM's grown workspaces on every device; false if a free failed.
bool release_gemm_workspaces();
// Drops the cached device addresses of the library's __device__ arrays.
void forget_symbol_addresses();

}  // namespace qmm
