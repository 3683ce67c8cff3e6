// api.cu -- the C ABI of libqmm (include/qmm.h): argument validation, kind
// geometry, path dispatch and the device error latch.
//
// Validation follows ferrox-cuda 0.21.0 src/mul_mm.rs `validate_shape`: empty
// shapes, K not a whole number of blocks and too-small buffers are refused by
// name before anything is launched.
#include "qmm.h"
#include "qmm_internal.cuh"

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

namespace qmm {

namespace {

struct KindRow {
    const char* name;
    int block_bytes;
    int block_elems;
};

constexpr KindRow kKinds[QMM_NKINDS] = {
    {"Q8_0", 34, 32},   {"Q4_0", 18, 32},   {"Q5_0", 22, 32},    {"Q4_K", 144, 256},
    {"Q5_K", 176, 256}, {"Q6_K", 210, 256}, {"Q2_K", 84, 256},   {"Q3_K", 110, 256},
    {"IQ4_NL", 18, 32}, {"IQ4_XS", 136, 256}, {"MXFP4", 17, 32}, {"Q4_1", 20, 32},
    {"Q5_1", 24, 32},   {"Q8_1", 36, 32},
};

std::atomic<uint64_t> g_launches{0};
thread_local int t_path = 0;        // kernel-path override of the calling thread
thread_local int t_last_path = 0;

constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;

__device__ unsigned g_dev_err;  // one latch per device (module-scope __device__)

bool kind_ok(int kind) { return kind >= 0 && kind < QMM_NKINDS; }

// Device latch address of the current device, looked up once per device.
int err_ptr(unsigned** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dev_err) != cudaSuccess) return QMM_ERR_CUDA;
        g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    *out = g_err_ptr[dev];
    return QMM_OK;
}

int finish(cudaError_t e, int path) {
    if (e == cudaErrorStreamCaptureUnsupported) return QMM_ERR_WORKSPACE_IN_CAPTURE;
    if (e != cudaSuccess) return QMM_ERR_CUDA;
    t_last_path = path;
    return QMM_OK;
}

int check_x(const void* x, int x_dtype) {
    if (x_dtype != QMM_F32 && x_dtype != QMM_F16) return QMM_ERR_BAD_DTYPE;
    const uintptr_t a = reinterpret_cast<uintptr_t>(x);
    if (a % (x_dtype == QMM_F32 ? 4 : 2)) return QMM_ERR_MISALIGNED;
    return QMM_OK;
}

}  // namespace

int sm_count(int device) {
    if (device < 0 || device >= kMaxDevices) return 1;
    if (!g_sms[device]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) n = 1;
        g_sms[device] = n;
    }
    return g_sms[device];
}

bool encode_tiled_map(CUtensorMap* tm, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw,
                      CUtensorMapL2promotion promo) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return fn(tm, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, promo,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

}  // namespace qmm

using namespace qmm;

extern "C" {

int qmm_kind_info(int kind, size_t* block_bytes, size_t* block_elems) {
    if (!kind_ok(kind)) return QMM_ERR_BAD_KIND;
    if (!block_bytes || !block_elems) return QMM_ERR_NULL_POINTER;
    *block_bytes = static_cast<size_t>(kKinds[kind].block_bytes);
    *block_elems = static_cast<size_t>(kKinds[kind].block_elems);
    return QMM_OK;
}

size_t qmm_row_bytes(int kind, int64_t K) {
    if (!kind_ok(kind) || K <= 0 || K % kKinds[kind].block_elems) return 0;
    return static_cast<size_t>(K / kKinds[kind].block_elems) * static_cast<size_t>(kKinds[kind].block_bytes);
}

const char* qmm_kind_name(int kind) { return kind_ok(kind) ? kKinds[kind].name : nullptr; }

const char* qmm_status_str(int status) {
    switch (status) {
    case QMM_OK: return "ok";
    case QMM_ERR_EMPTY_SHAPE: return "empty shape";
    case QMM_ERR_BAD_KIND: return "unknown block format";
    case QMM_ERR_BAD_DTYPE: return "unknown activation dtype";
    case QMM_ERR_COLS_NOT_BLOCK_ALIGNED: return "K is not a whole number of blocks";
    case QMM_ERR_WEIGHTS_TOO_SMALL: return "weight buffer too small";
    case QMM_ERR_ACTIVATIONS_TOO_SMALL: return "activation buffer too small";
    case QMM_ERR_NULL_POINTER: return "null pointer";
    case QMM_ERR_MISALIGNED: return "misaligned pointer";
    case QMM_ERR_BAD_EXPERT_ID: return "bad expert id, expert stride or activation row";
    case QMM_ERR_CUDA: return "CUDA runtime error";
    case QMM_ERR_DEVICE_TIMEOUT: return "device-side bounded wait timed out";
    case QMM_ERR_UNIMPLEMENTED: return "unimplemented";
    case QMM_ERR_BAD_ARGUMENT: return "bad argument";
    case QMM_ERR_OUTPUT_TOO_SMALL: return "output buffer too small";
    case QMM_ERR_WORKSPACE_TOO_SMALL: return "workspace too small (see qmoe_ffn_workspace_bytes)";
    case QMM_ERR_NOALLOC_LIMIT:
        return "problem needs more scratch than qgemm_noalloc's fixed array holds";
    case QMM_ERR_WORKSPACE_IN_CAPTURE:
        return "the library's workspace must grow, which cannot happen during stream capture: "
               "make one call of this shape outside capture first";
    default: return "unknown status";
    }
}

int qmm_set_path(int path) {
    if (path < 0 || path > 3) return -1;
    const int prev = t_path;
    t_path = path;
    return prev;
}

int qmm_last_path(void) { return t_last_path; }

uint64_t qmm_launch_count(void) { return g_launches.load(); }

int qmm_shutdown(void) {
    const bool ok = qmm::release_gemm_workspaces() & qmm::release_split_workspaces();
    // device addresses of the library's __device__ arrays are looked up again
    // on the next call (a new context may place them elsewhere)
    qmm::forget_symbol_addresses();
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int d = 0; d < kMaxDevices; ++d) g_err_ptr[d] = nullptr;
    }
    return ok ? QMM_OK : QMM_ERR_CUDA;
}

int qdequant(int kind, const void* blocks, size_t blocks_bytes, int64_t rows, int64_t cols,
             float* out, size_t out_elems, void* stream) {
    if (!kind_ok(kind)) return QMM_ERR_BAD_KIND;
    if (rows < 0 || cols < 0) return QMM_ERR_BAD_ARGUMENT;
    if (rows == 0 || cols == 0) return QMM_ERR_EMPTY_SHAPE;
    if (!blocks || !out) return QMM_ERR_NULL_POINTER;
    if (cols % kKinds[kind].block_elems) return QMM_ERR_COLS_NOT_BLOCK_ALIGNED;
    if (reinterpret_cast<uintptr_t>(out) % 4) return QMM_ERR_MISALIGNED;
    const size_t rb = qmm_row_bytes(kind, cols);
    if (blocks_bytes / rb < static_cast<size_t>(rows)) return QMM_ERR_WEIGHTS_TOO_SMALL;
    if (out_elems / static_cast<size_t>(cols) < static_cast<size_t>(rows)) return QMM_ERR_OUTPUT_TOO_SMALL;
    const int64_t nblocks = rows * (cols / kKinds[kind].block_elems);
    return finish(launch_dequant(kind, static_cast<const uint8_t*>(blocks), nblocks, out,
                                 static_cast<cudaStream_t>(stream)), 4);
}

int qgemm_ex(int kind, const void* W, size_t w_bytes, const void* X, int x_dtype, size_t x_elems,
             float* Y, size_t y_elems, int64_t M, int64_t K, int64_t N, uint32_t flags, void* stream) {
    if (!kind_ok(kind)) return QMM_ERR_BAD_KIND;
    constexpr uint32_t kKnown = QMM_FLAG_WEIGHTS_CONST | QMM_FLAG_Y_F16 | QMM_FLAG_Y_BF16;
    if ((flags & ~kKnown) || ((flags & QMM_FLAG_Y_F16) && (flags & QMM_FLAG_Y_BF16))) return QMM_ERR_BAD_ARGUMENT;
    const int y_dtype = (flags & QMM_FLAG_Y_F16) ? 1 : (flags & QMM_FLAG_Y_BF16) ? 2 : 0;
    if (M < 0 || K < 0 || N < 0) return QMM_ERR_BAD_ARGUMENT;
    if (M == 0 || K == 0 || N == 0) return QMM_ERR_EMPTY_SHAPE;
    if (!W || !X || !Y) return QMM_ERR_NULL_POINTER;
    if (int r = check_x(X, x_dtype)) return r;
    if (reinterpret_cast<uintptr_t>(Y) % y_size(y_dtype)) return QMM_ERR_MISALIGNED;
    if (K % kKinds[kind].block_elems) return QMM_ERR_COLS_NOT_BLOCK_ALIGNED;
    const size_t rb = qmm_row_bytes(kind, K);
    if (w_bytes / rb < static_cast<size_t>(M)) return QMM_ERR_WEIGHTS_TOO_SMALL;
    if (x_elems / static_cast<size_t>(K) < static_cast<size_t>(N)) return QMM_ERR_ACTIVATIONS_TOO_SMALL;
    if (y_elems / static_cast<size_t>(M) < static_cast<size_t>(N)) return QMM_ERR_OUTPUT_TOO_SMALL;
    unsigned* err = nullptr;
    if (int r = err_ptr(&err)) return r;

    Problem p;
    p.y_dtype = y_dtype;
    p.kind = kind;
    p.W = static_cast<const uint8_t*>(W);
    p.row_bytes = rb;
    p.M = M;
    p.K = K;
    p.N = N;
    p.X = X;
    p.x_dtype = x_dtype;
    p.Y = Y;
    p.flags = flags;
    p.err = err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int forced = t_path;
    if (forced == 1) return finish(launch_generic(p, s), 1);
    if (forced == 2) {
        if (!gemv_stream_ok(p)) return QMM_ERR_UNIMPLEMENTED;
        return finish(launch_gemv_stream(p, s), 2);
    }
    if (forced == 3) {
        if (!gemm_tc_ok(p)) return QMM_ERR_UNIMPLEMENTED;
        return finish(launch_gemm_tc(p, s), 3);
    }
    if (N > 8 && gemm_tc_ok(p)) return finish(launch_gemm_tc(p, s), 3);
    if (gemv_stream_ok(p)) return finish(launch_gemv_stream(p, s), 2);
    return finish(launch_generic(p, s), 1);
}

int qgemm(int kind, const void* W, size_t w_bytes, const void* X, int x_dtype, size_t x_elems,
          float* Y, size_t y_elems, int64_t M, int64_t K, int64_t N, void* stream) {
    return qgemm_ex(kind, W, w_bytes, X, x_dtype, x_elems, Y, y_elems, M, K, N, 0u, stream);
}

int qgemv(int kind, const void* W, size_t w_bytes, const void* x, int x_dtype, size_t x_elems,
          float* y, size_t y_elems, int64_t M, int64_t K, void* stream) {
    return qgemm_ex(kind, W, w_bytes, x, x_dtype, x_elems, y, y_elems, M, K, 1, 0u, stream);
}

int qgemm_grouped(int kind, const void* W, size_t w_bytes, size_t expert_stride, int n_experts,
                  const void* X, int x_dtype, size_t x_elems, int64_t n_x_rows,
                  const int32_t* x_row, const int32_t* expert_id, int64_t n_assign,
                  float* Y, size_t y_elems, int64_t M, int64_t K, void* stream) {
    if (!kind_ok(kind)) return QMM_ERR_BAD_KIND;
    if (M < 0 || K < 0 || n_assign < 0 || n_x_rows < 0 || n_experts < 0) return QMM_ERR_BAD_ARGUMENT;
    if (M == 0 || K == 0 || n_assign == 0) return QMM_ERR_EMPTY_SHAPE;
    if (!W || !X || !Y || !x_row || !expert_id) return QMM_ERR_NULL_POINTER;
    if (int r = check_x(X, x_dtype)) return r;
    if (reinterpret_cast<uintptr_t>(Y) % 4 || reinterpret_cast<uintptr_t>(x_row) % 4 ||
        reinterpret_cast<uintptr_t>(expert_id) % 4)
        return QMM_ERR_MISALIGNED;
    if (K % kKinds[kind].block_elems) return QMM_ERR_COLS_NOT_BLOCK_ALIGNED;
    const size_t rb = qmm_row_bytes(kind, K);
    if (n_experts == 0 || expert_stride / rb < static_cast<size_t>(M)) return QMM_ERR_BAD_EXPERT_ID;
    // the last expert's rows must lie inside W
    const size_t need = static_cast<size_t>(n_experts - 1) * expert_stride + static_cast<size_t>(M) * rb;
    if (w_bytes < need) return QMM_ERR_WEIGHTS_TOO_SMALL;
    if (n_x_rows == 0 || x_elems / static_cast<size_t>(K) < static_cast<size_t>(n_x_rows))
        return QMM_ERR_ACTIVATIONS_TOO_SMALL;
    if (y_elems / static_cast<size_t>(M) < static_cast<size_t>(n_assign)) return QMM_ERR_OUTPUT_TOO_SMALL;
    unsigned* err = nullptr;
    if (int r = err_ptr(&err)) return r;

    Problem p;
    p.kind = kind;
    p.W = static_cast<const uint8_t*>(W);
    p.row_bytes = rb;
    p.M = M;
    p.K = K;
    p.N = n_assign;
    p.X = X;
    p.x_dtype = x_dtype;
    p.Y = Y;
    p.x_row = x_row;
    p.expert_id = expert_id;
    p.expert_stride = expert_stride;
    p.n_experts = n_experts;
    p.n_x_rows = n_x_rows;
    p.err = err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every touched expert's rows stream once on the GEMV kernel; shapes it
    // does not take (unaligned rows, too many experts) run on the generic one
    if (t_path != 1 && gemv_stream_ok(p)) return finish(launch_gemv_stream(p, s), 5);
    return finish(launch_generic(p, s), 1);
}

int qgemm_noalloc(int kind, const void* W, size_t w_bytes, const void* X, int x_dtype, size_t x_elems,
                  float* Y, size_t y_elems, int64_t M, int64_t K, int64_t N, void* stream) {
    if (!kind_ok(kind)) return QMM_ERR_BAD_KIND;
    if (M < 0 || K < 0 || N < 0) return QMM_ERR_BAD_ARGUMENT;
    if (M == 0 || K == 0 || N == 0) return QMM_ERR_EMPTY_SHAPE;
    if (!W || !X || !Y) return QMM_ERR_NULL_POINTER;
    if (int r = check_x(X, x_dtype)) return r;
    if (reinterpret_cast<uintptr_t>(Y) % 4) return QMM_ERR_MISALIGNED;
    if (K % kKinds[kind].block_elems) return QMM_ERR_COLS_NOT_BLOCK_ALIGNED;
    const size_t rb = qmm_row_bytes(kind, K);
    if (w_bytes / rb < static_cast<size_t>(M)) return QMM_ERR_WEIGHTS_TOO_SMALL;
    if (x_elems / static_cast<size_t>(K) < static_cast<size_t>(N)) return QMM_ERR_ACTIVATIONS_TOO_SMALL;
    if (y_elems / static_cast<size_t>(M) < static_cast<size_t>(N)) return QMM_ERR_OUTPUT_TOO_SMALL;
    unsigned* err = nullptr;
    if (int r = err_ptr(&err)) return r;
    Problem p;
    p.kind = kind;
    p.W = static_cast<const uint8_t*>(W);
    p.row_bytes = rb;
    p.M = M;
    p.K = K;
    p.N = N;
    p.X = X;
    p.x_dtype = x_dtype;
    p.Y = Y;
    p.err = err;
    if (x_dtype != QMM_F16 || !gemm_tc_ok(p)) return QMM_ERR_UNIMPLEMENTED;
    const int r = launch_gemm_tc_noalloc(p, static_cast<cudaStream_t>(stream));
    if (r == QMM_OK) t_last_path = 3;
    return r;
}

size_t qrepack_bytes(int kind, int64_t rows, int64_t cols) {
    if (!kind_ok(kind)) return 0;
    return repack_bytes(kind, rows, cols);
}

int qrepack(int kind, const void* W, size_t w_bytes, int64_t rows, int64_t cols, void* out, size_t out_bytes,
            void* stream) {
    if (!kind_ok(kind)) return QMM_ERR_BAD_KIND;
    if (kind != QMM_Q8_0 && kind != QMM_Q4_0) return QMM_ERR_UNIMPLEMENTED;
    if (rows < 0 || cols < 0) return QMM_ERR_BAD_ARGUMENT;
    if (rows == 0 || cols == 0) return QMM_ERR_EMPTY_SHAPE;
    if (!W || !out) return QMM_ERR_NULL_POINTER;
    if (cols % 256) return QMM_ERR_COLS_NOT_BLOCK_ALIGNED;
    const size_t need = repack_bytes(kind, rows, cols);
    if (w_bytes < need) return QMM_ERR_WEIGHTS_TOO_SMALL;
    if (out_bytes < need) return QMM_ERR_OUTPUT_TOO_SMALL;
    return finish(launch_repack(kind, static_cast<const uint8_t*>(W), rows, cols, static_cast<uint8_t*>(out),
                                static_cast<cudaStream_t>(stream)), 4);
}

int qgemm_repacked(int kind, const void* R, size_t r_bytes, const void* X, int x_dtype, size_t x_elems, float* Y,
                   size_t y_elems, int64_t M, int64_t K, int64_t N, int split, uint32_t flags, void* stream) {
    if (!kind_ok(kind)) return QMM_ERR_BAD_KIND;
    if (kind != QMM_Q8_0 && kind != QMM_Q4_0) return QMM_ERR_UNIMPLEMENTED;
    constexpr uint32_t kKnown = QMM_FLAG_WEIGHTS_CONST | QMM_FLAG_Y_F16 | QMM_FLAG_Y_BF16;
    if ((flags & ~kKnown) || ((flags & QMM_FLAG_Y_F16) && (flags & QMM_FLAG_Y_BF16))) return QMM_ERR_BAD_ARGUMENT;
    const int y_dtype = (flags & QMM_FLAG_Y_F16) ? 1 : (flags & QMM_FLAG_Y_BF16) ? 2 : 0;
    if (M < 0 || K < 0 || N < 0 || split < 0) return QMM_ERR_BAD_ARGUMENT;
    if (M == 0 || K == 0 || N == 0) return QMM_ERR_EMPTY_SHAPE;
    if (!R || !X || !Y) return QMM_ERR_NULL_POINTER;
    if (int r = check_x(X, x_dtype)) return r;
    if (reinterpret_cast<uintptr_t>(Y) % y_size(y_dtype) || reinterpret_cast<uintptr_t>(R) % 16)
        return QMM_ERR_MISALIGNED;
    if (K % 256) return QMM_ERR_COLS_NOT_BLOCK_ALIGNED;
    if (N > 8) return QMM_ERR_UNIMPLEMENTED;
    if (split > 0 && (K / 256) % split) return QMM_ERR_BAD_ARGUMENT;
    const size_t rb = qmm_row_bytes(kind, K);
    if (r_bytes / rb < static_cast<size_t>(M)) return QMM_ERR_WEIGHTS_TOO_SMALL;
    if (x_elems / static_cast<size_t>(K) < static_cast<size_t>(N)) return QMM_ERR_ACTIVATIONS_TOO_SMALL;
    if (y_elems / static_cast<size_t>(M) < static_cast<size_t>(N)) return QMM_ERR_OUTPUT_TOO_SMALL;
    unsigned* err = nullptr;
    if (int r = err_ptr(&err)) return r;
    Problem p;
    p.kind = kind == QMM_Q8_0 ? kRepackedQ8_0 : kRepackedQ4_0;
    p.W = static_cast<const uint8_t*>(R);
    p.row_bytes = rb;
    p.M = M;
    p.K = K;
    p.N = N;
    p.X = X;
    p.x_dtype = x_dtype;
    p.Y = Y;
    p.y_dtype = y_dtype;
    p.flags = flags;
    p.err = err;
    const int r = launch_gemv_split(p, split, static_cast<cudaStream_t>(stream));
    if (r == QMM_OK) t_last_path = 7;
    return r;
}

size_t qmoe_ffn_workspace_bytes(int64_t T, int top_k, int64_t d_model, int64_t d_ff) {
    if (T <= 0 || top_k <= 0 || d_model <= 0 || d_ff <= 0) return 0;
    return moe_workspace_bytes(T, top_k, d_model, d_ff);
}

int qmoe_ffn(int kind, const void* W_gu, size_t w_gu_bytes, size_t gu_stride, const void* W_down,
             size_t w_down_bytes, size_t down_stride, int n_experts, const float* X, size_t x_elems,
             int64_t T, int64_t d_model, int64_t d_ff, const int32_t* topk_ids, const float* topk_w,
             int top_k, float* Y, size_t y_elems, void* workspace, size_t workspace_bytes, void* stream) {
    if (!kind_ok(kind)) return QMM_ERR_BAD_KIND;
    if (T < 0 || d_model < 0 || d_ff < 0 || top_k < 0 || n_experts < 0) return QMM_ERR_BAD_ARGUMENT;
    if (T == 0 || d_model == 0 || d_ff == 0 || top_k == 0) return QMM_ERR_EMPTY_SHAPE;
    if (!W_gu || !W_down || !X || !topk_ids || !topk_w || !Y || !workspace) return QMM_ERR_NULL_POINTER;
    if (reinterpret_cast<uintptr_t>(X) % 16 || reinterpret_cast<uintptr_t>(Y) % 4 ||
        reinterpret_cast<uintptr_t>(topk_ids) % 4 || reinterpret_cast<uintptr_t>(topk_w) % 4 ||
        reinterpret_cast<uintptr_t>(workspace) % 256)
        return QMM_ERR_MISALIGNED;
    const int be = kKinds[kind].block_elems;
    if (d_model % be || d_ff % be) return QMM_ERR_COLS_NOT_BLOCK_ALIGNED;
    const size_t rb_gu = qmm_row_bytes(kind, d_model), rb_dn = qmm_row_bytes(kind, d_ff);
    if (n_experts == 0 || gu_stride / rb_gu < static_cast<size_t>(2 * d_ff) ||
        down_stride / rb_dn < static_cast<size_t>(d_model))
        return QMM_ERR_BAD_EXPERT_ID;
    if (w_gu_bytes < static_cast<size_t>(n_experts - 1) * gu_stride + static_cast<size_t>(2 * d_ff) * rb_gu ||
        w_down_bytes < static_cast<size_t>(n_experts - 1) * down_stride + static_cast<size_t>(d_model) * rb_dn)
        return QMM_ERR_WEIGHTS_TOO_SMALL;
    if (x_elems / static_cast<size_t>(d_model) < static_cast<size_t>(T)) return QMM_ERR_ACTIVATIONS_TOO_SMALL;
    if (y_elems / static_cast<size_t>(d_model) < static_cast<size_t>(T)) return QMM_ERR_OUTPUT_TOO_SMALL;
    if (workspace_bytes < moe_workspace_bytes(T, top_k, d_model, d_ff)) return QMM_ERR_WORKSPACE_TOO_SMALL;
    unsigned* err = nullptr;
    if (int r = err_ptr(&err)) return r;
    const int r = launch_moe_ffn(kind, static_cast<const uint8_t*>(W_gu), gu_stride, rb_gu,
                                 static_cast<const uint8_t*>(W_down), down_stride, rb_dn, n_experts, X, T, d_model,
                                 d_ff, topk_ids, topk_w, top_k, Y, workspace, err, static_cast<cudaStream_t>(stream));
    if (r == QMM_OK) t_last_path = 6;
    return r;
}

int qmm_selftest_wait_timeout(int64_t cycles, void* stream) {
    if (cycles < 1 || cycles > (int64_t(1) << 32)) return QMM_ERR_BAD_ARGUMENT;
    unsigned* err = nullptr;
    if (int r = err_ptr(&err)) return r;
    return launch_wait_never(err, cycles, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

int qmm_check_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QMM_ERR_CUDA;
    unsigned* err = nullptr;
    if (int r = err_ptr(&err)) return r;
    unsigned v = 0;
    if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QMM_ERR_CUDA;
    if (v) {
        const unsigned zero = 0;
        if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return QMM_ERR_CUDA;
    }
    if (v & DEV_ERR_TIMEOUT) return QMM_ERR_DEVICE_TIMEOUT;
    if (v & DEV_ERR_BAD_INDEX) return QMM_ERR_BAD_EXPERT_ID;
    return QMM_OK;
}

}  // extern "C"
