// k_moe.cu -- qmoe_ffn: one mixture-of-experts feed-forward layer over
// block-quantized experts.
//
// For token t and routing slot j (expert e = ids[t, j], weight w[t, j]):
//   g, u = gate and up rows of W_gu_e times x_t   (gate rows first, then up)
//   h    = silu(g) * u                            (SwiGLU)
//   o    = W_down_e h
//   y_t  = sum_j w[t, j] o                        (top-k weighted combine)
// The decoder layer whose per-token weight traffic the inferencelayer 0.2.8
// src/cublas_prefill.rs page quotes for Qwen3-30B-A3B (about 2.1 GB per token
// in q4_0).
//
// Launches, all on the caller's stream:
//   1. k_moe_rows: the activation row of every assignment r = t * top_k + j
//      (t for the gate_up projection, r for the down projection);
//   2. the expert-grouped streaming GEMV over gate_up: every touched expert's
//      rows stream from HBM once per block of up to four of its assignments;
//   3. the same kernel over down, staging silu(g) * u from the gate_up output
//      rows as its activations (no separate SwiGLU pass or buffer);
//   4. k_moe_combine: the weighted sum over each token's slots, in slot
//      order (deterministic).
// The caller provides the scratch (qmoe_ffn_workspace_bytes); nothing is
// allocated here.
#include "qmm.h"
#include "qmm_internal.cuh"

namespace qmm {
namespace {

__global__ void k_moe_rows(int32_t* __restrict__ row_gu, int32_t* __restrict__ row_dn, int64_t A, int top_k) {
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < A;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        row_gu[r] = static_cast<int32_t>(r / top_k);
        row_dn[r] = static_cast<int32_t>(r);
    }
}

// Y[t * M + m] = sum_j w[t * top_k + j] * O[(t * top_k + j) * M + m]
// Launched as a programmatic dependent of the down projection: it may be
// resident before that grid ends, and reads O only after the wait.
__global__ void k_moe_combine(const float* __restrict__ O, const float* __restrict__ w, float* __restrict__ Y,
                              int64_t T, int top_k, int64_t M) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t total = T * M;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / M, m = i - t * M;
        const float* o = O + t * top_k * M + m;
        const float* wt = w + t * top_k;
        float acc = 0.f;
        for (int j = 0; j < top_k; ++j) acc = fmaf(wt[j], o[j * M], acc);
        Y[i] = acc;
    }
}

struct MoeScratch {
    int32_t* row_gu;
    int32_t* row_dn;
    float* gu;     // [A][2 d_ff]
    float* dn;     // [A][d_model]
};

size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

MoeScratch carve(void* ws, int64_t A, int64_t d_model, int64_t d_ff) {
    uint8_t* p = static_cast<uint8_t*>(ws);
    MoeScratch m;
    m.row_gu = reinterpret_cast<int32_t*>(p);
    p += up256(static_cast<size_t>(A) * 4);
    m.row_dn = reinterpret_cast<int32_t*>(p);
    p += up256(static_cast<size_t>(A) * 4);
    m.gu = reinterpret_cast<float*>(p);
    p += up256(static_cast<size_t>(A) * 2 * d_ff * 4);
    m.dn = reinterpret_cast<float*>(p);
    return m;
}

}  // namespace

size_t moe_workspace_bytes(int64_t T, int top_k, int64_t d_model, int64_t d_ff) {
    const int64_t A = T * top_k;
    return 2 * up256(static_cast<size_t>(A) * 4) + up256(static_cast<size_t>(A) * 2 * d_ff * 4) +
           up256(static_cast<size_t>(A) * d_model * 4);
}

// Returns a qmm_status value (QMM_OK = queued).
int launch_moe_ffn(int kind, const uint8_t* W_gu, size_t gu_stride, size_t gu_row_bytes, const uint8_t* W_down,
                   size_t down_stride, size_t down_row_bytes, int n_experts, const float* X, int64_t T,
                   int64_t d_model, int64_t d_ff, const int32_t* ids, const float* w, int top_k, float* Y,
                   void* workspace, unsigned* err, cudaStream_t s) {
    const int64_t A = T * top_k;
    const MoeScratch sc = carve(workspace, A, d_model, d_ff);

    Problem pg;   // gate_up: assignment r reads token r / top_k
    pg.kind = kind;
    pg.W = W_gu;
    pg.row_bytes = gu_row_bytes;
    pg.M = 2 * d_ff;
    pg.K = d_model;
    pg.N = A;
    pg.X = X;
    pg.x_dtype = 0;
    pg.Y = sc.gu;
    pg.x_row = sc.row_gu;
    pg.expert_id = ids;
    pg.expert_stride = gu_stride;
    pg.n_experts = n_experts;
    pg.n_x_rows = T;
    pg.err = err;
    Problem pd = pg;   // down: assignment r reads silu(g) * u of gate_up row r
    pd.W = W_down;
    pd.row_bytes = down_row_bytes;
    pd.M = d_model;
    pd.K = d_ff;
    pd.X = sc.gu;
    pd.x_mode = 1;
    pd.x_stride = 2 * d_ff;
    pd.Y = sc.dn;
    pd.x_row = sc.row_dn;
    pd.expert_stride = down_stride;
    pd.n_x_rows = A;
    if (!gemv_stream_ok(pg) || !gemv_stream_ok(pd)) return QMM_ERR_UNIMPLEMENTED;

    const int threads = 256;
    const int b1 = static_cast<int>(imin64((A + threads - 1) / threads, 1024));
    k_moe_rows<<<b1, threads, 0, s>>>(sc.row_gu, sc.row_dn, A, top_k);
    count_launch(1);
    if (cudaGetLastError() != cudaSuccess) return QMM_ERR_CUDA;
    if (launch_gemv_stream(pg, s) != cudaSuccess) return QMM_ERR_CUDA;
    if (launch_gemv_stream(pd, s) != cudaSuccess) return QMM_ERR_CUDA;
    const int64_t total = T * d_model;
    const int b2 = static_cast<int>(imin64((total + threads - 1) / threads, 4096));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(b2));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_moe_combine, static_cast<const float*>(sc.dn), w, Y, T, top_k,
                                             d_model);
    count_launch(1);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace qmm
