/*
 * qmm.h -- C ABI of libqmm: block-quantized weights times dense activations,
 * with the dequantization fused into the kernels, on one NVIDIA GB300 (sm_103a).
 *
 * The problem statement follows ferrox-cuda 0.21.0 src/mul_mm.rs (the `BODY_SRC`
 * GEMM body and `validate_shape`): a weight matrix of `M` rows, each row a run of
 * `K / block_elems` contiguous blocks in their on-disk (GGUF) byte layout; `N`
 * activation rows of `K` values; an fp32 output written token-major,
 * Y[n * M + m] = sum_k W[m, k] * X[n * K + k].
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers (cudaMalloc / PyTorch CUDA tensors)
 *     on the current CUDA device. The library never takes ownership; the caller
 *     keeps every buffer alive until the work queued on `stream` has finished.
 *     qdequant, qgemv, qgemm_grouped and qgemm_noalloc never allocate device
 *     memory. qgemm (and qgemm_ex) with N > 8 on the tensor-core path may grow
 *     a per-device workspace that the library owns (see qgemm); qmm_shutdown
 *     frees it.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call
 *     is asynchronous with respect to the host: it validates, queues kernels on
 *     `stream` and returns.
 *   - Errors in arguments (shape, kind, dtype, null or misaligned pointers, too
 *     small buffers) are reported synchronously as a qmm_status BEFORE anything
 *     is launched; nothing is written. A zero-sized shape is QMM_ERR_EMPTY_SHAPE
 *     and launches nothing (ferrox-cuda mul_mm.rs, `MulMmUnsupported::EmptyShape`).
 *   - A failed launch returns QMM_ERR_CUDA. Device-side conditions (a bounded
 *     wait that ran out) are latched in a device flag and reported by
 *     qmm_check_device_error().
 *   - There is no fallback to a different computation and no CPU path: a format
 *     this library does not implement is QMM_ERR_BAD_KIND (ferrox-cuda
 *     mul_mm.rs, `kind_by_name`: an unknown format is reported to the caller,
 *     who chooses another implementation).
 *   - Every output element is written exactly once per call (no accumulation
 *     into the output), so sentinel-prefilled outputs are fully overwritten.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Block formats. Geometry (bytes per block / elements per block):
 *   Q8_0 34/32, Q4_0 18/32, Q5_0 22/32, Q4_K 144/256, Q5_K 176/256,
 *   Q6_K 210/256, Q2_K 84/256, Q3_K 110/256, IQ4_NL 18/32, IQ4_XS 136/256,
 *   MXFP4 17/32 (ferrox-cuda mul_mm.rs `KINDS` and its geometry test;
 *   ferrox-cuda 0.20.0 src/mul_mm_kinds/codebook.rs for the codebook rows;
 *   Vulkore examples/llm/quant_test.cpp `kFormats`);
 *   Q4_1 20/32, Q5_1 24/32, Q8_1 36/32: the kinds that ferrox-cuda 0.21.0
 *   mul_mm.rs lists as having no mul_mm kernel, in the public GGUF layouts --
 *   Q4_1 and Q5_1 are Q4_0 and Q5_0 with unsigned codes and an f16 min after
 *   the f16 scale (w = d*q + m); Q8_1 is Q8_0 with an f16 field after d (d
 *   times the sum of the codes) that no element reads (w = d*q). */
typedef enum {
    QMM_Q8_0 = 0,
    QMM_Q4_0 = 1,
    QMM_Q5_0 = 2,
    QMM_Q4_K = 3,
    QMM_Q5_K = 4,
    QMM_Q6_K = 5,
    QMM_Q2_K = 6,
    QMM_Q3_K = 7,
    QMM_IQ4_NL = 8,
    QMM_IQ4_XS = 9,
    QMM_MXFP4 = 10,
    QMM_Q4_1 = 11,
    QMM_Q5_1 = 12,
    QMM_Q8_1 = 13,
    QMM_NKINDS = 14
} qmm_kind;

/* Activation element type. f32 activations must be 4-byte aligned, f16
 * activations (IEEE binary16) 2-byte aligned. */
typedef enum { QMM_F32 = 0, QMM_F16 = 1 } qmm_dtype;

/* Status codes. The shape refusals mirror ferrox-cuda mul_mm.rs
 * `MulMmUnsupported`. */
typedef enum {
    QMM_OK = 0,
    QMM_ERR_EMPTY_SHAPE = 1,             /* M, K, N or n_assign is 0 */
    QMM_ERR_BAD_KIND = 2,                /* kind outside qmm_kind */
    QMM_ERR_BAD_DTYPE = 3,               /* x_dtype outside qmm_dtype */
    QMM_ERR_COLS_NOT_BLOCK_ALIGNED = 4,  /* K not a multiple of block_elems */
    QMM_ERR_WEIGHTS_TOO_SMALL = 5,       /* w_bytes < M * row_bytes (or experts) */
    QMM_ERR_ACTIVATIONS_TOO_SMALL = 6,   /* x_elems < rows needed * K */
    QMM_ERR_NULL_POINTER = 7,
    QMM_ERR_MISALIGNED = 8,              /* activation/output pointer alignment */
    QMM_ERR_BAD_EXPERT_ID = 9,           /* bad n_experts / expert stride */
    QMM_ERR_CUDA = 10,                   /* a CUDA runtime call failed */
    QMM_ERR_DEVICE_TIMEOUT = 11,         /* a device-side bounded wait ran out */
    QMM_ERR_UNIMPLEMENTED = 12,
    QMM_ERR_BAD_ARGUMENT = 13,           /* negative size or other bad scalar */
    QMM_ERR_OUTPUT_TOO_SMALL = 14,       /* y_elems < outputs to write */
    QMM_ERR_WORKSPACE_IN_CAPTURE = 15,   /* workspace would grow during stream capture */
    QMM_ERR_NOALLOC_LIMIT = 16,          /* qgemm_noalloc: scratch needed exceeds its fixed array */
    QMM_ERR_WORKSPACE_TOO_SMALL = 17     /* caller-provided workspace smaller than required */
} qmm_status;

/* Geometry of `kind`: bytes and elements of one block. Returns QMM_OK or
 * QMM_ERR_BAD_KIND / QMM_ERR_NULL_POINTER. Host only, no CUDA call. */
QMM_API int qmm_kind_info(int kind, size_t* block_bytes, size_t* block_elems);

/* Bytes of one weight row of K elements: (K / block_elems) * block_bytes.
 * 0 when kind is bad or K is not a positive multiple of block_elems. */
QMM_API size_t qmm_row_bytes(int kind, int64_t K);

/* Static, NUL-terminated description of a status code (never NULL). */
QMM_API const char* qmm_status_str(int status);

/* GGUF name of a kind ("Q4_0", ...), or NULL for a bad kind. */
QMM_API const char* qmm_kind_name(int kind);

/*
 * qdequant -- expand `rows` x `cols` quantized weights to fp32.
 *
 *   out[r * cols + k] = value of element k of weight row r
 *
 * Element values follow each format's definition (Vulkore quant_test.cpp, the
 * `ref::` CPU references; ferrox-cuda codebook.rs for IQ4_NL / IQ4_XS / MXFP4).
 * Bit-exact: every product in every format is exact in fp32; the affine-min
 * formats (Q4_K, Q5_K, Q2_K) round once, at the final subtraction. No flush of
 * subnormals (MXFP4 with small E8M0 scales yields fp32 subnormals).
 *
 *   blocks       device, rows * qmm_row_bytes(kind, cols) bytes, any alignment
 *   blocks_bytes size of `blocks` in bytes (checked)
 *   out          device fp32, rows * cols elements, 4-byte aligned
 *   out_elems    size of `out` in elements (checked)
 */
QMM_API int qdequant(int kind, const void* blocks, size_t blocks_bytes, int64_t rows, int64_t cols,
             float* out, size_t out_elems, void* stream);

/*
 * qgemv -- decode GEMV, y[m] = sum_k W[m, k] * x[k] (one activation row).
 * Exactly qgemm with N = 1 (inferencelayer 0.2.8 src/cublas_prefill.rs,
 * `Q4_GEMV_KERNEL`: the decode-time GEMV, bound by reading the weights).
 *
 *   W        device, M * row_bytes bytes, any alignment (16-byte aligned W with
 *            16-byte-multiple rows takes the streaming fast path)
 *   w_bytes  size of W in bytes (checked)
 *   x        device, K activations of x_dtype
 *   x_elems  size of x in elements (checked)
 *   y        device fp32, M elements, 4-byte aligned; y_elems its size
 */
QMM_API int qgemv(int kind, const void* W, size_t w_bytes, const void* x, int x_dtype, size_t x_elems,
          float* y, size_t y_elems, int64_t M, int64_t K, void* stream);

/*
 * qgemm -- Y[n * M + m] = sum_k W[m, k] * X[n * K + k] for n < N, m < M
 * (ferrox-cuda mul_mm.rs `BODY_SRC`: src0 = W, src1 = X, dst token-major).
 * Small N runs the weight-streaming GEMV kernels; large N the tcgen05
 * tensor-core GEMM. fp32 activations reach the tensor cores as two f16 rows
 * per token: a pre-pass scales each token row by the power of two that puts
 * its largest magnitude in [2^9, 2^10) and splits it into hi = f16(x) and
 * lo = f16(x - hi) (together exact to about 2^-22 relative); the epilogue adds
 * the two products and removes the scale. This doubles the tensor-core work of
 * the call against f16 activations. With f16 activations, Q4_K, Q5_K, Q2_K,
 * Q4_1 and Q5_1 carry the sums of each 32 (Q2_K: 16) consecutive activations
 * in f16: their magnitudes must stay below 65504.
 *
 *   W, w_bytes   as qgemv
 *   X            device, N * K activations of x_dtype, row-major; x_elems its size
 *   Y            device fp32, N * M elements; y_elems its size
 *
 * Accuracy: |Y - Y_exact| <= 1e-3 * sum_k |W[m,k] * X[n,k]| + 1e-6 per element.
 * One condition on the tensor-core path: MXFP4 folds each block's exponent
 * into its f16 operands relative to the largest exponent of its 256-element
 * group. This is exact while the eight exponents of a group span at most 23.
 * At 24 the codes +-0.5 and +-1.5 of the smallest block round to even; a block
 * 25 or more below the largest contributes nothing. The bound then holds while
 * the group's largest-exponent block carries a nonzero code against
 * activations of comparable magnitude (quantizers derive a block's exponent
 * from its largest value). The GEMV (N <= 8) and qdequant have no such limit.
 *
 * Workspace: the tensor-core path keeps its scratch in a per-device workspace
 * the library owns and grows on demand (cudaMalloc): the f16 (hi, lo) rows of
 * fp32 activations and their scales (4 * N * K + 4 * N bytes), for Q4_K,
 * Q5_K, Q2_K, Q4_1 and Q5_1 the per-group activation sums (N * K/16 f16
 * values at most, twice that for fp32 activations), and, when the
 * 128 x 128 output tiles do not fill the GPU evenly, the partial tiles of
 * the tiles whose K range several CTAs share (2 * 64 KiB per SM). Those
 * partial sums are added in a fixed order by a second kernel, so results are
 * deterministic. Growth is refused during stream capture
 * (QMM_ERR_WORKSPACE_IN_CAPTURE): make one call of the largest shape before
 * capturing. Concurrent calls on different streams of one device share that
 * workspace and must not overlap.
 */
QMM_API int qgemm(int kind, const void* W, size_t w_bytes, const void* X, int x_dtype, size_t x_elems,
          float* Y, size_t y_elems, int64_t M, int64_t K, int64_t N, void* stream);

/* Per-call flags of qgemm_ex. */
enum {
    /* W is not written by any work still in flight on `stream` (the normal
     * case for model weights). The weight-streaming GEMV (N <= 8) may then
     * start reading W while the preceding kernel on the stream is still
     * running (programmatic dependent launch); activations are read, and
     * outputs written, only after that kernel has completed, with or without
     * the flag. Other paths ignore it. */
    QMM_FLAG_WEIGHTS_CONST = 1,
    /* Y holds IEEE binary16 (QMM_FLAG_Y_F16) or bfloat16 (QMM_FLAG_Y_BF16)
     * values instead of fp32: each output is the fp32 result rounded to
     * nearest even once, at the store. Y must then be 2-byte aligned and
     * y_elems counts 16-bit elements. At most one of the two. */
    QMM_FLAG_Y_F16 = 2,
    QMM_FLAG_Y_BF16 = 4
};

/*
 * qgemm_ex -- qgemm with per-call flags (a bitwise OR of QMM_FLAG_* values;
 * unknown bits are QMM_ERR_BAD_ARGUMENT). qgemm and qgemv are qgemm_ex with
 * flags 0.
 */
QMM_API int qgemm_ex(int kind, const void* W, size_t w_bytes, const void* X, int x_dtype, size_t x_elems,
                     float* Y, size_t y_elems, int64_t M, int64_t K, int64_t N, uint32_t flags,
                     void* stream);

/*
 * qgemm_noalloc -- qgemm on the tensor-core path that never allocates device
 * memory. The pages have no counterpart to it. It is for callers that cannot
 * let a library call cudaMalloc: serving runtimes that reserve all of the
 * GPU's memory at start-up and hand out only their own pools (a cudaMalloc
 * from a library then fails or steals from the pool), and callers on a hot
 * path where an allocation's implicit device synchronisation is not allowed.
 *
 * It computes what qgemm computes, with the same arguments, layouts and
 * accuracy (one CTA per output tile, never shared K ranges, so the rounding
 * of the sums can differ from qgemm's), but only on the tensor-core path:
 * f16 activations, K a multiple of 256, 16-byte aligned W and X, rows a
 * multiple of 16 bytes (QMM_ERR_UNIMPLEMENTED otherwise). The per-group
 * activation sums that Q4_K, Q5_K, Q2_K, Q4_1 and Q5_1 need go to a fixed
 * 4 MiB device array compiled into the library (held on every GPU that loads
 * it, until the process exits) instead of a grown workspace; a problem whose
 * sums need more, N * (K / 256) * 32 bytes for Q4_K / Q5_K / Q4_1 / Q5_1 or
 * N * (K / 256) * 64 bytes for Q2_K above 4 MiB, returns QMM_ERR_NOALLOC_LIMIT
 * before anything is launched. Each call rewrites all the scratch it reads,
 * so nothing is left to clear between calls. The array is shared by every call: calls that can
 * overlap on the GPU (different streams, same device) race on it and must
 * be ordered by the caller. The first call on a device looks the array's
 * address up with cudaGetSymbolAddress (no allocation), once per device.
 */
QMM_API int qgemm_noalloc(int kind, const void* W, size_t w_bytes, const void* X, int x_dtype,
                          size_t x_elems, float* Y, size_t y_elems, int64_t M, int64_t K, int64_t N,
                          void* stream);

/*
 * qgemm_grouped -- expert-indexed product (a mixture-of-experts layer's
 * routed matmul). For each assignment r < n_assign:
 *
 *   Y[r * M + m] = sum_k W_e[m, k] * X[x_row[r] * K + k],  e = expert_id[r]
 *
 * where W_e = W + e * expert_stride bytes holds expert e's M x K weights. Each
 * assignment writes its own output row (no top-k combine).
 *
 * On the weight-streaming kernel, the assignments are bucketed by expert on
 * the device. Every touched expert's rows are then read from memory once per
 * block of up to four of its assignments. That kernel needs 16-byte aligned W,
 * expert_stride and row bytes multiples of 16, n_experts <= 1024 and
 * n_assign <= 4096. Other shapes run on the generic kernel, one pass per
 * assignment. Accuracy is as for qgemm.
 *
 *   W               device, n_experts experts of M rows each; w_bytes its size
 *   expert_stride   bytes between experts (>= M * row_bytes)
 *   X               device activations, n_x_rows rows of K; x_elems its size
 *   x_row, expert_id device int32 arrays of n_assign entries. Values are read
 *                   on the device: an out-of-range expert id or x row makes
 *                   that assignment's output row NaN and latches
 *                   QMM_ERR_BAD_EXPERT_ID for qmm_check_device_error().
 *   Y               device fp32, n_assign * M elements; y_elems its size
 */
QMM_API int qgemm_grouped(int kind, const void* W, size_t w_bytes, size_t expert_stride, int n_experts,
                  const void* X, int x_dtype, size_t x_elems, int64_t n_x_rows,
                  const int32_t* x_row, const int32_t* expert_id, int64_t n_assign,
                  float* Y, size_t y_elems, int64_t M, int64_t K, void* stream);

/*
 * qrepack -- load-time repack of Q8_0 / Q4_0 weights into the layout
 * qgemm_repacked reads (the Vulkore examples/llm/quant_test.cpp page's
 * repacked fast path: scales split from codes, everything aligned, checked to
 * reconstruct every element bit-exactly). Rows stay contiguous and keep their
 * byte count; each 256-element unit of a row holds the code fields of its
 * eight blocks back to back (16 bytes per Q4_0 block, 32 per Q8_0 block, in
 * the block's own element order), then the eight f16 scales (16 bytes).
 *
 *   W, w_bytes     device, rows x cols native blocks
 *   out, out_bytes device, qrepack_bytes(kind, rows, cols) bytes (the same
 *                  size as the native tensor); any alignment for W and out,
 *                  16 bytes for qgemm_repacked
 * cols must be a multiple of 256; other kinds are QMM_ERR_UNIMPLEMENTED.
 */
QMM_API int qrepack(int kind, const void* W, size_t w_bytes, int64_t rows, int64_t cols, void* out,
                    size_t out_bytes, void* stream);

/* Bytes of the repacked tensor (0 for an unsupported kind or shape). */
QMM_API size_t qrepack_bytes(int kind, int64_t rows, int64_t cols);

/*
 * qgemm_repacked -- qgemm (N <= 8 activation rows) on a tensor repacked by
 * qrepack, with the reduction over K optionally split: split ways of K / split
 * elements each (split a divisor of K / 256; 0 = chosen so that every SM gets
 * about two items of rows; 1 = not split). Each K-slice of every row is
 * streamed by its own CTA work item and the partial products are added by a
 * second kernel in slice order (deterministic), the split-k matvec plus
 * reduce of the same page. flags as qgemm_ex.
 *
 * Scratch for split > 1 (the partial products, split * N * M fp32) lives in a
 * per-device workspace the library grows on demand; growth during stream
 * capture is refused (QMM_ERR_WORKSPACE_IN_CAPTURE), qmm_shutdown frees it.
 */
QMM_API int qgemm_repacked(int kind, const void* R, size_t r_bytes, const void* X, int x_dtype, size_t x_elems,
                           float* Y, size_t y_elems, int64_t M, int64_t K, int64_t N, int split, uint32_t flags,
                           void* stream);

/*
 * qmoe_ffn -- one mixture-of-experts feed-forward layer over block-quantized
 * experts (the decoder layer whose per-token weight traffic the inferencelayer
 * 0.2.8 src/cublas_prefill.rs page quotes for Qwen3-30B-A3B). For token t and
 * routing slot j < top_k, with e = topk_ids[t * top_k + j] and weight
 * topk_w[t * top_k + j]:
 *
 *   g, u = rows [0, d_ff) and [d_ff, 2 d_ff) of W_gu_e times x_t
 *   h    = silu(g) * u,   silu(v) = v / (1 + e^-v)          (SwiGLU)
 *   o    = W_down_e h
 *   Y[t] = sum_j topk_w[t * top_k + j] * o                 (in slot order)
 *
 * The projections run on the expert-grouped streaming GEMV (each touched
 * expert's rows stream once per block of up to four of its assignments); the
 * down projection computes silu(g) * u while it stages its activations. The
 * routing weights are applied as given (normalise them first if the model
 * does). Accuracy: within what qgemm's per-product bar implies through SwiGLU
 * and the down projection.
 *
 *   W_gu, w_gu_bytes     device, n_experts experts every gu_stride bytes, each
 *                        2 d_ff rows of d_model elements (gate rows first)
 *   W_down, w_down_bytes device, experts every down_stride bytes, each d_model
 *                        rows of d_ff elements
 *   X                    device fp32 [T][d_model], 16-byte aligned
 *   topk_ids, topk_w     device int32 / fp32 [T][top_k]; an expert id out of
 *                        range gives NaN in its token's row of Y and latches
 *                        QMM_ERR_BAD_EXPERT_ID for qmm_check_device_error()
 *   Y                    device fp32 [T][d_model]
 *   workspace            device scratch owned by the caller, 256-byte aligned,
 *                        at least qmoe_ffn_workspace_bytes(T, top_k, d_model,
 *                        d_ff) bytes; the library allocates nothing. Calls that
 *                        overlap on the GPU must not share a workspace.
 *
 * Both projections must take the streaming kernel: 16-byte aligned weights,
 * strides and rows that are multiples of 16 bytes, n_experts <= 1024 and
 * T * top_k <= 4096 (QMM_ERR_UNIMPLEMENTED otherwise).
 */
QMM_API int qmoe_ffn(int kind, const void* W_gu, size_t w_gu_bytes, size_t gu_stride, const void* W_down,
                     size_t w_down_bytes, size_t down_stride, int n_experts, const float* X, size_t x_elems,
                     int64_t T, int64_t d_model, int64_t d_ff, const int32_t* topk_ids, const float* topk_w,
                     int top_k, float* Y, size_t y_elems, void* workspace, size_t workspace_bytes, void* stream);

/* Scratch bytes qmoe_ffn needs for these sizes (0 for a non-positive size). */
QMM_API size_t qmoe_ffn_workspace_bytes(int64_t T, int top_k, int64_t d_model, int64_t d_ff);

/*
 * qmm_check_device_error -- synchronize `stream`, then read and clear the
 * device-side error latch of the current device. Returns QMM_OK,
 * QMM_ERR_DEVICE_TIMEOUT (a bounded wait in a kernel ran out; that kernel's
 * output is unspecified), QMM_ERR_BAD_EXPERT_ID, or QMM_ERR_CUDA.
 */
QMM_API int qmm_check_device_error(void* stream);

/*
 * qmm_selftest_wait_timeout -- test of the failure path (the pages have no
 * counterpart). Queues on `stream` one small kernel that waits on a shared-
 * memory barrier nothing ever completes, gives up after `cycles` SM clock
 * cycles (1 .. 2^32), and latches the same timeout status a real kernel's
 * bounded wait would. The next qmm_check_device_error() then returns
 * QMM_ERR_DEVICE_TIMEOUT and clears it; the CUDA context stays usable. No
 * trap, fault or unbounded wait is involved. Returns QMM_OK, or
 * QMM_ERR_BAD_ARGUMENT / QMM_ERR_CUDA without launching.
 */
QMM_API int qmm_selftest_wait_timeout(int64_t cycles, void* stream);

/* Kernel-path override, for tests and experiments: 0 = automatic (default),
 * 1 = force the generic CUDA-core kernels, 2 = force the streaming GEMV for
 * qgemm (N <= 8), 3 = force the tensor-core GEMM for qgemm. Applies to the
 * later calls of the calling host thread only (thread-local). Returns that
 * thread's previous value, or -1 for an unknown value (setting unchanged). */
QMM_API int qmm_set_path(int path);

/* Which kernel family the most recent successful call on this host thread
 * launched: 1 generic, 2 streaming GEMV, 3 tensor-core GEMM, 4 dequant,
 * 5 grouped GEMV, 6 MoE layer, 7 repacked (split-K) GEMV; 0 before any call. */
QMM_API int qmm_last_path(void);

/* Number of kernels this library has launched since load (all threads). */
QMM_API uint64_t qmm_launch_count(void);

/*
 * qmm_shutdown -- frees the per-device workspaces qgemm grows (activation
 * sums, partial tiles; see qgemm) on every device that has one, and forgets
 * the device addresses of the library's own device arrays (its error latch
 * and qgemm_noalloc's scratch), which the next call looks up again. cudaFree
 * waits for the work in flight on that device first. Later calls grow the
 * workspaces again as needed. Call it before anything that tears down a
 * device's context (cudaDeviceReset): addresses cached across that would be
 * stale. Not to be called while another thread is inside the library.
 * Returns QMM_OK, or QMM_ERR_CUDA if a free failed (the remaining ones are
 * still attempted). The current device is left as it was.
 */
QMM_API int qmm_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
