// k_gemm_tc.cu -- tcgen05 tensor-core quantized GEMM (prefill shapes).
#include "qmm_internal.cuh"

namespace qmm {

bool gemm_tc_ok(const Problem&) { return false; }

cudaError_t launch_gemm_tc(const Problem&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace qmm
