// tcgen05 / TMEM tensor-core projection (bf16 operands, fp32 accumulation).
#include "linear.cuh"

namespace llm {

bool gemm_tc_supported(const LinearParams&) { return false; }

cudaError_t launch_gemm_tc(const LinearParams&, int, cudaStream_t, bool) { return cudaErrorNotSupported; }

}  // namespace llm
