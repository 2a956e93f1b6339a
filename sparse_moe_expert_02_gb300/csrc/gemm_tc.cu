// Tensor-core grouped GEMM (placeholder until the tcgen05 kernel lands).
#include "common.cuh"
#include "internal.h"

namespace moe {
bool gemm_tc_supported(const GroupedGemm&) { return false; }
cudaError_t launch_gemm_tc(const GroupedGemm&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace moe
