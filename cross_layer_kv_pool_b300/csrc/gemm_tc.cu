// Tensor-core (tcgen05) GEMM engine for bf16 operands.
#include "kernels.h"

namespace wm {

bool gemm_tc_supported(const GemmDesc&) { return false; }
cudaError_t launch_gemm_tc(const GemmDesc&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace wm
