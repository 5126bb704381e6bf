// Tensor-core (tcgen05) grouped GEMM kernels. Placeholder until the kernels land: every
// mode reports "no tensor-core kernel" and the stages run the CUDA-core reference kernels.
#include "internal.h"

namespace moe {

bool tc_supported(const Plan&, int) { return false; }

cudaError_t launch_l1_tc(const Plan&, const void*, const void*, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t launch_l2_tc(const Plan&, const void*, const void*, const float*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace moe
