// tc_gemm.cu -- tcgen05 tensor-core GEMM of the 4-bit weight-quantized linear.
#include "q4lin_internal.h"

namespace q4lin {

bool tc_eligible(const Problem&, const LaunchCtx&) { return false; }

cudaError_t tc_launch(const Problem&, const LaunchCtx&) { return cudaErrorNotSupported; }

}  // namespace q4lin
