// ttt_linear_tc.cu -- tensor-core TTT-Linear kernel (bf16 I/O, d = 64, b = 16).
#include <cuda_runtime.h>

#include "ttt_internal.h"

namespace ttt {

bool linear_tc_supported(const ttt_desc &) { return false; }

cudaError_t launch_linear_tc(const LinearArgs &) { return cudaErrorNotSupported; }

}  // namespace ttt
