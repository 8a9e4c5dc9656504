// The library's CUDA-error bookkeeping, shared by the translation units that hold entry points:
// cuda_fail records the error for vp_get_last_cuda_error (per host thread) and returns VP_ERR_CUDA.
#pragma once
#include <cuda_runtime.h>

#include "verify.h"

namespace vp {

vp_status cuda_fail(cudaError_t e);
int last_cuda_error();

}  // namespace vp
