// Host-side declarations of the GEMM launchers (defined in gemm_nvfp4.cu / gemm_fp8.cu).
#pragma once
#include <cuda_runtime.h>

#include "internal.h"

namespace vp {
cudaError_t launch_gemm_nvfp4(const GemmParams& p, int mt, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_gemm_fp8(const GemmParams& p, int mt, int grid, cudaStream_t stream, bool pdl);
}  // namespace vp
