// NVFP4 instantiations of the verify-pass GEMM (M tiles 1..4).
#include "launch.cuh"

namespace vp {
cudaError_t launch_gemm_nvfp4(const GemmParams& p, int mt, int grid, cudaStream_t stream, bool pdl) {
  return launch_gemm_fmt<kFmtNvfp4>(p, mt, grid, stream, pdl);
}
}  // namespace vp
