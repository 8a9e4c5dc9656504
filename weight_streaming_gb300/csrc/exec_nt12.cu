// Instantiations of the streaming executor for 8 and 16 token columns (one translation
// unit per pair so the four variants compile in parallel).
#include <cuda_runtime.h>

#include "exec.cuh"
#include "exec_launch.h"

namespace vp {

cudaError_t launch_exec_nt12(const Program& prog, const Io& io, int NT, int grid, cudaStream_t s, bool coop) {
  return NT == 1 ? launch_exec_kernel<1, false>(prog, io, grid, s, coop)
                 : launch_exec_kernel<2, false>(prog, io, grid, s, coop);
}


// The phase timeline of the kernels of this translation unit (traced builds only).
cudaError_t trace_read_nt12(void* dst, size_t bytes, unsigned* launches) {
#ifdef VP_PHASE_TRACE
  if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
  cudaError_t e = cudaMemcpyFromSymbol(dst, g_trace, bytes);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(launches, g_trace_launches, sizeof(unsigned));
  return e;
#else
  (void)dst;
  (void)bytes;
  (void)launches;
  return cudaErrorNotSupported;
#endif
}

}  // namespace vp
