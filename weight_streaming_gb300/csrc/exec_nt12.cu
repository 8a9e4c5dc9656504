// Instantiations of the streaming executor for 8 and 16 token columns (one translation
// unit per pair so the four variants compile in parallel).
#include <cuda_runtime.h>

#include "exec.cuh"
#include "exec_launch.h"

namespace vp {

template <int NT>
static cudaError_t launch_nt(const Program& prog, const Io& io, int grid, cudaStream_t s, bool coop) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(exec_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = coop ? at : nullptr;
  cfg.numAttrs = coop ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, exec_kernel<NT>, prog, io);
}

cudaError_t launch_exec_nt12(const Program& prog, const Io& io, int NT, int grid, cudaStream_t s, bool coop) {
  return NT == 1 ? launch_nt<1>(prog, io, grid, s, coop) : launch_nt<2>(prog, io, grid, s, coop);
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
