// Host-side entry of the streaming executor (exec.cuh), instantiated in exec_nt12.cu / exec_nt34.cu
// (NVFP4 / FP8 phases) and exec_q4.cu (Q4 phases).
#pragma once
#include <cuda_runtime.h>

#include "internal.h"

namespace vp {

cudaError_t launch_exec_nt12(const Program& prog, const Io& io, int NT, int grid, cudaStream_t s, bool coop);
cudaError_t launch_exec_nt34(const Program& prog, const Io& io, int NT, int grid, cudaStream_t s, bool coop);
cudaError_t launch_exec_q4(const Program& prog, const Io& io, int NT, int grid, cudaStream_t s, bool coop);
// Copies the phase timeline of the NT = 1-2 / 3-4 kernels (trace.cuh) and the count of completed
// launches; cudaErrorNotSupported unless the library was built with VP_PHASE_TRACE.
cudaError_t trace_read_nt12(void* dst, size_t bytes, unsigned* launches);
cudaError_t trace_read_nt34(void* dst, size_t bytes, unsigned* launches);

// Runs `prog` (NT = ceil(M / 8) n-tiles of 8 tokens) on `grid` CTAs; cooperative when the program
// has grid barriers (more than one phase, or a phase cut into K slices), so that every CTA is
// resident.
inline cudaError_t launch_exec(const Program& prog, const Io& io, int grid, cudaStream_t s) {
  const int NT = (prog.M + 7) / 8;
  bool coop = prog.n > 1;
  for (int i = 0; i < prog.n && !coop; ++i) coop = prog.ph[i].ks > 1;
  if (prog.q4) return launch_exec_q4(prog, io, NT, grid, s, coop);
  return NT <= 2 ? launch_exec_nt12(prog, io, NT, grid, s, coop) : launch_exec_nt34(prog, io, NT, grid, s, coop);
}

}  // namespace vp
