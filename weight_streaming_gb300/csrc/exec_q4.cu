// Instantiations of the streaming executor with the Q4 (affine 4-bit, group 64) unit, for 8..32
// token columns.
#include <cuda_runtime.h>

#include "exec.cuh"
#include "exec_launch.h"

namespace vp {

cudaError_t launch_exec_q4(const Program& prog, const Io& io, int NT, int grid, cudaStream_t s, bool coop) {
  switch (NT) {
    case 1: return launch_exec_kernel<1, true>(prog, io, grid, s, coop);
    case 2: return launch_exec_kernel<2, true>(prog, io, grid, s, coop);
    case 3: return launch_exec_kernel<3, true>(prog, io, grid, s, coop);
    default: return launch_exec_kernel<4, true>(prog, io, grid, s, coop);
  }
}

}  // namespace vp
