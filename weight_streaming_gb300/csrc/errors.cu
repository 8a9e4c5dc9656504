// See errors.h.
#include "errors.h"

namespace vp {

namespace {
thread_local int g_last_cuda_error = 0;
}

vp_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return VP_ERR_CUDA;
}

int last_cuda_error() { return g_last_cuda_error; }

}  // namespace vp
