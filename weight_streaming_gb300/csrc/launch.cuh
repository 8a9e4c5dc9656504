// Launch helper for the GEMM kernel instantiations (one translation unit per weight format).
#pragma once
#include <cuda_runtime.h>

#include "gemm.cuh"

namespace vp {

template <int FMT, int MT>
cudaError_t launch_gemm_mt(const GemmParams& p, int grid, cudaStream_t stream, bool pdl) {
  auto kern = gemm_kernel<FMT, MT>;
  constexpr size_t smem = gemm_smem_bytes<FMT>();
  static int configured_mask = 0;  // one bit per device ordinal < 32
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 32 && !(configured_mask & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_mask |= 1 << dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int FMT>
cudaError_t launch_gemm_fmt(const GemmParams& p, int mt, int grid, cudaStream_t stream, bool pdl) {
  switch (mt) {
    case 1: return launch_gemm_mt<FMT, 1>(p, grid, stream, pdl);
    case 2: return launch_gemm_mt<FMT, 2>(p, grid, stream, pdl);
    case 3: return launch_gemm_mt<FMT, 3>(p, grid, stream, pdl);
    case 4: return launch_gemm_mt<FMT, 4>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_nvfp4(const GemmParams& p, int mt, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_gemm_fp8(const GemmParams& p, int mt, int grid, cudaStream_t stream, bool pdl);

}  // namespace vp
