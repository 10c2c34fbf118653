// Forward-pass instantiations of the tcgen05 GEMM: fc1 (GELU / SwiGLU epilogue) and fc2.
#include "gemm.cuh"
#include "kernels.h"

namespace mlpb {

cudaError_t gemm_fwd_set_smem_attrs() {
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<GemmKind::FC1_GELU>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_kernel<GemmKind::FC1_SWIGLU>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_kernel<GemmKind::FC2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  return e;
}

cudaError_t launch_gemm_fwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int grid, cudaStream_t s) {
  switch (kind) {
    case GemmKind::FC1_GELU:
      gemm_kernel<GemmKind::FC1_GELU><<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
      break;
    case GemmKind::FC1_SWIGLU:
      gemm_kernel<GemmKind::FC1_SWIGLU><<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
      break;
    case GemmKind::FC2:
      gemm_kernel<GemmKind::FC2><<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mlpb
