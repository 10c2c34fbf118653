// Backward-pass instantiations of the tcgen05 GEMM: dgrad with the fused activation
// derivative, dX, and the two weight gradients.
#include "gemm.cuh"
#include "kernels.h"

namespace mlpb {

template <GemmKind K>
static cudaError_t set_attr() {
  return cudaFuncSetAttribute(gemm_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kGemmSmem);
}

cudaError_t gemm_bwd_set_smem_attrs() {
  cudaError_t e = set_attr<GemmKind::DGRAD_GELU>();
  if (e == cudaSuccess) e = set_attr<GemmKind::DGRAD_SWIGLU>();
  if (e == cudaSuccess) e = set_attr<GemmKind::DX>();
  if (e == cudaSuccess) e = set_attr<GemmKind::WGRAD_W2>();
  if (e == cudaSuccess) e = set_attr<GemmKind::WGRAD_W1>();
  return e;
}

cudaError_t launch_gemm_bwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int grid, cudaStream_t s) {
  switch (kind) {
    case GemmKind::DGRAD_GELU:
      gemm_kernel<GemmKind::DGRAD_GELU><<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
      break;
    case GemmKind::DGRAD_SWIGLU:
      gemm_kernel<GemmKind::DGRAD_SWIGLU><<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
      break;
    case GemmKind::DX:
      gemm_kernel<GemmKind::DX><<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
      break;
    case GemmKind::WGRAD_W2:
      gemm_kernel<GemmKind::WGRAD_W2><<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
      break;
    case GemmKind::WGRAD_W1:
      gemm_kernel<GemmKind::WGRAD_W1><<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mlpb
