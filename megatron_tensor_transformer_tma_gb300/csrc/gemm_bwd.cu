// Backward-pass instantiations of the tcgen05 GEMM: dgrad with the fused activation
// derivative, dX, and the two weight gradients.
#include "gemm.cuh"
#include "kernels.h"

namespace mlpb {

template <GemmKind K>
static cudaError_t set_attr() {
  return cudaFuncSetAttribute(gemm_pair_kernel<K>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
}

// `clusters` clusters of kClusterM CTAs, one CTA per SM.
template <GemmKind K>
static cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                              int clusters, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * kClusterM), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterM;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<K>, a, b, p);
}

cudaError_t gemm_bwd_set_smem_attrs() {
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = set_attr<GemmKind::DGRAD_GELU>();
  if (e == cudaSuccess) e = set_attr<GemmKind::DGRAD_SWIGLU>();
  if (e == cudaSuccess) e = set_attr<GemmKind::DX>();
  if (e == cudaSuccess) e = set_attr<GemmKind::WGRAD_W1>();
  if (e == cudaSuccess) e = set_attr<GemmKind::WGRAD_W2T>();
  return e;
}

cudaError_t launch_gemm_bwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int clusters, cudaStream_t s) {
  switch (kind) {
    case GemmKind::DGRAD_GELU:
      return launch_one<GemmKind::DGRAD_GELU>(a, b, p, clusters, s);
    case GemmKind::DGRAD_SWIGLU:
      return launch_one<GemmKind::DGRAD_SWIGLU>(a, b, p, clusters, s);
    case GemmKind::DX:
      return launch_one<GemmKind::DX>(a, b, p, clusters, s);
    case GemmKind::WGRAD_W1:
      return launch_one<GemmKind::WGRAD_W1>(a, b, p, clusters, s);
    case GemmKind::WGRAD_W2T:
      return launch_one<GemmKind::WGRAD_W2T>(a, b, p, clusters, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace mlpb
