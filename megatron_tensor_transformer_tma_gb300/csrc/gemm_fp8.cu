// FP8 (E4M3) instantiations of the tcgen05 pair GEMM: all six contractions of the block.
#include "gemm.cuh"
#include "kernels.h"

namespace mlpb {

template <GemmKind K>
static cudaError_t set_attr_f8() {
  return cudaFuncSetAttribute(gemm_pair_kernel<K, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
}

template <GemmKind K>
static cudaError_t launch_f8(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
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
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<K, true>, a, b, p);
}

cudaError_t gemm_f8_set_smem_attrs() {
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = set_attr_f8<GemmKind::FC1_GELU>();
  if (e == cudaSuccess) e = set_attr_f8<GemmKind::FC1_SWIGLU>();
  if (e == cudaSuccess) e = set_attr_f8<GemmKind::FC2>();
  if (e == cudaSuccess) e = set_attr_f8<GemmKind::DGRAD_GELU>();
  if (e == cudaSuccess) e = set_attr_f8<GemmKind::DGRAD_SWIGLU>();
  if (e == cudaSuccess) e = set_attr_f8<GemmKind::DX>();
  if (e == cudaSuccess) e = set_attr_f8<GemmKind::WGRAD_W2>();
  if (e == cudaSuccess) e = set_attr_f8<GemmKind::WGRAD_W1>();
  return e;
}

cudaError_t launch_gemm_f8(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmParams& p, int clusters, cudaStream_t s) {
  switch (kind) {
    case GemmKind::FC1_GELU: return launch_f8<GemmKind::FC1_GELU>(a, b, p, clusters, s);
    case GemmKind::FC1_SWIGLU: return launch_f8<GemmKind::FC1_SWIGLU>(a, b, p, clusters, s);
    case GemmKind::FC2: return launch_f8<GemmKind::FC2>(a, b, p, clusters, s);
    case GemmKind::DGRAD_GELU: return launch_f8<GemmKind::DGRAD_GELU>(a, b, p, clusters, s);
    case GemmKind::DGRAD_SWIGLU: return launch_f8<GemmKind::DGRAD_SWIGLU>(a, b, p, clusters, s);
    case GemmKind::DX: return launch_f8<GemmKind::DX>(a, b, p, clusters, s);
    case GemmKind::WGRAD_W2: return launch_f8<GemmKind::WGRAD_W2>(a, b, p, clusters, s);
    case GemmKind::WGRAD_W1: return launch_f8<GemmKind::WGRAD_W1>(a, b, p, clusters, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mlpb
