// Forward-pass instantiations of the tcgen05 GEMM: fc1 (GELU / SwiGLU epilogue) and fc2.
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

cudaError_t gemm_fwd_set_smem_attrs() {
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = set_attr<GemmKind::FC1_GELU>();
  if (e == cudaSuccess) e = set_attr<GemmKind::FC1_SWIGLU>();
  if (e == cudaSuccess) e = set_attr<GemmKind::FC2>();
  return e;
}

cudaError_t launch_gemm_fwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int clusters, cudaStream_t s) {
  switch (kind) {
    case GemmKind::FC1_GELU:
      return launch_one<GemmKind::FC1_GELU>(a, b, p, clusters, s);
    case GemmKind::FC1_SWIGLU:
      return launch_one<GemmKind::FC1_SWIGLU>(a, b, p, clusters, s);
    case GemmKind::FC2:
      return launch_one<GemmKind::FC2>(a, b, p, clusters, s);
    default:
      return cudaErrorInvalidValue;
  }
}

// Clusters of kClusterM GEMM CTAs that can be resident at once on this device.
cudaError_t gemm_max_active_clusters(int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kClusterM, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterM;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, gemm_pair_kernel<GemmKind::FC1_GELU>, &cfg);
}

}  // namespace mlpb
