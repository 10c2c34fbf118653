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

// Sums the tail tiles' partial K-ranges in part order and applies the fp32 epilogue of
// FC2 / DX / WGRAD_W1: Y[m][n] = ((sum_p P_p) + bias[n]) + resid[m][n] (bias, resid
// optional), or Y[m][n] += sum_p P_p when accumulating.  Y is [M][H] (dW1: M = F1), fp32,
// or bf16 for FC2 / DX with out_bf16.  A CTA covers 8 rows x 256 columns of one CTA half
// of one tile; a thread 8 columns.
__global__ void __launch_bounds__(256) split_fixup_kernel(const GemmParams p) {
  const int tiles_rows = kBM / 8;  // row groups a CTA half
  const int j = blockIdx.x / (2 * tiles_rows);
  const int rank = (blockIdx.x / tiles_rows) & 1;
  const int r = (blockIdx.x % tiles_rows) * 8 + threadIdx.x / 32;
  const int c = (threadIdx.x & 31) * 8;
  const int num_pm = (p.num_m_tiles + 1) / 2;
  int mp, nt;
  tile_coords(p.split_start + j, num_pm, p.num_n_tiles, p.raster_group, mp, nt);
  const int m = (mp * 2 + rank) * kBM + r;
  const int n = nt * kBN + c;
  if (m >= p.M || n >= p.H) return;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int part = 0; part < p.split; ++part) {
    const float* P = p.partial +
                     ((static_cast<size_t>(j) * p.split + part) * 2 + rank) * (kBM * kBN) +
                     static_cast<size_t>(r) * kBN + c;
    const float4 a = __ldcg(reinterpret_cast<const float4*>(P));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(P + 4));
    v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
    v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
  }
  if (p.bias != nullptr) {
    const uint4 u = ld_global_nc_v4(p.bias + n);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16x2(w[e]);
      v[2 * e] += f.x;
      v[2 * e + 1] += f.y;
    }
  }
  if (p.aux != nullptr) {
    const uint4 u = ld_global_nc_v4(p.aux + static_cast<size_t>(m) * p.H + n);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16x2(w[e]);
      v[2 * e] += f.x;
      v[2 * e + 1] += f.y;
    }
  }
  if (p.out_bf16) {  // one rounding of the finished fp32 sum
    __nv_bfloat16* Yb = static_cast<__nv_bfloat16*>(p.out0) + static_cast<size_t>(m) * p.H + n;
    st_global_v4(Yb, make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7])));
    return;
  }
  float* Y = static_cast<float*>(p.out0) + static_cast<size_t>(m) * p.H + n;
  if (p.accumulate) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(Y));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(Y + 4));
    v[0] = a.x + v[0]; v[1] = a.y + v[1]; v[2] = a.z + v[2]; v[3] = a.w + v[3];
    v[4] = b.x + v[4]; v[5] = b.y + v[5]; v[6] = b.z + v[6]; v[7] = b.w + v[7];
  }
  st_global_v4(Y, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                             __float_as_uint(v[3])));
  st_global_v4(Y + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]),
                                 __float_as_uint(v[6]), __float_as_uint(v[7])));
}

cudaError_t launch_split_fixup(const GemmParams& p, cudaStream_t s) {
  const int num_pm = (p.num_m_tiles + 1) / 2;
  const int tail = num_pm * p.num_n_tiles - p.split_start;
  if (p.split <= 1 || tail <= 0) return cudaSuccess;
  split_fixup_kernel<<<tail * 2 * (kBM / 8), 256, 0, s>>>(p);
  return cudaGetLastError();
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
