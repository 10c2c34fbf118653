// Sequence-parallel LayerNorm forward and backward.
//
// Forward: one CTA per row, ceil(H/16) threads (a multiple of 32, at most 1024); each
// thread keeps two 16-byte bf16 vectors of the row in registers, so mean and variance are
// two passes over registers (warp shuffles, then one value per warp through shared
// memory).  Sequence shard s owns rows [s T/t, (s+1) T/t); rows are independent, so the
// shard structure only matters for the parameter gradients.
//
// Backward: a grid of t x B CTAs; CTA (s, b) walks rows b, b+B, ... of shard s, computes
// dx = rstd (g - mean(g) - xhat mean(g xhat)) with g = dy gamma, and accumulates its own
// dgamma/dbeta partials in registers.  The partials [t*B][H] are then summed in shard
// order (the all-reduce of per-shard partials), deterministically.
#include "common.cuh"
#include "kernels.h"

namespace mlpb {

// kLnVpt: 16-byte vectors (8 elements) per thread; 2 for H <= 8192, 4 for H <= 16384,
// with at most 512 threads per CTA.
constexpr int kLnMaxThreads = 512;

template <int NV>
__device__ __forceinline__ void block_sum(float (&v)[NV], float* sh /* [32*NV] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
  __syncthreads();  // `sh` may still be read from a previous call
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < NV; ++k) sh[warp * NV + k] = v[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += sh[w * NV + k];
    v[k] = s;
  }
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = unpack_bf16x2(w[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

template <int kLnVpt>
__global__ void __launch_bounds__(kLnMaxThreads) ln_fwd_kernel(const __nv_bfloat16* __restrict__ X,
                                                      const __nv_bfloat16* __restrict__ gamma,
                                                      const __nv_bfloat16* __restrict__ beta,
                                                      __nv_bfloat16* __restrict__ Xn,
                                                      float* __restrict__ mean,
                                                      float* __restrict__ rstd, int H,
                                                      float eps) {
  __shared__ float sh[32];
  const int64_t row = blockIdx.x;
  const __nv_bfloat16* x = X + row * H;
  float v[kLnVpt][8];
  bool ok[kLnVpt];
  float s[1] = {0.f};
#pragma unroll
  for (int k = 0; k < kLnVpt; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    ok[k] = c < H;
    uint4 u = make_uint4(0, 0, 0, 0);
    if (ok[k]) u = ld_global_nc_v4(x + c);
    bf16x8_to_f32(u, v[k]);
#pragma unroll
    for (int e = 0; e < 8; ++e) s[0] += v[k][e];
  }
  block_sum<1>(s, sh);
  const float mu = s[0] / static_cast<float>(H);
  float q[1] = {0.f};
#pragma unroll
  for (int k = 0; k < kLnVpt; ++k)
    if (ok[k])
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = v[k][e] - mu;
        q[0] += d * d;
      }
  block_sum<1>(q, sh);
  const float r = rsqrtf(q[0] / static_cast<float>(H) + eps);
#pragma unroll
  for (int k = 0; k < kLnVpt; ++k) {
    if (!ok[k]) continue;
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    float g[8], b[8], o[8];
    bf16x8_to_f32(ld_global_nc_v4(gamma + c), g);
    bf16x8_to_f32(ld_global_nc_v4(beta + c), b);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = (v[k][e] - mu) * r * g[e] + b[e];
    st_global_v4(Xn + row * H + c, make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                              pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7])));
  }
  if (threadIdx.x == 0) {
    mean[row] = mu;
    rstd[row] = r;
  }
}

template <int kLnVpt>
__global__ void __launch_bounds__(kLnMaxThreads) ln_bwd_kernel(
    const __nv_bfloat16* __restrict__ X, const __nv_bfloat16* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd,
    const float* __restrict__ dXn, float* __restrict__ dX, float* __restrict__ part_dg,
    float* __restrict__ part_db, int64_t rows_per_shard, int blocks_per_shard, int H) {
  __shared__ float sh[64];
  const int shard = blockIdx.x / blocks_per_shard;
  const int b = blockIdx.x - shard * blocks_per_shard;
  float gm[kLnVpt][8], adg[kLnVpt][8], adb[kLnVpt][8];
  bool ok[kLnVpt];
#pragma unroll
  for (int k = 0; k < kLnVpt; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    ok[k] = c < H;
    uint4 u = make_uint4(0, 0, 0, 0);
    if (ok[k]) u = ld_global_nc_v4(gamma + c);
    bf16x8_to_f32(u, gm[k]);
#pragma unroll
    for (int e = 0; e < 8; ++e) adg[k][e] = adb[k][e] = 0.f;
  }
  const int64_t rbeg = shard * rows_per_shard;
  for (int64_t lr = b; lr < rows_per_shard; lr += blocks_per_shard) {
    const int64_t row = rbeg + lr;
    const float mu = mean[row], rs = rstd[row];
    float xh[kLnVpt][8], g[kLnVpt][8], dy[kLnVpt][8];
    float s[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kLnVpt; ++k) {
      const int c = (threadIdx.x + k * blockDim.x) * 8;
      uint4 ux = make_uint4(0, 0, 0, 0), d0 = ux, d1 = ux;
      if (ok[k]) {
        ux = ld_global_nc_v4(X + row * H + c);
        d0 = ld_global_nc_v4(dXn + row * H + c);
        d1 = ld_global_nc_v4(dXn + row * H + c + 4);
      }
      bf16x8_to_f32(ux, xh[k]);
      dy[k][0] = __uint_as_float(d0.x); dy[k][1] = __uint_as_float(d0.y);
      dy[k][2] = __uint_as_float(d0.z); dy[k][3] = __uint_as_float(d0.w);
      dy[k][4] = __uint_as_float(d1.x); dy[k][5] = __uint_as_float(d1.y);
      dy[k][6] = __uint_as_float(d1.z); dy[k][7] = __uint_as_float(d1.w);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        xh[k][e] = ok[k] ? (xh[k][e] - mu) * rs : 0.f;
        g[k][e] = dy[k][e] * gm[k][e];
        s[0] += g[k][e];
        s[1] += g[k][e] * xh[k][e];
      }
    }
    block_sum<2>(s, sh);
    const float mg = s[0] / static_cast<float>(H);
    const float mgx = s[1] / static_cast<float>(H);
#pragma unroll
    for (int k = 0; k < kLnVpt; ++k) {
      if (!ok[k]) continue;
      const int c = (threadIdx.x + k * blockDim.x) * 8;
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        o[e] = rs * (g[k][e] - mg - xh[k][e] * mgx);
        adg[k][e] += dy[k][e] * xh[k][e];
        adb[k][e] += dy[k][e];
      }
      float* d = dX + row * H + c;
      st_global_v4(d, make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]),
                                 __float_as_uint(o[2]), __float_as_uint(o[3])));
      st_global_v4(d + 4, make_uint4(__float_as_uint(o[4]), __float_as_uint(o[5]),
                                     __float_as_uint(o[6]), __float_as_uint(o[7])));
    }
  }
#pragma unroll
  for (int k = 0; k < kLnVpt; ++k) {
    if (!ok[k]) continue;
    const int c = (threadIdx.x + k * blockDim.x) * 8;
    float* pg = part_dg + static_cast<int64_t>(blockIdx.x) * H + c;
    float* pb = part_db + static_cast<int64_t>(blockIdx.x) * H + c;
    st_global_v4(pg, make_uint4(__float_as_uint(adg[k][0]), __float_as_uint(adg[k][1]),
                                __float_as_uint(adg[k][2]), __float_as_uint(adg[k][3])));
    st_global_v4(pg + 4, make_uint4(__float_as_uint(adg[k][4]), __float_as_uint(adg[k][5]),
                                    __float_as_uint(adg[k][6]), __float_as_uint(adg[k][7])));
    st_global_v4(pb, make_uint4(__float_as_uint(adb[k][0]), __float_as_uint(adb[k][1]),
                                __float_as_uint(adb[k][2]), __float_as_uint(adb[k][3])));
    st_global_v4(pb + 4, make_uint4(__float_as_uint(adb[k][4]), __float_as_uint(adb[k][5]),
                                    __float_as_uint(adb[k][6]), __float_as_uint(adb[k][7])));
  }
}

static unsigned ln_threads(int64_t H, int vpt) {
  int64_t t = (H + 8 * vpt - 1) / (8 * vpt);
  t = (t + 31) / 32 * 32;
  return static_cast<unsigned>(t < 32 ? 32 : t);
}

cudaError_t launch_ln_fwd(const void* X, const void* gamma, const void* beta, void* Xn,
                          float* mean, float* rstd, int64_t T, int64_t H, float eps,
                          cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const auto* x = static_cast<const __nv_bfloat16*>(X);
  const auto* g = static_cast<const __nv_bfloat16*>(gamma);
  const auto* b = static_cast<const __nv_bfloat16*>(beta);
  auto* xn = static_cast<__nv_bfloat16*>(Xn);
  if (H <= 8192)
    ln_fwd_kernel<2><<<static_cast<unsigned>(T), ln_threads(H, 2), 0, s>>>(
        x, g, b, xn, mean, rstd, static_cast<int>(H), eps);
  else
    ln_fwd_kernel<4><<<static_cast<unsigned>(T), ln_threads(H, 4), 0, s>>>(
        x, g, b, xn, mean, rstd, static_cast<int>(H), eps);
  return cudaGetLastError();
}

cudaError_t launch_ln_bwd(const void* X, const void* gamma, const float* mean, const float* rstd,
                          const float* dXn, float* dX, float* part_dg, float* part_db,
                          int64_t T, int64_t H, int shards, int blocks_per_shard,
                          cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(shards * blocks_per_shard);
  const auto* x = static_cast<const __nv_bfloat16*>(X);
  const auto* g = static_cast<const __nv_bfloat16*>(gamma);
  if (H <= 8192)
    ln_bwd_kernel<2><<<grid, ln_threads(H, 2), 0, s>>>(x, g, mean, rstd, dXn, dX, part_dg,
                                                       part_db, T / shards, blocks_per_shard,
                                                       static_cast<int>(H));
  else
    ln_bwd_kernel<4><<<grid, ln_threads(H, 4), 0, s>>>(x, g, mean, rstd, dXn, dX, part_dg,
                                                       part_db, T / shards, blocks_per_shard,
                                                       static_cast<int>(H));
  return cudaGetLastError();
}

}  // namespace mlpb
