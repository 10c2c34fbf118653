// Sequence-parallel LayerNorm forward and backward.
//
// Both kernels stream whole rows into a ring of shared-memory buffers with TMA bulk
// copies (cp.async.bulk), so the next rows' loads stay in flight while the CTA reduces
// and writes the current one.  Thread i of a CTA owns the 16-byte vectors i, i+NT, ...
// of the row (kVpt vectors), so every global store is coalesced.  256-thread CTAs, two
// or more per SM, so that several rows' reduction chains overlap on every SM.
//
// Forward: persistent grid, CTA c handles rows c, c + grid, ...; per row two block
// reductions (the sum, then the squared deviations from the mean) give the mean and the
// biased variance of the register-resident row; Xn = (x - mu) rstd gamma + beta in bf16.
// Sequence shard s owns rows [s T/t, (s+1) T/t); rows are independent, so the forward
// needs no shard structure and the emulated all-gather is the row layout of Xn itself.
//
// Backward: a grid of t x B CTAs; CTA (s, b) walks rows b, b+B, ... of shard s, computes
// dx = rstd (g - mean(g) - xhat mean(g xhat)) with g = dy gamma, and accumulates its own
// dgamma/dbeta partials in registers.  The partials [t*B][H] are summed afterwards in
// shard order (the all-reduce of per-shard partials), deterministically.
//
// Every mbarrier wait is bounded; a CTA that gives up records the device error word,
// waits for the copies it issued and exits.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mlpb {

constexpr int kLnFwdThreads = 256;
constexpr int kLnBwdThreads = 256;

template <int NT, int NV>
__device__ __forceinline__ void block_sum(float (&v)[NV], float* sh /* [NT/32 * NV] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) s += sh[w * NV + k];
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

// Dynamic shared memory of the LN kernels (rows, then the ring's mbarriers).
extern __shared__ __align__(128) uint8_t ln_smem[];

// 16-byte load from the ring at byte offset `off` of the dynamic shared memory.  A plain
// load, so batches of them can be issued together; the mbarrier wait before them is an
// asm volatile with a memory clobber, which they cannot be moved above.
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t off) {
  return *reinterpret_cast<const uint4*>(ln_smem + off);
}

__device__ __forceinline__ void st_f32x8(float* p, const float* o) {
  st_global_v4(p, make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                             __float_as_uint(o[3])));
  st_global_v4(p + 4, make_uint4(__float_as_uint(o[4]), __float_as_uint(o[5]),
                                 __float_as_uint(o[6]), __float_as_uint(o[7])));
}

// ------------------------------------------------------------------ forward
// Row statistics by the textbook two-pass method over the register-resident row: one
// block reduction of the sum gives the mean, a second of the squared deviations from
// that mean gives the biased variance.  Unlike a single pass of (shifted) sums of
// squares, nothing large is subtracted, so a row with a common offset far larger than
// its spread, or with one far outlier, keeps its variance to fp32 rounding; per element
// it costs an add, a subtract and an FMA, and per row one more block reduction.
template <int kVpt>
__global__ void __launch_bounds__(kLnFwdThreads) ln_fwd_kernel(
    const __nv_bfloat16* __restrict__ X, const __nv_bfloat16* __restrict__ gamma,
    const __nv_bfloat16* __restrict__ beta, __nv_bfloat16* __restrict__ Xn,
    float* __restrict__ mean, float* __restrict__ rstd, int64_t T, int H, float eps, int nbuf,
    uint32_t* err, uint64_t wait_ns) {
  constexpr int NT = kLnFwdThreads;
  __shared__ float sh[NT / 32];
  __shared__ uint32_t abort_flag;
  const uint32_t row_bytes = static_cast<uint32_t>(H) * 2u;
  const uint32_t buf0 = smem_u32(ln_smem);
  const uint32_t bar0 = buf0 + nbuf * row_bytes;
  const int64_t n_mine = (T - blockIdx.x + gridDim.x - 1) / gridDim.x;
  const WaitCtx wc{&abort_flag, err, wait_ns};
  const float hf = static_cast<float>(H);

  if (threadIdx.x == 0) {
    abort_flag = 0u;
    for (int b = 0; b < nbuf; ++b) mbar_init(bar0 + 8 * b, 1);
    mbar_fence_init();
    for (int b = 0; b < nbuf && b < n_mine; ++b) {
      const int64_t row = blockIdx.x + static_cast<int64_t>(b) * gridDim.x;
      mbar_arrive_expect_tx(bar0 + 8 * b, row_bytes);
      bulk_load(buf0 + b * row_bytes, X + row * H, row_bytes, bar0 + 8 * b);
    }
  }
  float gm[kVpt][8], bt[kVpt][8];
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int c = (threadIdx.x + k * NT) * 8;
    uint4 g = make_uint4(0, 0, 0, 0), b = g;
    if (c < H) {
      g = ld_global_nc_v4(gamma + c);
      b = ld_global_nc_v4(beta + c);
    }
    bf16x8_to_f32(g, gm[k]);
    bf16x8_to_f32(b, bt[k]);
  }
  __syncthreads();

  int64_t issued = nbuf < n_mine ? nbuf : n_mine;
  for (int64_t i = 0; i < n_mine; ++i) {
    const int b = static_cast<int>(i % nbuf);
    const uint32_t par = static_cast<uint32_t>((i / nbuf) & 1);
    int ok = wait_bounded(bar0 + 8 * b, par, wc, kSiteLnFull) ? 1 : 0;
    if (!__syncthreads_and(ok)) break;
    const int64_t row = blockIdx.x + i * gridDim.x;
    float v[kVpt][8];
    float sum[1] = {0.f};
#pragma unroll
    for (int k = 0; k < kVpt; ++k) {
      const int vi = threadIdx.x + k * NT;
      const bool in = vi * 8 < H;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (in) u = ld_shared_v4(b * row_bytes + vi * 16);
      bf16x8_to_f32(u, v[k]);
#pragma unroll
      for (int e = 0; e < 8; ++e) sum[0] += v[k][e];  // zero beyond the row
    }
    block_sum<NT, 1>(sum, sh);  // every thread has read buffer b once this returns
    if (threadIdx.x == 0 && issued < n_mine) {
      const int64_t nrow = blockIdx.x + issued * gridDim.x;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar0 + 8 * b, row_bytes);
      bulk_load(buf0 + b * row_bytes, X + nrow * H, row_bytes, bar0 + 8 * b);
    }
    ++issued;
    const float mu = sum[0] / hf;
    float ssd[1] = {0.f};  // second pass: squared deviations from the row mean
#pragma unroll
    for (int k = 0; k < kVpt; ++k) {
      if ((threadIdx.x + k * NT) * 8 >= H) continue;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = v[k][e] - mu;
        ssd[0] = fmaf(d, d, ssd[0]);
      }
    }
    block_sum<NT, 1>(ssd, sh);
    const float var = ssd[0] / hf;
    const float r = rsqrtf(var + eps);
#pragma unroll
    for (int k = 0; k < kVpt; ++k) {
      const int c = (threadIdx.x + k * NT) * 8;
      if (c >= H) continue;
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = fmaf((v[k][e] - mu) * r, gm[k][e], bt[k][e]);
      st_global_v4(Xn + row * H + c, make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                                pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7])));
    }
    if (threadIdx.x == 0) {
      mean[row] = mu;
      rstd[row] = r;
    }
  }
  // Copies still in flight (only after an abort) must land before the CTA exits.
  if (threadIdx.x == 0 && abort_flag) {
    const int64_t first = issued - nbuf > 0 ? issued - nbuf : 0;
    for (int64_t i = first; i < issued && i < n_mine; ++i)
      wait_drain(bar0 + 8 * static_cast<int>(i % nbuf), static_cast<uint32_t>((i / nbuf) & 1), wc);
  }
}

// ------------------------------------------------------------------ backward
// With kRes, dX also receives the residual branch's gradient dres (bf16 [T][H]):
// dX = dres + LN'(dXn).  With kBf16, dXn is read and dX written as bf16 (the block's
// bf16-output mode; the arithmetic is the same fp32, with one rounding of dX at the end).
// dXn and dX may be the same buffer: each row of dXn is copied whole into shared memory
// (and waited for) before any element of that row of dX is written, and no other CTA
// touches the row.
template <int kVpt, bool kRes, bool kBf16>
__global__ void __launch_bounds__(kLnBwdThreads, 2) ln_bwd_kernel(
    const __nv_bfloat16* __restrict__ X, const __nv_bfloat16* __restrict__ gamma,
    const float* __restrict__ mean, const float* __restrict__ rstd, const void* dXn,
    const __nv_bfloat16* __restrict__ dres, void* dX, float* __restrict__ part_dg,
    float* __restrict__ part_db, int64_t rows_per_shard, int blocks_per_shard, int H, int nbuf,
    uint32_t* err, uint64_t wait_ns) {
  constexpr int NT = kLnBwdThreads;
  constexpr uint32_t kGradBytes = kBf16 ? 2u : 4u;  // bytes of a dXn / dX element
  __shared__ float sh[2 * NT / 32];
  __shared__ uint32_t abort_flag;
  const uint32_t xbytes = static_cast<uint32_t>(H) * 2u;
  const uint32_t row_bytes = static_cast<uint32_t>(H) * (2u + kGradBytes);  // X, then dXn
  const uint32_t buf0 = smem_u32(ln_smem);
  const uint32_t bar0 = buf0 + nbuf * row_bytes;
  const int shard = blockIdx.x / blocks_per_shard;
  const int bidx = blockIdx.x - shard * blocks_per_shard;
  const int64_t rbeg = shard * rows_per_shard;
  const int64_t n_mine =
      bidx < rows_per_shard ? (rows_per_shard - bidx + blocks_per_shard - 1) / blocks_per_shard : 0;
  const WaitCtx wc{&abort_flag, err, wait_ns};

  auto issue = [&](int b, int64_t i) {
    const int64_t row = rbeg + bidx + i * blocks_per_shard;
    mbar_arrive_expect_tx(bar0 + 8 * b, row_bytes);
    bulk_load(buf0 + b * row_bytes, X + row * H, xbytes, bar0 + 8 * b);
    bulk_load(buf0 + b * row_bytes + xbytes,
              static_cast<const uint8_t*>(dXn) + static_cast<size_t>(row) * H * kGradBytes,
              kGradBytes * H, bar0 + 8 * b);
    // the residual gradient's row is read with plain loads in pass 2; start it towards L2
    if constexpr (kRes) bulk_prefetch_l2(dres + row * H, xbytes);
  };
  if (threadIdx.x == 0) {
    abort_flag = 0u;
    for (int b = 0; b < nbuf; ++b) mbar_init(bar0 + 8 * b, 1);
    mbar_fence_init();
    for (int b = 0; b < nbuf && b < n_mine; ++b) issue(b, b);
  }
  __syncthreads();

  uint4 gpk[kVpt];  // gamma, kept packed (bf16) to leave registers for the partials
  float adg[kVpt][8], adb[kVpt][8];
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int c = (threadIdx.x + k * NT) * 8;
    gpk[k] = make_uint4(0, 0, 0, 0);
    if (c < H) gpk[k] = ld_global_nc_v4(gamma + c);
#pragma unroll
    for (int e = 0; e < 8; ++e) adg[k][e] = adb[k][e] = 0.f;
  }

  // x and dy of vector vi of the row in buffer (xb, db)
  auto load_vec = [&](uint32_t xb, uint32_t db, int vi, float* x, float* dy) {
    bf16x8_to_f32(ld_shared_v4(xb + vi * 16), x);
    if constexpr (kBf16) {
      bf16x8_to_f32(ld_shared_v4(db + vi * 16), dy);
    } else {
      const uint4 d0 = ld_shared_v4(db + vi * 32);
      const uint4 d1 = ld_shared_v4(db + vi * 32 + 16);
      dy[0] = __uint_as_float(d0.x); dy[1] = __uint_as_float(d0.y);
      dy[2] = __uint_as_float(d0.z); dy[3] = __uint_as_float(d0.w);
      dy[4] = __uint_as_float(d1.x); dy[5] = __uint_as_float(d1.y);
      dy[6] = __uint_as_float(d1.z); dy[7] = __uint_as_float(d1.w);
    }
  };

  int64_t issued = nbuf < n_mine ? nbuf : n_mine;
  for (int64_t i = 0; i < n_mine; ++i) {
    const int b = static_cast<int>(i % nbuf);
    const uint32_t par = static_cast<uint32_t>((i / nbuf) & 1);
    int ok = wait_bounded(bar0 + 8 * b, par, wc, kSiteLnFull) ? 1 : 0;
    if (!__syncthreads_and(ok)) break;
    const int64_t row = rbeg + bidx + i * blocks_per_shard;
    const float mu = mean[row], rs = rstd[row];
    const uint32_t xb = b * row_bytes;  // offsets into ln_smem
    const uint32_t db = xb + xbytes;
    // pass 1: sum g and sum g*xhat
    float s[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kVpt; ++k) {
      const int vi = threadIdx.x + k * NT;
      if (vi * 8 >= H) continue;
      float x[8], dy[8], gm[8];
      load_vec(xb, db, vi, x, dy);
      bf16x8_to_f32(gpk[k], gm);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xh = (x[e] - mu) * rs;
        const float g = dy[e] * gm[e];
        s[0] += g;
        s[1] += g * xh;
      }
    }
    block_sum<NT, 2>(s, sh);
    const float mg = s[0] / static_cast<float>(H);
    const float mgx = s[1] / static_cast<float>(H);
    // pass 2: dx, and this CTA's dgamma / dbeta partials.  The residual gradient's row
    // is fetched first, all of this thread's vectors at once, ahead of the stores.
    uint4 rpk[kRes ? kVpt : 1];
    if constexpr (kRes) {
#pragma unroll
      for (int k = 0; k < kVpt; ++k) {
        const int vi = threadIdx.x + k * NT;
        rpk[k] = vi * 8 < H ? ld_global_nc_v4(dres + row * H + vi * 8) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int k = 0; k < kVpt; ++k) {
      const int vi = threadIdx.x + k * NT;
      if (vi * 8 >= H) continue;
      float x[8], dy[8], gm[8], o[8];
      load_vec(xb, db, vi, x, dy);
      bf16x8_to_f32(gpk[k], gm);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xh = (x[e] - mu) * rs;
        o[e] = rs * (dy[e] * gm[e] - mg - xh * mgx);
        adg[k][e] += dy[e] * xh;
        adb[k][e] += dy[e];
      }
      if constexpr (kRes) {
        float r[8];
        bf16x8_to_f32(rpk[k], r);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = __fadd_rn(o[e], r[e]);  // a plain add, never an FMA
      }
      if constexpr (kBf16)
        st_global_v4(static_cast<__nv_bfloat16*>(dX) + row * H + vi * 8,
                     make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7])));
      else
        st_f32x8(static_cast<float*>(dX) + row * H + vi * 8, o);
    }
    __syncthreads();  // every thread has read buffer b
    if (threadIdx.x == 0 && issued < n_mine) {
      fence_proxy_async_smem();
      issue(b, issued);
    }
    ++issued;
  }
  if (threadIdx.x == 0 && abort_flag) {
    const int64_t first = issued - nbuf > 0 ? issued - nbuf : 0;
    for (int64_t i = first; i < issued && i < n_mine; ++i)
      wait_drain(bar0 + 8 * static_cast<int>(i % nbuf), static_cast<uint32_t>((i / nbuf) & 1), wc);
  }
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int c = (threadIdx.x + k * NT) * 8;
    if (c >= H) continue;
    st_f32x8(part_dg + static_cast<int64_t>(blockIdx.x) * H + c, adg[k]);
    st_f32x8(part_db + static_cast<int64_t>(blockIdx.x) * H + c, adb[k]);
  }
}

// ------------------------------------------------------------------ launchers
static int ln_vpt(int64_t H, int threads) {
  const int64_t v = (H / 8 + threads - 1) / threads;
  return v <= 1 ? 1 : v <= 2 ? 2 : v <= 4 ? 4 : 8;  // H <= 16384
}

template <class K>
static cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

cudaError_t launch_ln_fwd(const void* X, const void* gamma, const void* beta, void* Xn,
                          float* mean, float* rstd, int64_t T, int64_t H, float eps, int num_sms,
                          uint32_t* err, uint64_t wait_ns, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const size_t row = static_cast<size_t>(H) * 2;
  const int nbuf = static_cast<int>(std::min<size_t>(3, std::max<size_t>(2, (48u << 10) / row)));
  const size_t smem = nbuf * row + 8 * nbuf;
  const auto* x = static_cast<const __nv_bfloat16*>(X);
  const auto* g = static_cast<const __nv_bfloat16*>(gamma);
  const auto* b = static_cast<const __nv_bfloat16*>(beta);
  auto* xn = static_cast<__nv_bfloat16*>(Xn);
  const int Hi = static_cast<int>(H);
  cudaError_t e = cudaSuccess;
  switch (ln_vpt(H, kLnFwdThreads)) {
#define MLPB_LN_FWD(V)                                                                        \
  case V: {                                                                                   \
    e = set_smem(ln_fwd_kernel<V>, smem);                                                     \
    int per_sm = 1;                                                                           \
    if (e == cudaSuccess)                                                                     \
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ln_fwd_kernel<V>,            \
                                                        kLnFwdThreads, smem);                 \
    const unsigned grid =                                                                     \
        static_cast<unsigned>(std::min<int64_t>(T, std::max(1, per_sm) * num_sms));           \
    if (e == cudaSuccess)                                                                     \
      ln_fwd_kernel<V><<<grid, kLnFwdThreads, smem, s>>>(x, g, b, xn, mean, rstd, T, Hi, eps, \
                                                         nbuf, err, wait_ns);                 \
    break;                                                                                    \
  }
    MLPB_LN_FWD(1)
    MLPB_LN_FWD(2)
    MLPB_LN_FWD(4)
    MLPB_LN_FWD(8)
#undef MLPB_LN_FWD
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_ln_bwd(const void* X, const void* gamma, const float* mean, const float* rstd,
                          const void* dXn, const void* dres, void* dX, bool bf16_grads,
                          float* part_dg, float* part_db, int64_t T, int64_t H, int shards,
                          int blocks_per_shard, uint32_t* err, uint64_t wait_ns, cudaStream_t s) {
  const size_t row = static_cast<size_t>(H) * (bf16_grads ? 4 : 6);
  const int nbuf = 2;  // two 256-thread CTAs per SM, each with a two-row ring
  const size_t smem = nbuf * row + 8 * nbuf;
  const unsigned grid = static_cast<unsigned>(shards * blocks_per_shard);
  const auto* x = static_cast<const __nv_bfloat16*>(X);
  const auto* g = static_cast<const __nv_bfloat16*>(gamma);
  const auto* r = static_cast<const __nv_bfloat16*>(dres);
  const int Hi = static_cast<int>(H);
  const int64_t rps = T / shards;
  cudaError_t e = cudaSuccess;
  switch (ln_vpt(H, kLnBwdThreads)) {
#define MLPB_LN_BWD_RES(V, R, B)                                                             \
  e = set_smem(ln_bwd_kernel<V, R, B>, smem);                                                \
  if (e == cudaSuccess)                                                                      \
    ln_bwd_kernel<V, R, B><<<grid, kLnBwdThreads, smem, s>>>(x, g, mean, rstd, dXn, r, dX,   \
                                                             part_dg, part_db, rps,          \
                                                             blocks_per_shard, Hi, nbuf,     \
                                                             err, wait_ns);
#define MLPB_LN_BWD(V)                 \
  case V:                              \
    if (r != nullptr && bf16_grads) {  \
      MLPB_LN_BWD_RES(V, true, true)   \
    } else if (r != nullptr) {         \
      MLPB_LN_BWD_RES(V, true, false)  \
    } else if (bf16_grads) {           \
      MLPB_LN_BWD_RES(V, false, true)  \
    } else {                           \
      MLPB_LN_BWD_RES(V, false, false) \
    }                                  \
    break;
    MLPB_LN_BWD(1)
    MLPB_LN_BWD(2)
    MLPB_LN_BWD(4)
    MLPB_LN_BWD(8)
#undef MLPB_LN_BWD
#undef MLPB_LN_BWD_RES
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mlpb
