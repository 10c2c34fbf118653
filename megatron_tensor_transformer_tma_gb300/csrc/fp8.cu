// E4M3 quantization: the absolute maximum of a bf16 tensor, and its cast to E4M3 codes in
// the tensor's own layout and/or transposed (the FP8 GEMMs read every operand K-major, so
// an operand used in both orientations gets both copies).
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/mlpb.h"
#include "common.cuh"
#include "fp8.cuh"
#include "kernels.h"

namespace mlpb {

constexpr int kAmaxThreads = 256;
constexpr int kAmaxBatch = 4;   // 16-byte loads in flight per thread
constexpr int kCastRows = 64;   // CTA tile rows (R)
constexpr int kCastCols = 256;  // CTA tile columns (C)
constexpr int kCastThreads = 256;

// *amax = max(*amax, max |in|) as fp32 bits.  |x| of a bf16 is its bits without the sign,
// and for non-negative values the bit patterns order like the values, so the reduction
// runs on 16-bit lanes (__vmaxu2) and the result is the bf16 amax widened to fp32.
__global__ void __launch_bounds__(kAmaxThreads) amax_bf16_kernel(const uint4* __restrict__ in,
                                                                 int64_t n16,
                                                                 uint32_t* __restrict__ amax) {
  uint32_t m = 0u;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kAmaxThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kAmaxThreads + threadIdx.x;
  for (; i + (kAmaxBatch - 1) * stride < n16; i += kAmaxBatch * stride) {
    uint4 u[kAmaxBatch];
#pragma unroll
    for (int b = 0; b < kAmaxBatch; ++b) u[b] = __ldg(in + i + b * stride);
#pragma unroll
    for (int b = 0; b < kAmaxBatch; ++b) {
      m = __vmaxu2(m, u[b].x & 0x7fff7fffu);
      m = __vmaxu2(m, u[b].y & 0x7fff7fffu);
      m = __vmaxu2(m, u[b].z & 0x7fff7fffu);
      m = __vmaxu2(m, u[b].w & 0x7fff7fffu);
    }
  }
  for (; i < n16; i += stride) {
    const uint4 u = __ldg(in + i);
    m = __vmaxu2(m, u.x & 0x7fff7fffu);
    m = __vmaxu2(m, u.y & 0x7fff7fffu);
    m = __vmaxu2(m, u.z & 0x7fff7fffu);
    m = __vmaxu2(m, u.w & 0x7fff7fffu);
  }
  uint32_t v = max(m & 0xffffu, m >> 16) << 16;  // the bf16 bits widened to fp32 bits
  v = __reduce_max_sync(0xffffffffu, v);
  __shared__ uint32_t red[kAmaxThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    v = threadIdx.x < kAmaxThreads / 32 ? red[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xffffffffu, v);
    if (threadIdx.x == 0) atomicMax(amax, v);
  }
}

// Transpose of an 8 x 8 byte block held as eight 8-byte rows: out[j] = column j.
__device__ __forceinline__ void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3,
                                             uint32_t& c0, uint32_t& c1, uint32_t& c2,
                                             uint32_t& c3) {
  const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r0, r1, 0x7362);
  const uint32_t t2 = __byte_perm(r2, r3, 0x5140), t3 = __byte_perm(r2, r3, 0x7362);
  c0 = __byte_perm(t0, t2, 0x5410);
  c1 = __byte_perm(t0, t2, 0x7632);
  c2 = __byte_perm(t1, t3, 0x5410);
  c3 = __byte_perm(t1, t3, 0x7632);
}

__device__ __forceinline__ void transpose8x8(const uint2 (&row)[8], uint2 (&col)[8]) {
  uint32_t a[4], b[4], c[4], d[4];
  transpose4x4(row[0].x, row[1].x, row[2].x, row[3].x, a[0], a[1], a[2], a[3]);  // cols 0-3, rows 0-3
  transpose4x4(row[4].x, row[5].x, row[6].x, row[7].x, b[0], b[1], b[2], b[3]);  // cols 0-3, rows 4-7
  transpose4x4(row[0].y, row[1].y, row[2].y, row[3].y, c[0], c[1], c[2], c[3]);  // cols 4-7, rows 0-3
  transpose4x4(row[4].y, row[5].y, row[6].y, row[7].y, d[0], d[1], d[2], d[3]);  // cols 4-7, rows 4-7
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    col[j] = make_uint2(a[j], b[j]);
    col[4 + j] = make_uint2(c[j], d[j]);
  }
}

// in bf16 [B][R][C] -> q e4m3 [B][R][C] (if kQ) and qt e4m3 [B][C][R] (if kQT), scale 2^k
// from *amax.  Each thread converts an 8 x 8 block (eight 16-byte row loads), transposes
// the codes in registers, and writes eight 8-byte rows of q and of qt.  With qt a warp is
// 8 row blocks x 4 column blocks (64 x 32 elements), so each load covers 64 contiguous
// bytes of a row, each q store 32 bytes of a row and each qt store 64 bytes of a qt row;
// a CTA stacks its 8 warps along C (64 x 256).  Requires R % 8 == 0 and C % 8 == 0.
template <bool kQ, bool kQT>
__global__ void __launch_bounds__(kCastThreads) cast_e4m3_kernel(
    const __nv_bfloat16* __restrict__ in, uint8_t* __restrict__ q, uint8_t* __restrict__ qt,
    const uint32_t* __restrict__ amax, int32_t* __restrict__ k_out, int64_t R, int64_t C) {
  const int k = e4m3_scale_exp(*amax);
  if (k_out != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
      threadIdx.x == 0)
    *k_out = k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // with qt: a warp is 8 row blocks x 4 column blocks; without: 1 row block x 32 column
  // blocks (512 contiguous bytes a load, 256 a store).  Either way a CTA covers 64 x 256.
  const int rb = kQT ? (lane & 7) : warp;
  const int cb = kQT ? warp * 4 + (lane >> 3) : lane;
  const int64_t r = static_cast<int64_t>(blockIdx.y) * kCastRows + rb * 8;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * kCastCols + cb * 8;
  if (r >= R || c >= C) return;
  const int64_t plane = R * C;
  const __nv_bfloat16* src = in + blockIdx.z * plane + r * C + c;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(src + i * C));
  uint2 rows[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) rows[i] = e4m3x8_from_bf16x8(v[i], k);
  if constexpr (kQ) {
    uint8_t* dst = q + blockIdx.z * plane + r * C + c;
#pragma unroll
    for (int i = 0; i < 8; ++i) *reinterpret_cast<uint2*>(dst + i * C) = rows[i];
  }
  if constexpr (kQT) {
    uint2 cols[8];
    transpose8x8(rows, cols);
    uint8_t* dst = qt + blockIdx.z * plane + c * R + r;
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint2*>(dst + j * R) = cols[j];
  }
}

cudaError_t launch_amax_bf16(const void* in, int64_t n, uint32_t* amax, int num_sms,
                             cudaStream_t s) {
  const int64_t n16 = n / 8;
  if (n16 == 0) return cudaSuccess;
  const int64_t want = (n16 + kAmaxThreads * kAmaxBatch - 1) / (kAmaxThreads * kAmaxBatch);
  const unsigned grid = static_cast<unsigned>(std::max<int64_t>(
      1, std::min<int64_t>(want, static_cast<int64_t>(num_sms) * 8)));
  amax_bf16_kernel<<<grid, kAmaxThreads, 0, s>>>(static_cast<const uint4*>(in), n16, amax);
  return cudaGetLastError();
}

cudaError_t launch_cast_e4m3(const void* in, int batches, int64_t R, int64_t C, void* q,
                             void* qt, const uint32_t* amax, int32_t* k_out, cudaStream_t s) {
  if (R == 0 || C == 0 || batches == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((C + kCastCols - 1) / kCastCols),
                  static_cast<unsigned>((R + kCastRows - 1) / kCastRows),
                  static_cast<unsigned>(batches));
  const auto* x = static_cast<const __nv_bfloat16*>(in);
  auto* q8 = static_cast<uint8_t*>(q);
  auto* qt8 = static_cast<uint8_t*>(qt);
  if (q != nullptr && qt != nullptr)
    cast_e4m3_kernel<true, true><<<grid, kCastThreads, 0, s>>>(x, q8, qt8, amax, k_out, R, C);
  else if (q != nullptr)
    cast_e4m3_kernel<true, false><<<grid, kCastThreads, 0, s>>>(x, q8, qt8, amax, k_out, R, C);
  else
    cast_e4m3_kernel<false, true><<<grid, kCastThreads, 0, s>>>(x, q8, qt8, amax, k_out, R, C);
  return cudaGetLastError();
}

}  // namespace mlpb

extern "C" mlpb_status mlpb_quantize_e4m3(const void* in, int64_t batches, int64_t rows,
                                          int64_t cols, void* q, void* qt, uint32_t* amax,
                                          int32_t* scale_exp, mlpb_stream_t stream) {
  if (batches < 0 || rows < 0 || cols < 0) return MLPB_EINVAL;
  if (amax == nullptr || (q == nullptr && qt == nullptr)) return MLPB_EINVAL;
  if (rows % 16 != 0 || cols % 16 != 0) return MLPB_EUNSUPPORTED;  // (the kernels need 8)
  const int64_t n = batches * rows * cols;
  if (n > 0 && in == nullptr) return MLPB_EINVAL;
  for (const void* p : {in, static_cast<const void*>(q), static_cast<const void*>(qt)})
    if (p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) != 0) return MLPB_EINVAL;
  if ((reinterpret_cast<uintptr_t>(amax) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(scale_exp) & 3u) != 0)
    return MLPB_EINVAL;
  // grid: z = batches, y = 64-row tiles (both at most 65535)
  if (batches > 65535 || rows > int64_t(65535) * 64 || cols > (int64_t(1) << 31))
    return MLPB_EUNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLPB_ECUDA;
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = mlpb::launch_amax_bf16(in, n, amax, sms, s);
  if (e == cudaSuccess && n == 0 && scale_exp != nullptr)
    e = cudaMemsetAsync(scale_exp, 0, sizeof(int32_t), s);
  if (e == cudaSuccess)
    e = mlpb::launch_cast_e4m3(in, static_cast<int>(batches), rows, cols, q, qt, amax, scale_exp,
                               s);
  return e == cudaSuccess ? MLPB_OK : MLPB_ECUDA;
}
