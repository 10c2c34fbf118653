// E4M3 helpers shared by the quantization kernels and the FP8 GEMM epilogues.
//
// Per-tensor current scaling with a power-of-two scale: for a tensor whose largest
// magnitude is amax, k is the largest integer with amax * 2^k <= 448 (E4M3's largest
// finite value), 0 for an all-zero tensor; its codes are q = e4m3(x * 2^k) rounded to
// nearest, ties to even, and a GEMM of two such operands rescales its fp32 sums by
// 2^-(k_a + k_b).  amax is carried as the bit pattern of a non-negative fp32, so that
// unsigned atomicMax orders it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace mlpb {

// k for the bf16 value of amax (the largest magnitude of the stored bf16 tensor: rounding
// is monotone, so this is the bf16 rounding of an fp32 maximum taken before storing).
__device__ __forceinline__ int e4m3_scale_exp(uint32_t amax_bits) {
  const float a = __bfloat162float(__float2bfloat16_rn(__uint_as_float(amax_bits)));
  if (!(a > 0.0f)) return 0;
  int e;
  const float m = frexpf(a, &e);  // a = m 2^e, 0.5 <= m < 1;  448 = 0.875 2^9
  return m <= 0.875f ? 9 - e : 8 - e;
}

// Two fp32 values, already scaled, to two E4M3 codes (lo in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Eight bf16 values (one 16-byte word) scaled by 2^k, to eight E4M3 codes.
__device__ __forceinline__ uint2 e4m3x8_from_bf16x8(uint4 u, int k) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    c[i] = e4m3x2(ldexpf(f.x, k), ldexpf(f.y, k));
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

}  // namespace mlpb
