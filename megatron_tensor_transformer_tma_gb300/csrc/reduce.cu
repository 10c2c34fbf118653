// Bias-gradient column reductions (db2 = sum_t dY, db1 = sum_t dZ) and helpers.
//
// Pass 1: a CTA of 256 threads owns 512 columns x one split of rows; each thread keeps
// 8 fp32 column sums (one 16-byte bf16 vector per row) over every 4th row of the split,
// and the 4 row lanes are combined through shared memory into part[split][col].
// Pass 2 sums the splits in a fixed order, so results are bitwise reproducible.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mlpb {

constexpr int kColsPerCta = 512;
constexpr int kRowLanes = 4;
constexpr int kBatch = 8;  // 16-byte loads in flight per thread

// acc[0..8) += column sums of 8 bf16 columns at p over rows r, r+4, ... < r1.  Loads are
// issued in explicit batches of kBatch before any is consumed.
__device__ __forceinline__ void add_bf16x8(const uint4& u, float (&acc)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = unpack_bf16x2(w[e]);
    acc[2 * e] += f.x;
    acc[2 * e + 1] += f.y;
  }
}

__device__ __forceinline__ void colsum_rows(const __nv_bfloat16* p, int64_t C, int64_t r,
                                            int64_t r1, float (&acc)[8]) {
  // full batches: kBatch unconditional loads, then their sums
  for (; r + (kBatch - 1) * kRowLanes < r1; r += kBatch * kRowLanes) {
    uint4 u[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) u[j] = ld_global_nc_v4(p + (r + j * kRowLanes) * C);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) add_bf16x8(u[j], acc);
  }
  for (; r < r1; r += kRowLanes) add_bf16x8(ld_global_nc_v4(p + r * C), acc);
}

__global__ void __launch_bounds__(256) colsum_bf16_kernel(const __nv_bfloat16* __restrict__ in,
                                                          int64_t R, int64_t C,
                                                          int64_t rows_per_split,
                                                          float* __restrict__ part) {
  __shared__ float red[kRowLanes - 1][64][9];
  const int cv = threadIdx.x & 63;
  const int rl = threadIdx.x >> 6;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * kColsPerCta + cv * 8;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_split;
  const int64_t r1 = min(R, r0 + rows_per_split);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if (col < C) {
    colsum_rows(in + col, C, r0 + rl, r1, acc);
  }
  if (rl > 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) red[rl - 1][cv][e] = acc[e];
  }
  __syncthreads();
  if (rl == 0 && col < C) {
#pragma unroll
    for (int l = 0; l < kRowLanes - 1; ++l)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += red[l][cv][e];
    float* o = part + static_cast<int64_t>(blockIdx.y) * C + col;
    st_global_v4(o, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                               __float_as_uint(acc[2]), __float_as_uint(acc[3])));
    st_global_v4(o + 4, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                   __float_as_uint(acc[6]), __float_as_uint(acc[7])));
  }
}

// A 16-byte streaming load (read once: no L1 allocation).  An asm volatile, so that a
// batch of them is issued in program order before the adds that consume it.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// out[c] = sum_k part[k][c] (or out[c] += ... with `accumulate`) for one or two partial
// arrays (blockIdx.y picks the array; each has its own part count and width).
// A CTA owns 32 columns: warp w sums parts w, w+8, ... of its lane's column, then the
// eight warp sums are added in warp order -- a fixed order, so results are reproducible.
__global__ void __launch_bounds__(256) sum_partials_kernel(const float* part_a, int np_a,
                                                           int64_t C_a, float* out_a,
                                                           const float* part_b, int np_b,
                                                           int64_t C_b, float* out_b,
                                                           int accumulate) {
  __shared__ float red[8][33];
  const bool second = blockIdx.y != 0;
  const float* part = second ? part_b : part_a;
  float* out = second ? out_b : out_a;
  const int nparts = second ? np_b : np_a;
  const int64_t C = second ? C_b : C_a;
  if (static_cast<int64_t>(blockIdx.x) * 32 >= C) return;  // the narrower array's spare CTAs
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  float s = 0.f;
  if (c < C) {
#pragma unroll 4
    for (int k = warp; k < nparts; k += 8) s += part[static_cast<int64_t>(k) * C + c];
  }
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && c < C) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[w][lane];
    out[c] = accumulate ? out[c] + t : t;
  }
}

__global__ void fill_zero_kernel(uint4* p, size_t n16, uint8_t* tail, size_t ntail) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0, 0, 0, 0);
  if (blockIdx.x == 0 && threadIdx.x < ntail) tail[threadIdx.x] = 0;
}

cudaError_t launch_colsum_bf16(const void* in, int64_t R, int64_t C, int splits,
                               int64_t rows_per_split, float* part, float* out, cudaStream_t s,
                               int accumulate) {
  const dim3 grid(static_cast<unsigned>((C + kColsPerCta - 1) / kColsPerCta),
                  static_cast<unsigned>(splits));
  colsum_bf16_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(in), R, C,
                                           rows_per_split, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_sum_partials(part, splits, C, out, s, accumulate);
}

cudaError_t launch_sum_partials(const float* part, int nparts, int64_t C, float* out,
                                cudaStream_t s, int accumulate) {
  const dim3 grid(static_cast<unsigned>((C + 31) / 32), 1);
  sum_partials_kernel<<<grid, 256, 0, s>>>(part, nparts, C, out, part, nparts, C, out,
                                           accumulate);
  return cudaGetLastError();
}

cudaError_t launch_sum_partials2(const float* part_a, const float* part_b, int nparts, int64_t C,
                                 float* out_a, float* out_b, cudaStream_t s, int accumulate) {
  return launch_sum_partials_pair(part_a, nparts, C, out_a, part_b, nparts, C, out_b, s,
                                  accumulate);
}

cudaError_t launch_sum_partials_pair(const float* part_a, int np_a, int64_t C_a, float* out_a,
                                     const float* part_b, int np_b, int64_t C_b, float* out_b,
                                     cudaStream_t s, int accumulate) {
  const int64_t C = C_a > C_b ? C_a : C_b;
  const dim3 grid(static_cast<unsigned>((C + 31) / 32), 2);
  sum_partials_kernel<<<grid, 256, 0, s>>>(part_a, np_a, C_a, out_a, part_b, np_b, C_b, out_b,
                                           accumulate);
  return cudaGetLastError();
}

// W2t[i][j][h] = W2[i][h][j]: each shard's [H][Fs] slice of W2 transposed into the rows
// i Fs + j of a K-major [F][H] copy, which the dgrad GEMM reads as its B operand (read
// column-wise from W2 itself, as an MN-major operand, the GEMM measured 7 % slower).  A CTA
// moves a 64 (h) x 128 (j) tile: eight lanes load each 128-byte run of a W2 row, and eight
// lanes store each 128-byte run of a W2t row, so both sides move whole lines.
// H % 64 == 0, Fs % 8 == 0.
__device__ __forceinline__ void transpose_w2_tile(const __nv_bfloat16* __restrict__ w2,
                                                  __nv_bfloat16* __restrict__ w2t, int H, int Fs,
                                                  int fx, int hy, int i, uint32_t (*tileT)[33]) {
  // tileT holds the tile transposed as 32-bit words, each the pair (h, h + 1) at one f:
  // row f of 32 words (+1 of padding) is the 128-byte run of row f of the copy.
  const int h0 = hy * 64, f0 = fx * 128;
  const int c8 = threadIdx.x & 7, p = threadIdx.x >> 3;  // f chunk of 8, h pair
  const __nv_bfloat16* src = w2 + (static_cast<size_t>(i) * H + h0 + 2 * p) * Fs + f0;
  uint4 u[2][2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {  // both f halves, rows 2p and 2p + 1: four loads in flight
    const int c = (c8 + 8 * q) * 8;
#pragma unroll
    for (int r = 0; r < 2; ++r)
      u[q][r] = f0 + c < Fs ? ld_global_nc_v4(src + static_cast<size_t>(r) * Fs + c)
                            : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint32_t lo[4] = {u[q][0].x, u[q][0].y, u[q][0].z, u[q][0].w};
    const uint32_t hi[4] = {u[q][1].x, u[q][1].y, u[q][1].z, u[q][1].w};
    const int f = (c8 + 8 * q) * 8;
#pragma unroll
    for (int e = 0; e < 4; ++e) {  // columns f + 2e and f + 2e + 1 of rows 2p, 2p + 1
      tileT[f + 2 * e][p] = (lo[e] & 0xffffu) | (hi[e] << 16);
      tileT[f + 2 * e + 1][p] = (lo[e] >> 16) | (hi[e] & 0xffff0000u);
    }
  }
  __syncthreads();
  // eight lanes write one 128-byte row of the copy: whole lines, no partial sectors
  const int k = threadIdx.x & 7;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int f = (threadIdx.x >> 3) + 32 * r;
    if (f0 + f >= Fs) break;
    const uint4 v = make_uint4(tileT[f][4 * k], tileT[f][4 * k + 1], tileT[f][4 * k + 2],
                               tileT[f][4 * k + 3]);
    st_global_v4(w2t + (static_cast<size_t>(i) * Fs + f0 + f) * H + h0 + 8 * k, v);
  }
}

constexpr int kTcBatch = 4;  // 16-byte loads in flight a thread in the column-sum blocks

// The start of the bf16 backward in one launch.  Blocks [0, n_tr) write W2's transposed
// copy, one 64 x 128 tile each (tiles in (f, h, shard) order).  With a bias, blocks
// [n_tr, n_tr + chunks * splits) take the first pass of db2 = sum_t dY: block (split,
// chunk) sums the 256 columns of `chunk` over its row range; warp w reads rows w, w + 8,
// ... (each warp load is 512 contiguous bytes of one row), kTcBatch loads in flight a
// thread, and the 8 warps' partial rows are added in warp order through shared memory
// into part[split][256 chunk ..] (a fixed order: reproducible).  Both halves are DRAM
// streams; the column sums fill the GPU beside the transpose instead of in a launch of
// their own, and the final sum over the splits joins db1's.  At most 40 registers a
// thread (6 CTAs an SM), for the transpose's loads in flight.
__global__ void __launch_bounds__(256, 6)
    transpose_w2_colsum_kernel(const __nv_bfloat16* __restrict__ w2,
                               __nv_bfloat16* __restrict__ w2t, int H, int Fs, int n_tr,
                               const __nv_bfloat16* __restrict__ dy, int64_t T, int64_t rps,
                               float* __restrict__ part) {
  __shared__ __align__(16) uint32_t smem[128 * 33];
  const int b = blockIdx.x;
  if (b < n_tr) {
    const int ntx = (Fs + 127) / 128, nty = H / 64;
    const int i = b / (ntx * nty);
    const int r = b - i * ntx * nty;
    const int hy = r / ntx;
    transpose_w2_tile(w2, w2t, H, Fs, r - hy * ntx, hy, i,
                      reinterpret_cast<uint32_t (*)[33]>(smem));
    return;
  }
  const int chunks = (H + 255) / 256;
  const int cb = b - n_tr;
  const int split = cb / chunks, chunk = cb - split * chunks;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t col = static_cast<int64_t>(chunk) * 256 + lane * 8;
  const int64_t r0 = static_cast<int64_t>(split) * rps;
  const int64_t r1 = min(T, r0 + rps);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if (col < H) {
    const int64_t step = 8 * static_cast<int64_t>(H);
    int64_t r = r0 + w;
    const __nv_bfloat16* p = dy + r * H + col;
    for (; r + (kTcBatch - 1) * 8 < r1; r += kTcBatch * 8) {
      uint4 u[kTcBatch];
#pragma unroll
      for (int j = 0; j < kTcBatch; ++j) u[j] = ld_stream_v4(p + j * step);
#pragma unroll
      for (int j = 0; j < kTcBatch; ++j) add_bf16x8(u[j], acc);
      p += kTcBatch * step;
    }
    for (; r < r1; r += 8, p += step) add_bf16x8(ld_global_nc_v4(p), acc);
  }
  float (*red)[256] = reinterpret_cast<float (*)[256]>(smem);  // [8][256]
#pragma unroll
  for (int e = 0; e < 8; ++e) red[w][lane * 8 + e] = acc[e];
  __syncthreads();
  const int c = threadIdx.x;
  if (static_cast<int64_t>(chunk) * 256 + c < H) {
    float t = 0.f;
#pragma unroll
    for (int l = 0; l < 8; ++l) t += red[l][c];
    part[static_cast<int64_t>(split) * H + static_cast<int64_t>(chunk) * 256 + c] = t;
  }
}

cudaError_t launch_transpose_w2(const void* w2, void* w2t, int t, int64_t H, int64_t Fs,
                                const void* dy, int64_t T, int splits, float* part,
                                cudaStream_t s) {
  const int64_t n_tr = w2 != nullptr ? ((Fs + 127) / 128) * (H / 64) * t : 0;
  const int64_t n_cs = dy != nullptr ? ((H + 255) / 256) * splits : 0;
  const int64_t rps = splits > 0 ? (T + splits - 1) / splits : 0;
  if (n_tr + n_cs == 0) return cudaSuccess;
  transpose_w2_colsum_kernel<<<static_cast<unsigned>(n_tr + n_cs), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(w2), static_cast<__nv_bfloat16*>(w2t),
      static_cast<int>(H), static_cast<int>(Fs), static_cast<int>(n_tr),
      static_cast<const __nv_bfloat16*>(dy), T, rps, part);
  return cudaGetLastError();
}

// dst[i] = src[i] over n16 16-byte words: the emulated sequence-parallel gathers and
// scatters.  Grid-stride, four independent words in flight per thread.
__global__ void __launch_bounds__(256) copy16_kernel(uint4* __restrict__ dst,
                                                     const uint4* __restrict__ src, size_t n16) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = ld_global_nc_v4(src + i + j * stride);
#pragma unroll
    for (int j = 0; j < 4; ++j) st_global_v4(dst + i + j * stride, v[j]);
  }
  for (; i < n16; i += stride) st_global_v4(dst + i, ld_global_nc_v4(src + i));
}

cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, int num_sms, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const size_t want = (n16 + 4 * 256 - 1) / (4 * 256);
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>(want, 4 * static_cast<size_t>(num_sms)));
  copy16_kernel<<<blocks, 256, 0, s>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src),
                                       n16);
  return cudaGetLastError();
}

cudaError_t launch_fill_zero(void* p, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  const size_t n16 = bytes / 16;
  const size_t ntail = bytes - n16 * 16;
  const unsigned blocks = static_cast<unsigned>(n16 / 256 + 1 < 4096 ? n16 / 256 + 1 : 4096);
  fill_zero_kernel<<<blocks, 256, 0, s>>>(static_cast<uint4*>(p), n16,
                                          static_cast<uint8_t*>(p) + n16 * 16, ntail);
  return cudaGetLastError();
}

}  // namespace mlpb
