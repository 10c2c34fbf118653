// Tile shapes, kinds and launch parameters of the tcgen05 GEMM (shared by host and device).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace mlpb {

enum class GemmKind : int {
  FC1_GELU = 0,
  FC1_SWIGLU,
  FC2,
  DGRAD_GELU,
  DGRAD_SWIGLU,
  DX,
  WGRAD_W2,
  WGRAD_W1,
  WGRAD_W2T,  // dW2 computed as its transpose: M = F, N = H (written into dW2's layout)
};

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;  // k-block depth: 64 bf16 = 128-byte K-major rows (128-byte swizzle;
                         // 32-deep blocks with a 64-byte swizzle measured much slower)
constexpr int kChunk = 64 * kBK * 2;  // one 64(MN) x kBK(K) MN-major box, 8 KB
constexpr int kGemmThreads = 192;  // producer, MMA / relay, four epilogue warps
constexpr int kTmemCols = 512;
constexpr int kClusterM = 2;  // CTAs per cluster: the pair along M

// A pair computes a 256 x 256 tile; each CTA keeps its 128 rows of A and its 128-row half
// of B per stage, so a stage is 32 KB per CTA.
constexpr int kPairStages = 7;
constexpr int kPairAStage = kBM * kBK * 2;         // 16 KB
constexpr int kPairBStage = (kBN / 2) * kBK * 2;   // 16 KB
constexpr int kPairStageBytes = kPairAStage + kPairBStage;
constexpr int kPairSmem = kPairStages * kPairStageBytes + 1024 + 512;  // 225.5 KB

struct GemmParams {
  int num_m_tiles, num_n_tiles, num_kb;
  int kb_per_shard;     // FC2: ceil(Fs / 64)
  int tiles_per_shard;  // FC1_SWIGLU: ceil(Fs/128); DGRAD_*, WGRAD_W2: ceil(Fs/256)
  int M;                // valid output rows
  int T, H, F, Fs, t;
  const __nv_bfloat16* bias;  // FC1_GELU: b1; FC2: b2 (nullable)
  const __nv_bfloat16* aux;   // DGRAD_*: saved Z or G|U;  FC2: residual R [T][H] or NULL
  void* out0;
  void* out1;  // FC1_*: A;  DGRAD_*: A recomputed from the saved Z, or NULL
  uint32_t* err;
  uint64_t wait_ns;
  int fault_inject;
  int accumulate;  // weight-gradient kinds: add into the fp32 output instead of overwriting
  int out_bf16;    // FC2, DX: write Y / dX as bf16 (rounded once, from the fp32 sum)
  // FP8 (E4M3) variants: the amax words of the two operands (their power-of-two scales
  // are derived from them), and where FC1 / DGRAD record the amax of the bf16 A / dZ
  // they write (the next GEMMs' operand)
  const uint32_t* amax_a;
  const uint32_t* amax_b;
  uint32_t* amax_out;
  // Tail split: when split > 1, the tiles from super-tile `split_start` on (the last,
  // partly filled wave) are each computed as `split` K-ranges by different pairs, which
  // write raw fp32 partial tiles to `partial` ([tile][part][rank][128][256]); a fixup
  // kernel sums them in part order and applies the epilogue.
  int split;
  int split_start;
  float* partial;
  // DGRAD_GELU with a bias: each warp writes the column sums of its 32 rows of the bf16 dZ
  // it stores, colsum[m / 32][f] ([T/32][F] fp32), for the db1 reduction; NULL: none.
  float* colsum;
  // DGRAD_* (bf16): N tiles run over all F columns of dA, across shard seams (B is W2's
  // transposed copy [F][H], one K-major matrix), so no shard pads its last tile; the
  // SwiGLU epilogue needs Fs % 32 == 0 for this (a 32-column chunk in one shard).  0: N
  // tiles of 256 within each shard (tiles_per_shard a shard).
  int flat_n;
  // M-tile pairs in a raster group (tile_coords); 0: 8.
  int raster_group;
  // MN-major operands loaded through a 3-D map, one box of both 64-wide chunks a stage:
  // bit 0 A, bit 1 B (else two 2-D boxes).
  int mn3d;
};

// FP8 stage: the same 16 KB A and B-half tiles, 128 one-byte elements deep.
constexpr int kBK8 = 128;

}  // namespace mlpb
