// Host-side launch functions of the library's kernels (internal; not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "gemm_params.h"

namespace mlpb {

// gemm_fwd.cu / gemm_bwd.cu: one persistent launch of the tcgen05 GEMM of `kind` on
// `clusters` clusters of kClusterM CTAs.
cudaError_t gemm_fwd_set_smem_attrs();
cudaError_t gemm_bwd_set_smem_attrs();
cudaError_t gemm_max_active_clusters(int* out);
// gemm_fwd.cu: the fixup of a tail-split FC2 / DX / WGRAD_W1 launch (sums the partial
// K-ranges of the tail tiles in part order, adds p.bias and p.aux when set, writes or
// with p.accumulate adds into p.out0, fp32 [M][H]).
cudaError_t launch_split_fixup(const GemmParams& p, cudaStream_t s);
// gemm_fp8.cu: the same GEMMs on E4M3 operands (every operand K-major).
cudaError_t gemm_f8_set_smem_attrs();
cudaError_t launch_gemm_f8(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmParams& p, int clusters, cudaStream_t s);
cudaError_t launch_gemm_fwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int clusters, cudaStream_t s);
cudaError_t launch_gemm_bwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int clusters, cudaStream_t s);

// reduce.cu: column sums of a [R][C] bf16 matrix into fp32, deterministic two passes.
//   pass 1: part[split][C] over row splits of `rows_per_split` rows; pass 2: out[C]
//   (added to the existing out[C] when `accumulate`).
cudaError_t launch_colsum_bf16(const void* in, int64_t R, int64_t C, int splits,
                               int64_t rows_per_split, float* part, float* out, cudaStream_t s,
                               int accumulate = 0);
cudaError_t launch_sum_partials(const float* part, int nparts, int64_t C, float* out,
                                cudaStream_t s, int accumulate = 0);
// Two [nparts][C] partial arrays summed into two outputs in one launch.
cudaError_t launch_sum_partials2(const float* part_a, const float* part_b, int nparts, int64_t C,
                                 float* out_a, float* out_b, cudaStream_t s, int accumulate = 0);
// Two partial arrays of their own sizes ([np_a][C_a], [np_b][C_b]) summed in one launch.
cudaError_t launch_sum_partials_pair(const float* part_a, int np_a, int64_t C_a, float* out_a,
                                     const float* part_b, int np_b, int64_t C_b, float* out_b,
                                     cudaStream_t s, int accumulate = 0);
cudaError_t launch_fill_zero(void* p, size_t bytes, cudaStream_t s);
// reduce.cu: W2 [t][H][Fs] bf16 -> its per-shard transpose W2t [t][Fs][H] (= [F][H]);
// H % 64 == 0, Fs % 8 == 0.  With dy != NULL the same launch writes the first pass of
// db2 = sum_t dY [T][H]: part[split][h] over `splits` row ranges (w2 == NULL: only that).
cudaError_t launch_transpose_w2(const void* w2, void* w2t, int t, int64_t H, int64_t Fs,
                                const void* dy, int64_t T, int splits, float* part,
                                cudaStream_t s);
// reduce.cu: a device copy of `bytes` (a multiple of 16, both pointers 16-byte aligned).
cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, int num_sms, cudaStream_t s);

// layernorm.cu: rows streamed through a shared-memory ring by TMA bulk copies; bounded
// waits report to `err`.
cudaError_t launch_ln_fwd(const void* X, const void* gamma, const void* beta, void* Xn,
                          float* mean, float* rstd, int64_t T, int64_t H, float eps, int num_sms,
                          uint32_t* err, uint64_t wait_ns, cudaStream_t s);
// dres (bf16 [T][H], or NULL) is added to dX: the gradient of a residual around the
// normalised branch.  dXn and dX are fp32, or bf16 with bf16_grads.  dXn may equal dX
// (in place, row by row).
cudaError_t launch_ln_bwd(const void* X, const void* gamma, const float* mean, const float* rstd,
                          const void* dXn, const void* dres, void* dX, bool bf16_grads,
                          float* part_dg, float* part_db, int64_t T, int64_t H, int shards,
                          int blocks_per_shard, uint32_t* err, uint64_t wait_ns, cudaStream_t s);

// fp8.cu: *amax = max(*amax, max|in|) over n bf16 values (n % 8 == 0), as fp32 bits.
cudaError_t launch_amax_bf16(const void* in, int64_t n, uint32_t* amax, int num_sms,
                             cudaStream_t s);
// fp8.cu: bf16 [batches][R][C] -> E4M3 codes q [batches][R][C] and/or qt [batches][C][R]
// (either may be NULL) with the power-of-two scale of *amax; *k_out (if not NULL) gets
// the scale exponent.  R % 8 == 0 and C % 8 == 0.
cudaError_t launch_cast_e4m3(const void* in, int batches, int64_t R, int64_t C, void* q,
                             void* qt, const uint32_t* amax, int32_t* k_out, cudaStream_t s);

}  // namespace mlpb
