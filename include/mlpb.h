/*
 * mlpb.h -- C ABI of libmlpb: the tensor-parallel transformer MLP block and
 * the sequence-parallel LayerNorm on one GB300 (sm_103a).
 *
 * What the library computes.  "Megatron-LM" source tour (pyshine.com/megatron-lm),
 * section "The Tensor-Parallel Primitives": fc1 is a ColumnParallelLinear (its
 * weight split along the output dimension; every rank sees the full input),
 * fc2 a RowParallelLinear (weight split along the input dimension, partial
 * sums all-reduced at the end), so the block needs one all-reduce.  Section
 * "The Transformer Stack": a fused bias-GELU sits between them; gated
 * variants (SwiGLU) multiply a gate by an up projection.  "Megatron-LM /
 * Megatron-Core" concept note, section "Key math / How it works": the
 * conjugate operators f (identity forward, all-reduce backward) and g
 * (all-reduce forward, identity backward), and sequence parallelism (LN split
 * along the sequence, gathers and reduce-scatters at the GEMM boundaries).
 *
 * The t tensor-parallel ranks are emulated on one device as partitions of the
 * weights.  The g all-reduce is the accumulation of all t shards' K-blocks
 * into one tensor-memory accumulator in the fc2 GEMM; the f all-reduce of the
 * backward is the same accumulation in the dX GEMM.  Sequence shards are
 * contiguous row blocks, so the SP gather / reduce-scatter are index ranges.
 *
 *   GELU:   Z = X W1^T + b1, A = gelu_tanh(Z), Y = A W2^T + b2
 *   SwiGLU: G = X Wg^T, U = X Wu^T, A = silu(G) * U, Y = A W2^T   (no biases)
 *
 * Conventions for every entry point
 *   - Pointers named as tensors are DEVICE pointers, 16-byte aligned, owned by
 *     the caller; the library never frees or retains them past the call.
 *   - bf16 means IEEE bfloat16 (2 bytes); all matrices are row-major.
 *   - Layouts (shard-major, as each tensor-parallel rank stores its slice):
 *       X, Xn, dY           [T][H] bf16
 *       W1 (GELU)           [t][Fs][H] bf16        W1 (SwiGLU) [t][2][Fs][H] (gate, up)
 *       b1                  [F] bf16 (shard i owns b1[i*Fs .. (i+1)*Fs))
 *       W2                  [t][H][Fs] bf16        b2 [H] bf16
 *       Z saved (GELU)      [T][F]  bf16, column i*Fs+j = shard i, feature j
 *       Z saved (SwiGLU)    [T][t][2][Fs] bf16 (G then U of each shard)
 *       A saved             [T][F]  bf16
 *       Y, dX               [T][H] fp32 (bf16 under MLPB_FLAG_BF16_OUT)
 *       dW1, dW2            fp32 in the layouts of W1, W2;  db1 [F], db2 [H] fp32
 *     where T = tokens, H = hidden, F = ffn, t = tp, Fs = F / t.
 *   - With T = 0 the per-row pointers (X, Y, Z/A saved, dY, dX, Xn, mean, rstd, dXn,
 *     workspace) may be NULL; forwards do nothing and backwards write zero parameter
 *     grads (weights, biases, gamma, beta), or leave them as they are when accumulating.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Argument errors are returned synchronously and launch
 *     nothing.  Outputs are overwritten, except the parameter gradients of a handle
 *     created with MLPB_FLAG_ACCUMULATE_GRADS, which are added into.
 *   - A device-side bounded wait that expires (about one second) is recorded in
 *     a per-handle error word and reported by mlpb_last_device_error().
 *   - A handle may be used from one host thread at a time, and its calls must not
 *     overlap on the GPU (issue them on one stream, or order the streams).
 *     mlpb_backward runs part of its work on a second stream that the handle owns,
 *     forked from and joined back into `stream` with events, so all of its work is
 *     ordered before later work on `stream`.
 */
#ifndef MLPB_H_
#define MLPB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mlpb_stream_t; /* identical to cudaStream_t */

typedef enum {
  MLPB_OK = 0,
  MLPB_EINVAL = -1,       /* null / misaligned pointer, bad config value          */
  MLPB_EUNSUPPORTED = -2, /* shape outside the supported set (see mlpb_create)    */
  MLPB_ECUDA = -3,        /* a CUDA runtime call or launch failed                 */
  MLPB_ETIMEOUT = -4,     /* a device-side bounded wait expired (kernel bailed)   */
  MLPB_ENOMEM = -5        /* host allocation failed                               */
} mlpb_status;

typedef enum { MLPB_ACT_GELU_TANH = 0, MLPB_ACT_SWIGLU = 1 } mlpb_act;

/* mlpb_config.flags */
#define MLPB_FLAG_FAULT_INJECT 0x1u    /* test only: the first GEMM launch of the  \
                                          next forward skips one producer arrive, so \
                                          its consumers' bounded wait expires        */
/* Gradient-accumulation fusion ("The Tensor-Parallel Primitives": the linear layers'
 * shared autograd function accumulates weight gradients).  With this flag the parameter
 * gradients of mlpb_backward (dW1, dW2, db1, db2) and mlpb_layernorm_sp_bwd (dgamma,
 * dbeta) are ADDED to what their fp32 buffers hold (main-grad buffers carried across
 * micro-batches) instead of overwriting them; the weight-gradient GEMM epilogues read,
 * add and write each fp32 element once, the bias/LN parameter reductions add their final
 * sums.  The caller zeroes the buffers before the first micro-batch.  With T = 0 the
 * buffers are left as they are.  dX (an activation gradient) is always overwritten. */
#define MLPB_FLAG_ACCUMULATE_GRADS 0x2u
/* Selective activation recomputation (the concept note's "Key math": activation
 * recomputation, selective granularity).  With this flag mlpb_backward does not read
 * the forward's A: the dgrad GEMM's epilogue, which already reads the saved Z (or G, U)
 * for the activation derivative, also rewrites A = act(Z) into the Asaved buffer, and
 * the dW2 GEMM runs after it on that A.  Only Z (G, U) must survive from the forward to
 * the backward; the T*F bf16 A buffer can be scratch shared with other work (the
 * forward writes it for fc2, the backward rewrites it).  A is recomputed from the
 * bf16-rounded Z, so dW2 can differ from the stored-A path by bf16 rounding. */
#define MLPB_FLAG_RECOMPUTE_ACT 0x4u
/* FP8 GEMMs ("Why Megatron-LM Matters" / "Key Features" of the onegen.ai page: mixed
 * precision down to FP8; the concept note's "Key math": FP8 through Transformer Engine).
 * All six GEMMs of mlpb_forward / mlpb_backward run on E4M3 operands (tcgen05
 * kind::f8f6f4, fp32 accumulation) with per-tensor current scaling: each operand tensor
 * (X, W1, W2, A, dY, dZ; every shard at once) gets the power-of-two scale of
 * mlpb_quantize_e4m3 from its own absolute maximum, and each GEMM rescales its sums by
 * the inverse of its two operands' scales.  Everything else keeps the bf16 path's
 * precision: Z (G, U), A and dZ are bf16, Y, dX and the parameter gradients fp32, the
 * bias sums and the LayerNorm unchanged.  The workspace (mlpb_workspace_size) then also
 * holds the E4M3 copies and is required by mlpb_forward too.  Requires F/tp % 16 == 0;
 * not combined with MLPB_FLAG_RECOMPUTE_ACT. */
#define MLPB_FLAG_FP8 0x8u
/* bf16 outputs (the mixed precision of the parallel linears in "The Tensor-Parallel
 * Primitives": activations and their gradients travel in bf16).  With this flag Y
 * (mlpb_forward, mlpb_branch_forward) and dX (mlpb_backward, mlpb_layernorm_sp_bwd,
 * mlpb_branch_backward) are bf16 [T][H] instead of fp32, and mlpb_layernorm_sp_bwd reads
 * its dXn as bf16 (what mlpb_backward then writes).  The sums are the same fp32 values
 * as without the flag, rounded once to bf16 (nearest, ties to even) when stored; the
 * parameter gradients stay fp32.  Halves those tensors' bytes, at the cost of one bf16
 * rounding of Y and dX (up to 2^-9 of each value). */
#define MLPB_FLAG_BF16_OUT 0x10u
/* Emulated sequence-parallel exchange as copies (requires seq_parallel_ln; "The
 * Tensor-Parallel Primitives": with sequence parallelism the linear layers all-gather the
 * sequence-sharded activations in front of the column-parallel GEMM and reduce-scatter
 * after the row-parallel one, and the conjugates in the backward).  Without the flag the
 * gathered tensor is the row-block layout itself (shard s owns rows [s T/t, (s+1) T/t))
 * and no byte moves.  With it, mlpb_forward first copies the input X into a gathered
 * buffer in the workspace and writes fc2's output there before copying its rows out to Y
 * (the scatter; the reduction over shards happened in the accumulator); mlpb_backward
 * gathers X and dY and scatters dX the same way.  Results are bit for bit those of the
 * view; the copies' bytes are reported apart from the algorithmic bytes (timing records
 * "sp_gather_x", "sp_gather_dy", "sp_scatter_y", "sp_scatter_dx").  mlpb_forward then
 * needs the workspace; the workspace holds 8*T*H more bytes. */
#define MLPB_FLAG_EMULATE_COPIES 0x20u

typedef struct {
  int64_t tokens;          /* T: rows of X; multiple of 128 (0 allowed)           */
  int64_t hidden;          /* H: multiple of 64, >= 64                            */
  int64_t ffn;             /* F: divisible by tp, with F/tp a multiple of 8       */
  int32_t tp;              /* t: emulated tensor-parallel degree, 1..1024         */
  int32_t act;             /* mlpb_act                                            */
  int32_t has_bias;        /* GELU only: b1, b2 present (SwiGLU requires 0)       */
  int32_t seq_parallel_ln; /* LN entry points enabled; requires T % t == 0        */
  float ln_eps;            /* LayerNorm epsilon (inside the square root)          */
  uint32_t flags;          /* MLPB_FLAG_*                                         */
} mlpb_config;

typedef struct mlpb_handle mlpb_handle; /* opaque; owns no tensors */

/* Per-kernel timing record (filled when timing is enabled). */
typedef struct {
  char name[32];  /* kernel name, e.g. "fc1_gelu", "colsum_db2"                  */
  float ms;       /* device time between CUDA events recorded around the launch   */
  double flops;   /* algorithmic GEMM flops of the launch (0 for memory kernels)  */
  double bytes;   /* algorithmic HBM bytes of the launch (minimum reads + writes) */
  int32_t kernels; /* CUDA kernels launched inside this record (e.g. 2 for a       \
                      two-pass reduction)                                          */
} mlpb_kernel_time;

/* Validates *cfg, queries the current device and allocates the 4-byte device
 * error word.  Returns EINVAL for a null argument or an out-of-range field,
 * EUNSUPPORTED for shapes outside: T % 128 == 0, H % 64 == 0 and H >= 64,
 * F % tp == 0 and (F/tp) % 8 == 0, SwiGLU without bias, SP with T % tp == 0
 * and H <= 16384.  On success *out owns host state only. */
mlpb_status mlpb_create(const mlpb_config *cfg, mlpb_handle **out);

/* Frees the handle and its error word.  NULL is ignored. */
void mlpb_destroy(mlpb_handle *h);

/* Bytes of device scratch the caller passes as `workspace` to mlpb_forward,
 * mlpb_backward and mlpb_layernorm_sp_bwd (it holds dZ [T][F1] bf16, with a bias the
 * db1 column sums of each 32-row group of dZ that the dgrad epilogue writes, two regions
 * of fp32 partial tiles for the K-range split of a GEMM's last wave -- dX and dW1 run at
 * once on two streams -- a transposed copy of W2 ([F][H] bf16, the dgrad GEMM's operand)
 * (not under MLPB_FLAG_FP8), with a bias db2's column sums over row ranges of dY, and,
 * under MLPB_FLAG_FP8, the E4M3 operand copies and their amax words). */
mlpb_status mlpb_workspace_size(const mlpb_handle *h, size_t *bytes);

/* Bytes of the saved activations: z_bytes for Z (GELU, T*F*2) or G|U (SwiGLU,
 * T*2F*2); a_bytes for A (T*F*2). */
mlpb_status mlpb_saved_size(const mlpb_handle *h, size_t *z_bytes, size_t *a_bytes);

/* Forward of the block ("The Tensor-Parallel Primitives" and "The Transformer
 * Stack" of the source tour; f and g of "Key math").  fc1 over all t column
 * shards with the fused bias+GELU or SwiGLU epilogue writes Zsaved and Asaved;
 * fc2 accumulates all t row shards into one accumulator per output tile (the
 * emulated g all-reduce) and adds b2 once, writing Y [T][H] fp32.  b1 and b2
 * must be NULL when has_bias is 0.  `workspace` is NULL or mlpb_workspace_size() bytes:
 * when given, fc2 uses it to split the K range of the tiles of its last, partly filled
 * wave across idle SM pairs (their partial sums are added by a fixup kernel, in a fixed
 * order); it is required under MLPB_FLAG_FP8. */
mlpb_status mlpb_forward(mlpb_handle *h, const void *X, const void *W1, const void *b1,
                         const void *W2, const void *b2, void *Y, void *Zsaved,
                         void *Asaved, void *workspace, mlpb_stream_t stream);

/* Backward of the block for an upstream gradient dY [T][H] bf16.  g backward is
 * the identity (every shard reads the same dY); dZ = (dY W2_i) * act'(.) per
 * shard; dW2_i = dY^T A_i; dW1_i = dZ_i^T X; db1 = sum_t dZ (column sums of the bf16
 * dZ taken in the dgrad epilogue, then added in row order); db2 = sum_t dY (column sums
 * over row ranges taken in the launch that transposes W2 -- under MLPB_FLAG_FP8 in one of
 * its own -- then added in row-range order);
 * dX = sum_i dZ_i W1_i with the sum over shards accumulated in one tensor-memory
 * accumulator (the emulated f all-reduce).  db1/db2 must be NULL without bias.
 * `workspace` must hold mlpb_workspace_size() bytes.  Asaved is read only (the
 * forward's A), except under MLPB_FLAG_RECOMPUTE_ACT, where it is scratch that the
 * backward writes before reading. */
mlpb_status mlpb_backward(mlpb_handle *h, const void *X, const void *W1, const void *W2,
                          const void *Zsaved, void *Asaved, const void *dY,
                          void *dX, float *dW1, float *dW2, float *db1, float *db2,
                          void *workspace, mlpb_stream_t stream);

/* Sequence-parallel LayerNorm forward ("The Tensor-Parallel Primitives": norms
 * run on sequence-sharded activations).  Shard s owns rows [s*T/t, (s+1)*T/t);
 * each row r gets mean[r], rstd[r] = 1/sqrt(var + eps) (biased variance) and
 * Xn[r] = (X[r]-mean)*rstd*gamma + beta in bf16.  The emulated all-gather is
 * the row-block layout of Xn itself: shard s writes rows s*T/t.. of the gathered
 * tensor that fc1 reads, so no copy is made.
 * X, gamma, beta bf16; mean, rstd [T] fp32.  Requires seq_parallel_ln. */
mlpb_status mlpb_layernorm_sp_fwd(mlpb_handle *h, const void *X, const void *gamma,
                                  const void *beta, void *Xn, float *mean, float *rstd,
                                  mlpb_stream_t stream);

/* Sequence-parallel LayerNorm backward for dXn [T][H] fp32 (the dX output of
 * mlpb_backward run on Xn; bf16 under MLPB_FLAG_BF16_OUT).  dX [T][H] fp32 (bf16 under
 * MLPB_FLAG_BF16_OUT; it may be the dXn buffer itself); dgamma, dbeta [H] fp32 are the sum
 * over shards of each shard's partials (the all-reduce the SP layout implies).
 * `workspace` must hold mlpb_workspace_size() bytes. */
mlpb_status mlpb_layernorm_sp_bwd(mlpb_handle *h, const void *X, const void *gamma,
                                  const float *mean, const float *rstd, const void *dXn,
                                  void *dX, float *dgamma, float *dbeta, void *workspace,
                                  mlpb_stream_t stream);

/* Pre-norm MLP branch of a transformer layer ("The Transformer Stack": the layer runs
 * its MLP branch on the layer-normalised input and adds the branch input back through a
 * residual connection; dropout is left out), sequence-parallel:
 *     Y = X + MLP(LN(X))        (Y [T][H] fp32, bf16 under MLPB_FLAG_BF16_OUT; X, gamma,
 *                                beta bf16)
 * Runs mlpb_layernorm_sp_fwd (writes Xn, mean, rstd, kept for the backward) and the
 * forward of mlpb_forward on Xn, with X added to every output element in fc2's epilogue
 * after b2 (the residual of a row lives on the sequence shard that owns the row).
 * Requires seq_parallel_ln.  Arguments as in the two calls it combines. */
mlpb_status mlpb_branch_forward(mlpb_handle *h, const void *X, const void *gamma,
                                const void *beta, const void *W1, const void *b1,
                                const void *W2, const void *b2, void *Y, void *Xn,
                                float *mean, float *rstd, void *Zsaved, void *Asaved,
                                void *workspace, mlpb_stream_t stream);

/* Backward of mlpb_branch_forward for an upstream gradient dY [T][H] bf16:
 *     dX = dY + LN'(dXn),  dXn = the MLP backward's input gradient on Xn
 * plus dW1, dW2, db1, db2 (as mlpb_backward, on Xn) and dgamma, dbeta (as
 * mlpb_layernorm_sp_bwd).  dXn is formed in the dX buffer and the LayerNorm backward
 * rewrites it in place with the residual gradient dY added in its epilogue, so the call
 * needs no [T][H] buffer beyond dX.  `workspace` holds mlpb_workspace_size() bytes.
 * Honours MLPB_FLAG_ACCUMULATE_GRADS for the parameter gradients. */
mlpb_status mlpb_branch_backward(mlpb_handle *h, const void *X, const void *gamma,
                                 const void *W1, const void *W2, const void *Xn,
                                 const float *mean, const float *rstd, const void *Zsaved,
                                 void *Asaved, const void *dY, void *dX, float *dW1,
                                 float *dW2, float *db1, float *db2, float *dgamma,
                                 float *dbeta, void *workspace, mlpb_stream_t stream);

/* Synchronises `stream`, reads and clears the device error word.  Returns
 * MLPB_ETIMEOUT if a bounded wait expired since the last call, MLPB_ECUDA if
 * the stream reported an error, else MLPB_OK. */
mlpb_status mlpb_last_device_error(mlpb_handle *h, mlpb_stream_t stream);

/* Enables (1) or disables (0) per-kernel CUDA-event timing on the handle.  While it is
 * on, mlpb_backward issues all of its kernels on the caller's stream, one after the other,
 * so that every recorded interval belongs to one kernel. */
mlpb_status mlpb_enable_timing(mlpb_handle *h, int enable);

/* Copies up to `capacity` timing records of the launches since the last read
 * (waiting on their events), sets *count, and clears the list. */
mlpb_status mlpb_read_timings(mlpb_handle *h, mlpb_kernel_time *out, int capacity, int *count);

/* Column sums out[c] = sum_r in[r][c] of a bf16 [rows][cols] matrix into fp32 -- the
 * bias-gradient reduction of mlpb_backward (db2 = sum_t dY, db1 = sum_t dZ) -- for
 * callers that cannot allocate device memory where they need it (code under a memory
 * manager that owns all of the GPU's memory, or inside that manager's own callbacks).
 * The pages have no counterpart: this is an allocation-free variant of the same kernels.
 * It needs no handle and no workspace: its scratch is a fixed 4 MiB device array inside
 * the library (held by every GPU that loads the library until the process exits).
 * Each call looks up that array's device address on the current device (a host-side
 * lookup, so a device reset or a re-created context cannot leave a stale address); the
 * first call on a device also loads the library's device code there, so make it before
 * any stream capture.  Every call shares the one array and the array keeps the last
 * call's partial sums; each call writes every partial it reads before reading it, so
 * nothing needs clearing.  Calls whose kernels overlap on the GPU (other streams, other
 * host threads) race on the array and must be serialised by the caller.
 * Requires cols % 8 == 0 and cols <= 1048576 (one split of fp32 partials must fit the
 * scratch; larger widths return MLPB_EUNSUPPORTED), 16-byte aligned `in` and `out`;
 * rows may be 0 (out becomes zeros, `in` may then be NULL).  Allocates nothing. */
mlpb_status mlpb_bias_grad_noalloc(const void *in, int64_t rows, int64_t cols, float *out,
                                   mlpb_stream_t stream);

/* E4M3 quantization of a bf16 tensor [batches][rows][cols] with one power-of-two scale
 * for the whole tensor (the FP8 recipe of MLPB_FLAG_FP8; "Why Megatron-LM Matters" and
 * "Key Features" of the onegen.ai page name FP8 mixed precision, the concept note's "Key
 * math" FP8 through Transformer Engine).  With amax the largest |x| and k the largest
 * integer such that amax * 2^k <= 448, each code is e4m3(x * 2^k), round to nearest even
 * (x * 2^k is exact).  Writes q [batches][rows][cols] and/or qt [batches][cols][rows]
 * (the transposed codes; either may be NULL, not both), *amax = the fp32 bit pattern of
 * the tensor's largest magnitude (device word, overwritten), and *scale_exp = k (device
 * int, may be NULL).  rows % 16 == 0, cols % 16 == 0, 16-byte aligned tensors, 4-byte
 * aligned words.  Allocates nothing; no handle. */
mlpb_status mlpb_quantize_e4m3(const void *in, int64_t batches, int64_t rows, int64_t cols,
                               void *q, void *qt, uint32_t *amax, int32_t *scale_exp,
                               mlpb_stream_t stream);

/* Static English text of a status code. */
const char *mlpb_status_str(mlpb_status s);

#ifdef __cplusplus
}
#endif
#endif /* MLPB_H_ */
