// C ABI of libmlpb: handle, validation, tensor-map encoding, launch plans, timing.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/mlpb.h"
#include "kernels.h"

using namespace mlpb;

namespace {

struct TimedLaunch {
  char name[32];
  double flops, bytes;
  int kernels;
  cudaEvent_t start, stop;
};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

mlpb_status load_encoder() {
  std::lock_guard<std::mutex> lock(g_encode_mu);
  if (g_encode != nullptr) return MLPB_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) return MLPB_ECUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return MLPB_OK;
}

// A bf16 tensor map with the swizzle matching its box row.  dims[0] is contiguous;
// strides_bytes[k] is the byte stride of dimension k+1.
bool encode_bf16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box) {
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int k = 0; k < rank; ++k) {
    gd[k] = dims[k];
    bx[k] = box[k];
    es[k] = 1;
    if (k + 1 < rank) gs[k] = strides_bytes[k];
  }
  // the swizzle span is the box's innermost row: 128 B (64 bf16) or 64 B (32 bf16)
  const CUtensorMapSwizzle sw =
      box[0] * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                        const_cast<void*>(ptr), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An E4M3 operand map (one-byte elements, 128-byte swizzle, boxes 128 elements deep).
bool encode_u8(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
               const uint64_t* strides_bytes, const uint32_t* box) {
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int k = 0; k < rank; ++k) {
    gd[k] = dims[k];
    bx[k] = box[k];
    es[k] = 1;
    if (k + 1 < rank) gs[k] = strides_bytes[k];
  }
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank),
                        const_cast<void*>(ptr), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [outer][inner] E4M3, K-major tiles of 128 x 128.
bool map_u8(CUtensorMap* m, const void* p, uint64_t inner, uint64_t outer) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t str[1] = {inner};
  const uint32_t box[2] = {128, 128};
  return encode_u8(m, p, 2, dims, str, box);
}

// [t][rows][inner] E4M3 as a 3-D map {inner, rows, t}, tiles of 128 x 128 in one shard.
bool map_u8_sharded(CUtensorMap* m, const void* p, uint64_t inner, uint64_t rows, uint64_t t,
                    uint64_t row_stride, uint64_t shard_stride) {
  const uint64_t dims[3] = {inner, rows, t};
  const uint64_t str[2] = {row_stride, shard_stride};
  const uint32_t box[3] = {128, 128, 1};
  return encode_u8(m, p, 3, dims, str, box);
}

bool map2d(CUtensorMap* m, const void* p, uint64_t inner, uint64_t outer, uint64_t ld_elems,
           uint32_t box_inner, uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t str[1] = {ld_elems * 2};
  const uint32_t box[2] = {box_inner, box_outer};
  return encode_bf16(m, p, 2, dims, str, box);
}

// An MN-major operand [rows][mn] (rows along K) as a 3-D map {64, rows, mn / 64} whose
// third dimension steps 64 columns (128 bytes): one box {64, 64, 2} brings both 64-column
// chunks of a CTA's 128-wide half, chunk after chunk, the order the MMA's MN-major
// descriptors read -- one copy a stage instead of two.  Needs mn % 64 == 0 (a chunk past
// the end then reads zeros, not the next row); false when it cannot be built.
bool map_mn3d(CUtensorMap* m, const void* p, uint64_t mn, uint64_t rows, uint64_t ld_elems) {
  if (mn % 64 != 0) return false;
  const uint64_t dims[3] = {64, rows, mn / 64};
  const uint64_t str[2] = {ld_elems * 2, 128};
  const uint32_t box[3] = {64, 64, 2};
  return encode_bf16(m, p, 3, dims, str, box);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

struct mlpb_handle {
  mlpb_config cfg;
  int64_t T, H, F, Fs, F1;
  int t;
  bool swiglu;
  int device;
  int num_sms;
  int max_clusters;  // co-resident GEMM clusters
  uint32_t* d_err;  // device error word
  bool fault_pending;
  bool accumulate;  // MLPB_FLAG_ACCUMULATE_GRADS: parameter gradients add into their outputs
  bool recompute;   // MLPB_FLAG_RECOMPUTE_ACT: the backward rewrites A from the saved Z
  bool fp8;         // MLPB_FLAG_FP8: E4M3 GEMMs, per-tensor power-of-two scales
  bool bf16_out;    // MLPB_FLAG_BF16_OUT: Y, dX (and the LN backward's dXn, dX) in bf16
  bool emulate;     // MLPB_FLAG_EMULATE_COPIES: the SP gathers / scatters as device copies
  uint64_t wait_ns;
  int ln_blocks_per_shard;
  // second stream of the backward: db2 at the fork, then (after dgrad) dW2, db1 and dW1
  // beside dX, filling the GEMMs' tails
  cudaStream_t side;
  cudaEvent_t ev_fork, ev_dz, ev_join;
  // timing
  bool timing;
  std::vector<TimedLaunch> launches;
  std::vector<cudaEvent_t> event_pool;

  cudaEvent_t take_event() {
    if (!event_pool.empty()) {
      cudaEvent_t e = event_pool.back();
      event_pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};

namespace {

// Brackets one launch with CUDA events on its stream when timing is enabled.
struct LaunchTimer {
  mlpb_handle* h;
  cudaStream_t s;
  TimedLaunch rec{};
  LaunchTimer(mlpb_handle* h_, cudaStream_t s_, const char* name, double flops, double bytes,
              int kernels = 1)
      : h(h_), s(s_) {
    if (!h->timing) return;
    std::snprintf(rec.name, sizeof(rec.name), "%s", name);
    rec.flops = flops;
    rec.bytes = bytes;
    rec.kernels = kernels;
    rec.start = h->take_event();
    rec.stop = h->take_event();
    cudaEventRecord(rec.start, s);
  }
  void done() {
    if (!h->timing) return;
    cudaEventRecord(rec.stop, s);
    h->launches.push_back(rec);
  }
};

mlpb_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MLPB_OK : MLPB_ECUDA; }

// One emulated sequence-parallel gather or scatter: a device copy, timed like a kernel
// and counted apart from the algorithmic bytes (read + write).
mlpb_status sp_copy(mlpb_handle* h, void* dst, const void* src, size_t bytes, cudaStream_t s,
                    const char* name) {
  LaunchTimer lt(h, s, name, 0.0, 2.0 * bytes);
  cudaError_t e = launch_copy16(dst, src, bytes, h->num_sms, s);
  lt.done();
  return from_cuda(e);
}

constexpr int kShortKRasterGroup = 16;

// Raster group of the two GEMMs whose K is H (fc1, dgrad).  Their 256-row panels are
// short (2.6 MB at H = 5120), so a larger group keeps more of A (X or dY) in L2 while B
// streams past it: 16 M-tile pairs measured 0.4-1 % faster than 8 on these GEMMs, and
// all 32 pairs of the T = 8192 workload 3-4 % slower (32 pairs then ask for each B
// k-block at once).
int short_k_raster_group(const mlpb_handle* h) {
  const int num_pm = static_cast<int>(cdiv(h->T, 2 * kBM));
  return std::max(1, std::min(num_pm, kShortKRasterGroup));
}

GemmParams base_params(const mlpb_handle* h) {
  GemmParams p{};
  p.T = static_cast<int>(h->T);
  p.H = static_cast<int>(h->H);
  p.F = static_cast<int>(h->F);
  p.Fs = static_cast<int>(h->Fs);
  p.t = h->t;
  p.err = h->d_err;
  p.wait_ns = h->wait_ns;
  p.kb_per_shard = static_cast<int>(cdiv(h->Fs, kBK));
  return p;
}

// Tail split of a launch whose last wave of pair tiles is at most half full (FC2 and DX
// with few, long-K tiles; dW1, the backward's last GEMM): the R tail tiles are cut into
// s = min(4, pairs / R) K-ranges computed by different pairs, whose fp32 partials go to
// `partial` (at most one pair tile a pair: max_clusters x 256 KB) and are summed by a
// fixup kernel.
void plan_tail_split(const mlpb_handle* h, GemmParams& p, float* partial) {
  const int super_tiles = static_cast<int>(cdiv(p.num_m_tiles, kClusterM)) * p.num_n_tiles;
  const int clusters = std::min(super_tiles, h->max_clusters);
  if (partial == nullptr || clusters <= 0) return;
  const int tail = super_tiles % clusters;
  if (tail == 0 || 2 * tail > clusters || p.num_kb < 2) return;
  p.split = std::min(std::min(4, clusters / tail), p.num_kb);
  p.split_start = super_tiles - tail;
  p.partial = partial;
}

mlpb_status run_gemm(mlpb_handle* h, GemmKind kind, bool fwd, const CUtensorMap& a,
                     const CUtensorMap& b, const GemmParams& p, cudaStream_t s, const char* name,
                     double flops, double bytes) {
  const int super_tiles = static_cast<int>(cdiv(p.num_m_tiles, kClusterM)) * p.num_n_tiles;
  if (super_tiles == 0) return MLPB_OK;
  const int clusters = std::min(super_tiles, h->max_clusters);
  LaunchTimer lt(h, s, name, flops, bytes, p.split > 1 ? 2 : 1);
  cudaError_t e = fwd ? launch_gemm_fwd(kind, a, b, p, clusters, s)
                      : launch_gemm_bwd(kind, a, b, p, clusters, s);
  if (e == cudaSuccess && p.split > 1) e = launch_split_fixup(p, s);
  lt.done();
  return from_cuda(e);
}

mlpb_status run_gemm_f8(mlpb_handle* h, GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                        const GemmParams& p, cudaStream_t s, const char* name, double flops,
                        double bytes) {
  const int super_tiles = static_cast<int>(cdiv(p.num_m_tiles, kClusterM)) * p.num_n_tiles;
  if (super_tiles == 0) return MLPB_OK;
  const int clusters = std::min(super_tiles, h->max_clusters);
  LaunchTimer lt(h, s, name, flops, bytes);
  cudaError_t e = launch_gemm_f8(kind, a, b, p, clusters, s);
  lt.done();
  return from_cuda(e);
}

// amax of a bf16 tensor of n elements into *slot (which must start at zero).
mlpb_status f8_amax(mlpb_handle* h, const void* x, int64_t n, uint32_t* slot, cudaStream_t s,
                    const char* name) {
  LaunchTimer lt(h, s, name, 0.0, 2.0 * n);
  cudaError_t e = launch_amax_bf16(x, n, slot, h->num_sms, s);
  lt.done();
  return from_cuda(e);
}

// E4M3 copies of a bf16 [batches][R][C] tensor: q (same layout) and/or qt (transposed).
mlpb_status f8_cast(mlpb_handle* h, const void* x, int batches, int64_t R, int64_t C, void* q,
                    void* qt, const uint32_t* slot, cudaStream_t s, const char* name) {
  const double n = static_cast<double>(batches) * R * C;
  LaunchTimer lt(h, s, name, 0.0, n * (2.0 + (q ? 1.0 : 0.0) + (qt ? 1.0 : 0.0)));
  cudaError_t e = launch_cast_e4m3(x, batches, R, C, q, qt, slot, nullptr, s);
  lt.done();
  return from_cuda(e);
}

size_t ws_dz_bytes(const mlpb_handle* h) { return align256(static_cast<size_t>(h->T * h->F1 * 2)); }

// Rows of db1 partial sums: one per 32-row group of dZ (a warp's rows in the dgrad epilogue).
size_t ws_db1_parts(const mlpb_handle* h) { return static_cast<size_t>(h->T / 32); }

// Workspace of the bf16 path: dZ [T][F1] bf16, the db1 partial sums that the dgrad
// epilogue writes ([T/32][F] fp32, with a bias), then the tail split's partial tiles (used
// by fc2 in the forward and by dX in the backward).
size_t ws_split_offset(const mlpb_handle* h) {
  size_t b = ws_dz_bytes(h);
  if (h->cfg.has_bias) b += align256(ws_db1_parts(h) * h->F * 4);
  return b;
}

// Two regions of at most one partial pair tile a pair: fc2 / dX use the first, dW1 (which
// runs beside dX on the other stream) the second.
size_t ws_split_region(const mlpb_handle* h) {
  return align256(static_cast<size_t>(h->max_clusters) * 2 * kBM * kBN * 4);
}

size_t ws_split_bytes(const mlpb_handle* h) { return 2 * ws_split_region(h); }

// The bf16 backward's transposed copy of W2 ([F][H] bf16, the dgrad GEMM's K-major B),
// after the split regions.
size_t ws_w2t_offset(const mlpb_handle* h) { return ws_split_offset(h) + ws_split_bytes(h); }

size_t ws_w2t_bytes(const mlpb_handle* h) {
  return h->fp8 ? 0 : align256(static_cast<size_t>(h->F * h->H * 2));
}

// Row ranges of db2's first pass (written beside the W2 transpose): 256 rows each, at most
// 64, so that the column-sum blocks (H / 256 per range) spread over the GPU.
int db2_splits(const mlpb_handle* h) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(64, h->T / 256)));
}

// db2's partial rows [splits][H] fp32 (with a bias), after W2's copy.
size_t ws_db2_offset(const mlpb_handle* h) { return ws_w2t_offset(h) + ws_w2t_bytes(h); }

size_t ws_db2_bytes(const mlpb_handle* h) {
  return h->cfg.has_bias ? align256(static_cast<size_t>(db2_splits(h)) * h->H * 4) : 0;
}

size_t ws_backward_bytes(const mlpb_handle* h) { return ws_db2_offset(h) + ws_db2_bytes(h); }

float* ws_split_partial(const mlpb_handle* h, void* workspace, int region = 0) {
  return workspace == nullptr
             ? nullptr
             : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ws_split_offset(h) +
                                        region * ws_split_region(h));
}

size_t ws_ln_bytes(const mlpb_handle* h) {
  if (!h->cfg.seq_parallel_ln) return 0;
  const size_t nblk = static_cast<size_t>(h->t) * h->ln_blocks_per_shard;
  return 2 * align256(nblk * h->H * 4);
}

// FP8 region of the workspace, after the bf16 path's scratch: the amax words, then the
// E4M3 copies of the six GEMM operands, each in its own layout and transposed.
enum F8Amax { kAmaxX = 0, kAmaxW1, kAmaxW2, kAmaxA, kAmaxDY, kAmaxDZ, kAmaxWords = 8 };
struct F8Layout {
  uint32_t* amax;
  uint8_t *Xq, *Xt, *W1q, *W1t, *W2q, *W2t, *Aq, *At, *dYq, *dYt, *dZq, *dZt;
};

size_t ws_base_bytes(const mlpb_handle* h) {
  return align256(std::max<size_t>(std::max(ws_backward_bytes(h), ws_ln_bytes(h)), 256));
}

size_t ws_f8_bytes(const mlpb_handle* h) {
  if (!h->fp8) return 0;
  const size_t TH = static_cast<size_t>(h->T * h->H), F1H = static_cast<size_t>(h->F1 * h->H),
               FH = static_cast<size_t>(h->F * h->H), TF = static_cast<size_t>(h->T * h->F),
               TF1 = static_cast<size_t>(h->T * h->F1);
  return 256 + 2 * (align256(TH) + align256(F1H) + align256(FH) + align256(TF) + align256(TH) +
                    align256(TF1));
}

F8Layout f8_layout(const mlpb_handle* h, void* workspace) {
  uint8_t* b = static_cast<uint8_t*>(workspace) + ws_base_bytes(h);
  F8Layout L;
  L.amax = reinterpret_cast<uint32_t*>(b);
  b += 256;
  auto take = [&b](size_t n) {
    uint8_t* p = b;
    b += align256(n);
    return p;
  };
  const size_t TH = static_cast<size_t>(h->T * h->H), F1H = static_cast<size_t>(h->F1 * h->H),
               FH = static_cast<size_t>(h->F * h->H), TF = static_cast<size_t>(h->T * h->F),
               TF1 = static_cast<size_t>(h->T * h->F1);
  L.Xq = take(TH);
  L.Xt = take(TH);
  L.W1q = take(F1H);
  L.W1t = take(F1H);
  L.W2q = take(FH);
  L.W2t = take(FH);
  L.Aq = take(TF);
  L.At = take(TF);
  L.dYq = take(TH);
  L.dYt = take(TH);
  L.dZq = take(TF1);
  L.dZt = take(TF1);
  return L;
}


// Regions of the emulated sequence-parallel exchange (MLPB_FLAG_EMULATE_COPIES), after
// everything else: the gathered input [T][H] bf16, the gathered upstream gradient [T][H]
// bf16, and the full output before its scatter [T][H] (fp32, or bf16 with bf16 outputs).
struct CopyLayout {
  void *xfull, *dyfull, *outfull;
};

size_t ws_copy_bytes(const mlpb_handle* h) {
  if (!h->emulate) return 0;
  const size_t TH = static_cast<size_t>(h->T * h->H);
  return 2 * align256(2 * TH) + align256(4 * TH);
}

CopyLayout copy_layout(const mlpb_handle* h, void* workspace) {
  const size_t TH = static_cast<size_t>(h->T * h->H);
  uint8_t* b = static_cast<uint8_t*>(workspace) + ws_base_bytes(h) + ws_f8_bytes(h);
  return CopyLayout{b, b + align256(2 * TH), b + 2 * align256(2 * TH)};
}

size_t ws_total_bytes(const mlpb_handle* h) {
  return ws_base_bytes(h) + ws_f8_bytes(h) + ws_copy_bytes(h);
}

}  // namespace

extern "C" {

const char* mlpb_status_str(mlpb_status s) {
  switch (s) {
    case MLPB_OK: return "ok";
    case MLPB_EINVAL: return "invalid argument";
    case MLPB_EUNSUPPORTED: return "unsupported shape or configuration";
    case MLPB_ECUDA: return "CUDA error";
    case MLPB_ETIMEOUT: return "device-side bounded wait expired";
    case MLPB_ENOMEM: return "out of host memory";
  }
  return "unknown status";
}

mlpb_status mlpb_create(const mlpb_config* cfg, mlpb_handle** out) {
  if (cfg == nullptr || out == nullptr) return MLPB_EINVAL;
  *out = nullptr;
  const mlpb_config& c = *cfg;
  if (c.tokens < 0 || c.hidden <= 0 || c.ffn <= 0 || c.tp < 1 || c.tp > 1024) return MLPB_EINVAL;
  if (c.act != MLPB_ACT_GELU_TANH && c.act != MLPB_ACT_SWIGLU) return MLPB_EINVAL;
  if (c.has_bias != 0 && c.has_bias != 1) return MLPB_EINVAL;
  if (c.seq_parallel_ln != 0 && c.seq_parallel_ln != 1) return MLPB_EINVAL;
  if ((c.flags & ~(MLPB_FLAG_FAULT_INJECT | MLPB_FLAG_ACCUMULATE_GRADS |
                   MLPB_FLAG_RECOMPUTE_ACT | MLPB_FLAG_FP8 | MLPB_FLAG_BF16_OUT |
                   MLPB_FLAG_EMULATE_COPIES)) != 0)
    return MLPB_EINVAL;
  if (c.seq_parallel_ln && !(c.ln_eps > 0.f)) return MLPB_EINVAL;
  if ((c.flags & MLPB_FLAG_EMULATE_COPIES) && !c.seq_parallel_ln) return MLPB_EUNSUPPORTED;
  if (c.tokens % 128 != 0 || c.hidden % 64 != 0) return MLPB_EUNSUPPORTED;
  if (c.ffn % c.tp != 0 || (c.ffn / c.tp) % 8 != 0) return MLPB_EUNSUPPORTED;
  if (c.act == MLPB_ACT_SWIGLU && c.has_bias) return MLPB_EUNSUPPORTED;
  if ((c.flags & MLPB_FLAG_FP8) &&
      ((c.ffn / c.tp) % 16 != 0 || (c.flags & MLPB_FLAG_RECOMPUTE_ACT)))
    return MLPB_EUNSUPPORTED;  // E4M3 rows must be 16-byte multiples for TMA
  if (c.seq_parallel_ln && (c.tokens % c.tp != 0 || c.hidden > 16384)) return MLPB_EUNSUPPORTED;
  const int64_t f1 = c.act == MLPB_ACT_SWIGLU ? 2 * c.ffn : c.ffn;
  // int32 tile/coordinate arithmetic inside the kernels
  if (c.tokens > (int64_t(1) << 30) || c.hidden > (int64_t(1) << 30) || f1 > (int64_t(1) << 30) ||
      c.hidden * c.tp > (int64_t(1) << 30))
    return MLPB_EUNSUPPORTED;

  mlpb_handle* h = new (std::nothrow) mlpb_handle();
  if (h == nullptr) return MLPB_ENOMEM;
  h->cfg = c;
  h->T = c.tokens;
  h->H = c.hidden;
  h->F = c.ffn;
  h->t = c.tp;
  h->Fs = c.ffn / c.tp;
  h->swiglu = c.act == MLPB_ACT_SWIGLU;
  h->F1 = f1;
  h->fault_pending = (c.flags & MLPB_FLAG_FAULT_INJECT) != 0;
  h->accumulate = (c.flags & MLPB_FLAG_ACCUMULATE_GRADS) != 0;
  h->recompute = (c.flags & MLPB_FLAG_RECOMPUTE_ACT) != 0;
  h->fp8 = (c.flags & MLPB_FLAG_FP8) != 0;
  h->bf16_out = (c.flags & MLPB_FLAG_BF16_OUT) != 0;
  h->emulate = (c.flags & MLPB_FLAG_EMULATE_COPIES) != 0;
  h->wait_ns = 1000000000ull;
  h->timing = false;
  h->d_err = nullptr;

  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
          cudaSuccess) {
    delete h;
    return MLPB_ECUDA;
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device);
  if (major != 10 || minor != 3) {  // the kernels are built for sm_103a only
    delete h;
    return MLPB_EUNSUPPORTED;
  }
  if (load_encoder() != MLPB_OK || gemm_fwd_set_smem_attrs() != cudaSuccess ||
      gemm_bwd_set_smem_attrs() != cudaSuccess ||
      (h->fp8 && gemm_f8_set_smem_attrs() != cudaSuccess) ||
      cudaMalloc(reinterpret_cast<void**>(&h->d_err), sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(h->d_err, 0, sizeof(uint32_t)) != cudaSuccess) {
    if (h->d_err) cudaFree(h->d_err);
    delete h;
    return MLPB_ECUDA;
  }
  if (gemm_max_active_clusters(&h->max_clusters) != cudaSuccess || h->max_clusters < 1) {
    cudaFree(h->d_err);
    delete h;
    return MLPB_ECUDA;
  }
  h->side = nullptr;
  h->ev_fork = h->ev_dz = h->ev_join = nullptr;
  if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_dz, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) {
    mlpb_destroy(h);
    return MLPB_ECUDA;
  }
  // LN backward: two CTAs per SM, split evenly over the t sequence shards
  h->ln_blocks_per_shard =
      static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(2 * h->num_sms, h->t),
                                                               h->t ? h->T / h->t : 1)));
  *out = h;
  return MLPB_OK;
}

void mlpb_destroy(mlpb_handle* h) {
  if (h == nullptr) return;
  for (auto& l : h->launches) {
    cudaEventDestroy(l.start);
    cudaEventDestroy(l.stop);
  }
  for (auto e : h->event_pool) cudaEventDestroy(e);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_dz) cudaEventDestroy(h->ev_dz);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->d_err) cudaFree(h->d_err);
  delete h;
}

mlpb_status mlpb_workspace_size(const mlpb_handle* h, size_t* bytes) {
  if (h == nullptr || bytes == nullptr) return MLPB_EINVAL;
  *bytes = ws_total_bytes(h);
  return MLPB_OK;
}

mlpb_status mlpb_saved_size(const mlpb_handle* h, size_t* z_bytes, size_t* a_bytes) {
  if (h == nullptr || z_bytes == nullptr || a_bytes == nullptr) return MLPB_EINVAL;
  *z_bytes = static_cast<size_t>(h->T * h->F1 * 2);
  *a_bytes = static_cast<size_t>(h->T * h->F * 2);
  return MLPB_OK;
}

static mlpb_status forward_impl(mlpb_handle* h, const void* X, const void* W1, const void* b1,
                                const void* W2, const void* b2, void* Y, void* Zsaved,
                                void* Asaved, const void* resid, void* workspace,
                                cudaStream_t s);
static mlpb_status backward_f8(mlpb_handle* h, const void* X, const void* W1, const void* W2,
                               const void* Zsaved, const void* Asaved, const void* dY,
                               void* dX, float* dW1, float* dW2, float* db1, float* db2,
                               void* workspace, cudaStream_t s);
static mlpb_status ln_bwd_impl(mlpb_handle* h, const void* X, const void* gamma,
                               const float* mean, const float* rstd, const void* dXn,
                               const void* dres, void* dX, float* dgamma, float* dbeta,
                               void* workspace, cudaStream_t s);

mlpb_status mlpb_forward(mlpb_handle* h, const void* X, const void* W1, const void* b1,
                         const void* W2, const void* b2, void* Y, void* Zsaved, void* Asaved,
                         void* workspace, mlpb_stream_t stream) {
  if (h == nullptr) return MLPB_EINVAL;
  const bool bias = h->cfg.has_bias != 0;
  if (!W1 || !W2) return MLPB_EINVAL;
  if (h->T > 0 && (!X || !Y || !Zsaved || !Asaved)) return MLPB_EINVAL;  // T = 0: empty tensors
  if (h->T > 0 && (h->fp8 || h->emulate) && (!workspace || !aligned16(workspace)))
    return MLPB_EINVAL;
  if (bias != (b1 != nullptr) || bias != (b2 != nullptr)) return MLPB_EINVAL;
  for (const void* p : {X, W1, W2, static_cast<const void*>(Y), static_cast<const void*>(Zsaved),
                        static_cast<const void*>(Asaved), b1, b2})
    if (p && !aligned16(p)) return MLPB_EINVAL;
  if (h->T == 0) return MLPB_OK;
  return forward_impl(h, X, W1, b1, W2, b2, Y, Zsaved, Asaved, nullptr, workspace,
                      reinterpret_cast<cudaStream_t>(stream));
}

// fc1 and fc2 of a validated forward; `resid` (bf16 [T][H] or NULL) is added to Y in
// fc2's epilogue after b2.
// The forward with E4M3 GEMMs: amax and E4M3 copies of X, W1, W2; fc1 (records amax(A));
// the E4M3 copies of A and W2; fc2; all on the caller's stream, each GEMM's operands cast
// right before it so that it finds them in L2.  (Running the weights' amax and casts on a
// second stream beside X's and fc1 measured no faster: a persistent GEMM CTA holds 225 KB
// of shared memory, so the casts cannot share its SMs.)
static mlpb_status forward_f8(mlpb_handle* h, const void* X, const void* W1, const void* b1,
                              const void* W2, const void* b2, void* Y, void* Zsaved,
                              void* Asaved, const void* resid, void* workspace, cudaStream_t s) {
  const bool bias = h->cfg.has_bias != 0;
  const int64_t T = h->T, H = h->H, F = h->F, Fs = h->Fs, t = h->t, F1 = h->F1;
  const F8Layout L = f8_layout(h, workspace);
  uint32_t* am = L.amax;

  // tensor maps first: an encoding error launches nothing
  CUtensorMap ta1, tb1, ta2, tb2;
  GemmParams p = base_params(h);
  p.M = static_cast<int>(T);
  p.num_m_tiles = static_cast<int>(T / kBM);
  p.num_kb = static_cast<int>(cdiv(H, kBK8));
  p.out0 = Zsaved;
  p.out1 = Asaved;
  p.amax_a = am + kAmaxX;
  p.amax_b = am + kAmaxW1;
  p.amax_out = am + kAmaxA;
  bool ok = map_u8(&ta1, L.Xq, H, T);
  if (!h->swiglu) {
    ok = ok && map_u8(&tb1, L.W1q, H, F);
    p.num_n_tiles = static_cast<int>(cdiv(F, kBN));
    p.bias = static_cast<const __nv_bfloat16*>(b1);
  } else {
    const uint64_t dims[4] = {static_cast<uint64_t>(H), static_cast<uint64_t>(Fs), 2,
                              static_cast<uint64_t>(t)};
    const uint64_t str[3] = {static_cast<uint64_t>(H), static_cast<uint64_t>(Fs * H),
                             static_cast<uint64_t>(2 * Fs * H)};
    const uint32_t box[4] = {128, 128, 1, 1};
    ok = ok && encode_u8(&tb1, L.W1q, 4, dims, str, box);
    p.tiles_per_shard = static_cast<int>(cdiv(Fs, 128));
    p.num_n_tiles = static_cast<int>(t * p.tiles_per_shard);
  }
  ok = ok && map_u8_sharded(&ta2, L.Aq, Fs, T, t, F, Fs) &&
       map_u8_sharded(&tb2, L.W2q, Fs, H, t, Fs, H * Fs);
  if (!ok) return MLPB_EINVAL;
  GemmParams q = base_params(h);
  q.M = static_cast<int>(T);
  q.num_m_tiles = static_cast<int>(T / kBM);
  q.num_n_tiles = static_cast<int>(cdiv(H, kBN));
  q.kb_per_shard = static_cast<int>(cdiv(Fs, kBK8));
  q.num_kb = static_cast<int>(t * q.kb_per_shard);
  q.bias = static_cast<const __nv_bfloat16*>(b2);
  q.aux = static_cast<const __nv_bfloat16*>(resid);
  q.out0 = Y;
  q.out_bf16 = h->bf16_out ? 1 : 0;
  q.amax_a = am + kAmaxA;
  q.amax_b = am + kAmaxW2;

  if (cudaMemsetAsync(am, 0, kAmaxWords * sizeof(uint32_t), s) != cudaSuccess)
    return MLPB_ECUDA;
  mlpb_status st = f8_amax(h, W1, F1 * H, am + kAmaxW1, s, "fp8_amax_w1");
  if (st == MLPB_OK) st = f8_amax(h, W2, F * H, am + kAmaxW2, s, "fp8_amax_w2");
  if (st == MLPB_OK) st = f8_amax(h, X, T * H, am + kAmaxX, s, "fp8_amax_x");
  if (st == MLPB_OK) st = f8_cast(h, X, 1, T, H, L.Xq, nullptr, am + kAmaxX, s, "fp8_cast_x");
  if (st == MLPB_OK)  // W1q last before fc1, so that fc1 finds it in L2
    st = f8_cast(h, W1, 1, F1, H, L.W1q, nullptr, am + kAmaxW1, s, "fp8_cast_w1");
  if (st == MLPB_OK) {
    p.fault_inject = h->fault_pending ? 1 : 0;
    h->fault_pending = false;
    st = run_gemm_f8(h, h->swiglu ? GemmKind::FC1_SWIGLU : GemmKind::FC1_GELU, ta1, tb1, p, s,
                     h->swiglu ? "fc1_swiglu_f8" : "fc1_gelu_f8",
                     (h->swiglu ? 4.0 : 2.0) * T * F * H,
                     h->swiglu ? 1.0 * (T * H + 2 * F * H) + 6.0 * T * F
                               : 1.0 * (T * H + F * H) + 4.0 * T * F + (bias ? 2.0 * F : 0.0));
  }
  if (st == MLPB_OK)
    st = f8_cast(h, Asaved, 1, T, F, L.Aq, nullptr, am + kAmaxA, s, "fp8_cast_a");
  if (st == MLPB_OK)
    st = f8_cast(h, W2, 1, t * H, Fs, L.W2q, nullptr, am + kAmaxW2, s, "fp8_cast_w2");
  if (st != MLPB_OK) return st;
  // ---- fc2 (the sum over shards accumulates in one TMEM tile; one scale for all shards)
  return run_gemm_f8(h, GemmKind::FC2, ta2, tb2, q, s, "fc2_f8", 2.0 * T * H * F,
                     1.0 * (T * F + H * F) + (h->bf16_out ? 2.0 : 4.0) * T * H +
                         (bias ? 2.0 * H : 0.0) + (resid ? 2.0 * T * H : 0.0));
}

static mlpb_status forward_core(mlpb_handle* h, const void* X, const void* W1, const void* b1,
                                const void* W2, const void* b2, void* Y, void* Zsaved,
                                void* Asaved, const void* resid, void* workspace,
                                cudaStream_t s) {
  if (h->fp8) return forward_f8(h, X, W1, b1, W2, b2, Y, Zsaved, Asaved, resid, workspace, s);
  const bool bias = h->cfg.has_bias != 0;
  const int64_t T = h->T, H = h->H, F = h->F, Fs = h->Fs, t = h->t;

  // Tensor maps of both GEMMs first: an encoding error launches nothing.
  CUtensorMap ta1, tb1, ta2, tb2;
  bool ok = map2d(&ta1, X, H, T, H, kBK, kBM);
  // Every operand as a 2-D map (measured faster than 3-D / 4-D maps with the pair's shared
  // barrier): the shard index folds into the row index (W1 [t][2][Fs][H] as [2F][H], W2
  // [t][H][Fs] as [tH][Fs]) or the column (A [T][t][Fs] as [T][F]).  A box that runs past
  // a shard's Fs columns or rows reads the next shard's values, which meet zero-filled B
  // columns (K past Fs) or land in output columns the epilogue drops.
  ok = ok && map2d(&tb1, W1, H, h->F1, H, kBK, h->swiglu ? 128 : kBN / 2);
  ok = ok && map2d(&ta2, Asaved, F, T, F, kBK, kBM) &&
       map2d(&tb2, W2, Fs, t * H, Fs, kBK, kBN / 2);
  if (!ok) return MLPB_EINVAL;

  // ---- fc1 (column-parallel; f forward = every shard reads the same X)
  GemmParams p = base_params(h);
  p.M = static_cast<int>(T);
  p.num_m_tiles = static_cast<int>(T / kBM);
  p.num_kb = static_cast<int>(cdiv(H, kBK));
  p.out0 = Zsaved;
  p.out1 = Asaved;
  p.fault_inject = h->fault_pending ? 1 : 0;
  h->fault_pending = false;
  p.raster_group = short_k_raster_group(h);
  mlpb_status st;
  if (!h->swiglu) {
    p.num_n_tiles = static_cast<int>(cdiv(F, kBN));
    p.bias = static_cast<const __nv_bfloat16*>(b1);
    st = run_gemm(h, GemmKind::FC1_GELU, true, ta1, tb1, p, s, "fc1_gelu", 2.0 * T * F * H,
                  2.0 * (T * H + F * H + 2 * T * F) + (bias ? 2.0 * F : 0.0));
  } else {
    p.tiles_per_shard = static_cast<int>(cdiv(Fs, 128));
    p.num_n_tiles = static_cast<int>(t * p.tiles_per_shard);
    st = run_gemm(h, GemmKind::FC1_SWIGLU, true, ta1, tb1, p, s, "fc1_swiglu", 4.0 * T * F * H,
                  2.0 * (T * H + 2 * F * H + 3 * T * F));
  }
  if (st != MLPB_OK) return st;

  // ---- fc2 (row-parallel; g forward = all t shards accumulate into one TMEM tile)
  GemmParams q = base_params(h);
  q.M = static_cast<int>(T);
  q.num_m_tiles = static_cast<int>(T / kBM);
  q.num_n_tiles = static_cast<int>(cdiv(H, kBN));
  q.num_kb = static_cast<int>(t * q.kb_per_shard);
  q.bias = static_cast<const __nv_bfloat16*>(b2);
  q.aux = static_cast<const __nv_bfloat16*>(resid);
  q.out0 = Y;
  q.out_bf16 = h->bf16_out ? 1 : 0;
  plan_tail_split(h, q, ws_split_partial(h, workspace));
  return run_gemm(h, GemmKind::FC2, true, ta2, tb2, q, s, "fc2", 2.0 * T * H * F,
                  2.0 * (T * F + H * F) + (h->bf16_out ? 2.0 : 4.0) * T * H +
                      (bias ? 2.0 * H : 0.0) + (resid ? 2.0 * T * H : 0.0));
}

// The forward of validated arguments.  With emulated sequence-parallel copies, the input's
// sequence shards are first gathered into one [T][H] tensor (the all-gather in front of
// fc1), and fc2's output -- already summed over the tensor-parallel shards in the
// accumulator -- is scattered back to the rows' own shards (the reduce-scatter's scatter).
static mlpb_status forward_impl(mlpb_handle* h, const void* X, const void* W1, const void* b1,
                                const void* W2, const void* b2, void* Y, void* Zsaved,
                                void* Asaved, const void* resid, void* workspace,
                                cudaStream_t s) {
  if (!h->emulate)
    return forward_core(h, X, W1, b1, W2, b2, Y, Zsaved, Asaved, resid, workspace, s);
  const CopyLayout C = copy_layout(h, workspace);
  const size_t TH = static_cast<size_t>(h->T * h->H);
  mlpb_status st = sp_copy(h, C.xfull, X, 2 * TH, s, "sp_gather_x");
  if (st == MLPB_OK)
    st = forward_core(h, C.xfull, W1, b1, W2, b2, C.outfull, Zsaved, Asaved, resid, workspace,
                      s);
  if (st == MLPB_OK) st = sp_copy(h, Y, C.outfull, (h->bf16_out ? 2 : 4) * TH, s, "sp_scatter_y");
  return st;
}

static mlpb_status backward_core(mlpb_handle* h, const void* X, const void* W1, const void* W2,
                                 const void* Zsaved, void* Asaved, const void* dY, void* dX,
                                 float* dW1, float* dW2, float* db1, float* db2, void* workspace,
                                 cudaStream_t s);

mlpb_status mlpb_backward(mlpb_handle* h, const void* X, const void* W1, const void* W2,
                          const void* Zsaved, void* Asaved, const void* dY, void* dX,
                          float* dW1, float* dW2, float* db1, float* db2, void* workspace,
                          mlpb_stream_t stream) {
  if (h == nullptr) return MLPB_EINVAL;
  const bool bias = h->cfg.has_bias != 0;
  if (!W1 || !W2 || !dW1 || !dW2) return MLPB_EINVAL;
  if (h->T > 0 && (!X || !Zsaved || !Asaved || !dY || !dX || !workspace))
    return MLPB_EINVAL;  // T = 0: the activation tensors are empty
  if (bias != (db1 != nullptr) || bias != (db2 != nullptr)) return MLPB_EINVAL;
  for (const void* p : {X, W1, W2, Zsaved, static_cast<const void*>(Asaved), dY,
                        static_cast<const void*>(dX), static_cast<const void*>(dW1),
                        static_cast<const void*>(dW2),
                        static_cast<const void*>(db1), static_cast<const void*>(db2),
                        static_cast<const void*>(workspace)})
    if (p && !aligned16(p)) return MLPB_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t T = h->T, H = h->H, F = h->F, Fs = h->Fs, t = h->t, F1 = h->F1;
  mlpb_status st = MLPB_OK;

  const int acc = h->accumulate ? 1 : 0;
  if (T == 0) {  // empty batch: every parameter gradient is zero (adds nothing when accumulating)
    if (acc) return MLPB_OK;
    st = from_cuda(launch_fill_zero(dW1, static_cast<size_t>(F1 * H * 4), s));
    if (st == MLPB_OK) st = from_cuda(launch_fill_zero(dW2, static_cast<size_t>(F * H * 4), s));
    if (st == MLPB_OK && bias) st = from_cuda(launch_fill_zero(db1, static_cast<size_t>(F * 4), s));
    if (st == MLPB_OK && bias) st = from_cuda(launch_fill_zero(db2, static_cast<size_t>(H * 4), s));
    return st;
  }

  if (!h->emulate)
    return backward_core(h, X, W1, W2, Zsaved, Asaved, dY, dX, dW1, dW2, db1, db2, workspace, s);
  // emulated sequence parallelism: gather the input again (for dW1) and the upstream
  // gradient (the all-gather that is the reduce-scatter's backward), scatter dX's rows
  const CopyLayout C = copy_layout(h, workspace);
  const size_t TH = static_cast<size_t>(T * H);
  st = sp_copy(h, C.xfull, X, 2 * TH, s, "sp_gather_x");
  if (st == MLPB_OK) st = sp_copy(h, C.dyfull, dY, 2 * TH, s, "sp_gather_dy");
  if (st == MLPB_OK)
    st = backward_core(h, C.xfull, W1, W2, Zsaved, Asaved, C.dyfull, C.outfull, dW1, dW2, db1,
                       db2, workspace, s);
  if (st == MLPB_OK)
    st = sp_copy(h, dX, C.outfull, (h->bf16_out ? 2 : 4) * TH, s, "sp_scatter_dx");
  return st;
}

// The backward of validated arguments with T > 0.
static mlpb_status backward_core(mlpb_handle* h, const void* X, const void* W1, const void* W2,
                                 const void* Zsaved, void* Asaved, const void* dY, void* dX,
                                 float* dW1, float* dW2, float* db1, float* db2, void* workspace,
                                 cudaStream_t s) {
  if (h->fp8)
    return backward_f8(h, X, W1, W2, Zsaved, Asaved, dY, dX, dW1, dW2, db1, db2, workspace, s);
  const bool bias = h->cfg.has_bias != 0;
  const int64_t T = h->T, H = h->H, F = h->F, Fs = h->Fs, t = h->t, F1 = h->F1;
  const int acc = h->accumulate ? 1 : 0;
  mlpb_status st = MLPB_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* dZ = ws;
  float* part1 = reinterpret_cast<float*>(ws + ws_dz_bytes(h));  // db1 partials [T/32][F]
  const bool recompute = h->recompute;

  // Tensor maps of all four GEMMs first: an encoding error launches nothing.
  CUtensorMap tdgA, tdgB, tw2A, tw2B, tw1A, tw1B, tdxA, tdxB;
  int mn3d_w2 = 0, mn3d_w1 = 0, mn3d_dx = 0;
  void* w2t = ws + ws_w2t_offset(h);
  {
    // the dgrad's B is W2's per-shard transpose [F][H] (K-major rows i Fs + j), written by
    // the transpose below; with N tiles per shard, a 128-row box past shard i's Fs rows
    // reads the next shard's rows, which land in output columns the epilogue drops
    if (!map2d(&tdgA, dY, H, T, H, kBK, kBM) || !map2d(&tdgB, w2t, H, F, H, kBK, kBN / 2) ||
        !map2d(&tdxA, dZ, F1, T, F1, kBK, kBM))
      return MLPB_EINVAL;
    // the MN-major operands: 3-D maps (one copy a stage) where they can be built
    mn3d_w2 = (map_mn3d(&tw2A, Asaved, F, T, F) ? 1 : 0) | (map_mn3d(&tw2B, dY, H, T, H) ? 2 : 0);
    mn3d_w1 = (map_mn3d(&tw1A, dZ, F1, T, F1) ? 1 : 0) | (map_mn3d(&tw1B, X, H, T, H) ? 2 : 0);
    mn3d_dx = map_mn3d(&tdxB, W1, H, F1, H) ? 2 : 0;
    if ((!(mn3d_w2 & 1) && !map2d(&tw2A, Asaved, F, T, F, 64, kBK)) ||
        (!(mn3d_w2 & 2) && !map2d(&tw2B, dY, H, T, H, 64, kBK)) ||
        (!(mn3d_w1 & 1) && !map2d(&tw1A, dZ, F1, T, F1, 64, kBK)) ||
        (!(mn3d_w1 & 2) && !map2d(&tw1B, X, H, T, H, 64, kBK)) ||
        (!(mn3d_dx & 2) && !map2d(&tdxB, W1, H, F1, H, 64, kBK)))
      return MLPB_EINVAL;
  }

  // With per-kernel timing on, everything stays on `stream`, so that each kernel's
  // CUDA-event interval is its own and not shared with a concurrent one.
  cudaStream_t s2 = h->timing ? s : h->side;

  // Fork: after dgrad, stream s2 runs dW2, the bias sums and dW1 beside dX.
  if (cudaEventRecord(h->ev_fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(s2, h->ev_fork, 0) != cudaSuccess)
    return MLPB_ECUDA;

  // ---- [s] W2's per-shard transpose for the dgrad (K-major B) and, in the same launch,
  // the first pass of db2 = sum_t dY (g backward is the identity: the bias sees dY itself)
  float* part2 = reinterpret_cast<float*>(ws + ws_db2_offset(h));  // db2 partials [splits][H]
  const int splits2 = db2_splits(h);
  {
    LaunchTimer lt(h, s, "w2_transpose_db2", 0.0,
                   4.0 * F * H + (bias ? 2.0 * T * H + 4.0 * splits2 * H : 0.0));
    cudaError_t e = launch_transpose_w2(W2, w2t, static_cast<int>(t), H, Fs,
                                        bias ? dY : nullptr, T, splits2, part2, s);
    lt.done();
    st = from_cuda(e);
  }

  // ---- [s] dgrad of fc2 with the fused activation derivative: dZ [T][F1]
  if (st == MLPB_OK) {
    GemmParams p = base_params(h);
    p.M = static_cast<int>(T);
    p.num_m_tiles = static_cast<int>(T / kBM);
    // N tiles over all F columns, across shard seams (no shard pads its last tile), when
    // every 32-column chunk of a tile lies in one shard's block of the saved activations:
    // always for GELU ([T][F] layouts), for SwiGLU ([T][2F], a gate and an up block a
    // shard) when Fs % 32 == 0
    p.flat_n = (!h->swiglu || Fs % 32 == 0) ? 1 : 0;
    p.raster_group = short_k_raster_group(h);
    p.tiles_per_shard = static_cast<int>(cdiv(Fs, kBN));
    p.num_n_tiles = static_cast<int>(p.flat_n ? cdiv(F, kBN) : t * p.tiles_per_shard);
    p.num_kb = static_cast<int>(cdiv(H, kBK));
    p.aux = static_cast<const __nv_bfloat16*>(Zsaved);
    p.out0 = dZ;
    p.out1 = recompute ? Asaved : nullptr;
    p.colsum = bias ? part1 : nullptr;
    st = run_gemm(h, h->swiglu ? GemmKind::DGRAD_SWIGLU : GemmKind::DGRAD_GELU, false, tdgA,
                  tdgB, p, s, h->swiglu ? "dgrad_swiglu" : "dgrad_gelu", 2.0 * T * F * H,
                  2.0 * (T * H + F * H + 2 * T * F1) + (recompute ? 2.0 * T * F : 0.0) +
                      (bias ? 4.0 * ws_db1_parts(h) * F : 0.0));
  }
  if (st == MLPB_OK && (cudaEventRecord(h->ev_dz, s) != cudaSuccess ||
                        cudaStreamWaitEvent(s2, h->ev_dz, 0) != cudaSuccess))
    st = MLPB_ECUDA;

  // ---- [s2] dW2_i^T = A_i^T dY  (M = F, N = H, K = T), written into dW2's layout; after
  // dgrad: with recomputation its epilogue rewrites A first, and without it the same order
  // (dW2 and dW1 beside dX, nothing beside dgrad) measured faster on the SwiGLU workloads
  if (st == MLPB_OK) {
    GemmParams p = base_params(h);
    p.M = static_cast<int>(F);
    p.num_m_tiles = static_cast<int>(cdiv(F, kBM));
    p.num_n_tiles = static_cast<int>(cdiv(H, kBN));
    p.num_kb = static_cast<int>(T / kBK);
    p.out0 = dW2;
    p.accumulate = acc;
    p.mn3d = mn3d_w2;
    st = run_gemm(h, GemmKind::WGRAD_W2T, false, tw2A, tw2B, p, s2, "wgrad_w2", 2.0 * H * F * T,
                  2.0 * (T * H + T * F) + 4.0 * (1 + acc) * H * F);
  }

  // ---- [s2] db1 = sum_t dZ and db2 = sum_t dY: the dgrad epilogue's per-warp column sums
  // and the transpose launch's per-range ones, each added in row order, in one launch
  if (st == MLPB_OK && bias) {
    const int np = static_cast<int>(ws_db1_parts(h));
    LaunchTimer lt(h, s2, "bias_sums", 0.0,
                   4.0 * np * F + 4.0 * splits2 * H + 4.0 * (1 + acc) * (F + H));
    cudaError_t e = launch_sum_partials_pair(part1, np, F, db1, part2, splits2, H, db2, s2, acc);
    lt.done();
    st = from_cuda(e);
  }

  // ---- [s2] dW1 = dZ^T X  (M = F1, N = H, K = T)
  if (st == MLPB_OK) {
    GemmParams p = base_params(h);
    p.M = static_cast<int>(F1);
    p.num_m_tiles = static_cast<int>(cdiv(F1, kBM));
    p.num_n_tiles = static_cast<int>(cdiv(H, kBN));
    p.num_kb = static_cast<int>(T / kBK);
    p.out0 = dW1;
    p.accumulate = acc;
    p.mn3d = mn3d_w1;
    plan_tail_split(h, p, ws_split_partial(h, workspace, 1));  // the last GEMM of the step
    st = run_gemm(h, GemmKind::WGRAD_W1, false, tw1A, tw1B, p, s2, "wgrad_w1", 2.0 * F1 * H * T,
                  2.0 * (T * F1 + T * H) + 4.0 * (1 + acc) * F1 * H);
  }

  // ---- [s] dX = sum_i dZ_i W1_i  (f backward: the sum over shards is the K loop)
  if (st == MLPB_OK) {
    GemmParams p = base_params(h);
    p.M = static_cast<int>(T);
    p.num_m_tiles = static_cast<int>(T / kBM);
    p.num_n_tiles = static_cast<int>(cdiv(H, kBN));
    p.num_kb = static_cast<int>(cdiv(F1, kBK));
    p.out0 = dX;
    p.out_bf16 = h->bf16_out ? 1 : 0;
    p.mn3d = mn3d_dx;
    plan_tail_split(h, p, ws_split_partial(h, workspace));
    st = run_gemm(h, GemmKind::DX, false, tdxA, tdxB, p, s, "dgrad_x", 2.0 * T * H * F1,
                  2.0 * (T * F1 + F1 * H) + (h->bf16_out ? 2.0 : 4.0) * T * H);
  }

  // Join: the caller's stream waits for s2 whatever happened above.
  if (cudaEventRecord(h->ev_join, s2) != cudaSuccess ||
      cudaStreamWaitEvent(s, h->ev_join, 0) != cudaSuccess)
    return MLPB_ECUDA;
  return st;
}

// The backward with E4M3 GEMMs, on the caller's stream.  Every amax first (they only
// read); then each GEMM's E4M3 operands are written right before it, so that the GEMM
// finds them in L2: dY (both ways) and W2 (transposed), dgrad (records amax(dZ)), db2;
// dZ (both ways) and W1 (transposed), dX; A (transposed), dW2, db1; X (transposed), dW1.
// (Casting beside the GEMMs on a second stream, like the bf16 backward's schedule,
// measured 1-2 % slower: a persistent GEMM CTA holds 225 KB of shared memory, so the
// casts cannot share its SMs.)
static mlpb_status backward_f8(mlpb_handle* h, const void* X, const void* W1, const void* W2,
                               const void* Zsaved, const void* Asaved, const void* dY,
                               void* dX, float* dW1, float* dW2, float* db1, float* db2,
                               void* workspace, cudaStream_t s) {
  const bool bias = h->cfg.has_bias != 0;
  const int64_t T = h->T, H = h->H, F = h->F, Fs = h->Fs, t = h->t, F1 = h->F1;
  const int acc = h->accumulate ? 1 : 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* dZ = ws;
  float* part1 = reinterpret_cast<float*>(ws + ws_dz_bytes(h));  // db1 partials [T/32][F]
  const F8Layout L = f8_layout(h, workspace);
  uint32_t* am = L.amax;

  // tensor maps first: an encoding error launches nothing
  CUtensorMap tdA, tdB, txA, txB, tw2A, tw2B, tw1A, tw1B;
  if (!map_u8(&tdA, L.dYq, H, T) || !map_u8_sharded(&tdB, L.W2t, H, Fs, t, H, Fs * H) ||
      !map_u8(&txA, L.dZq, F1, T) || !map_u8(&txB, L.W1t, F1, H) ||
      !map_u8(&tw2A, L.dYt, T, H) || !map_u8_sharded(&tw2B, L.At, T, Fs, t, T, Fs * T) ||
      !map_u8(&tw1A, L.dZt, T, F1) || !map_u8(&tw1B, L.Xt, T, H))
    return MLPB_EINVAL;
  if (cudaMemsetAsync(am, 0, kAmaxWords * sizeof(uint32_t), s) != cudaSuccess)
    return MLPB_ECUDA;

  mlpb_status st = f8_amax(h, dY, T * H, am + kAmaxDY, s, "fp8_amax_dy");
  if (st == MLPB_OK) st = f8_amax(h, W2, F * H, am + kAmaxW2, s, "fp8_amax_w2");
  if (st == MLPB_OK) st = f8_amax(h, X, T * H, am + kAmaxX, s, "fp8_amax_x");
  if (st == MLPB_OK) st = f8_amax(h, W1, F1 * H, am + kAmaxW1, s, "fp8_amax_w1");
  if (st == MLPB_OK) st = f8_amax(h, Asaved, T * F, am + kAmaxA, s, "fp8_amax_a");

  // ---- dgrad of fc2 with the fused activation derivative: dZ [T][F1] bf16
  if (st == MLPB_OK)
    st = f8_cast(h, dY, 1, T, H, L.dYq, L.dYt, am + kAmaxDY, s, "fp8_cast_dy");
  if (st == MLPB_OK)
    st = f8_cast(h, W2, static_cast<int>(t), H, Fs, nullptr, L.W2t, am + kAmaxW2, s,
                 "fp8_cast_w2t");
  if (st == MLPB_OK) {
    GemmParams p = base_params(h);
    p.M = static_cast<int>(T);
    p.num_m_tiles = static_cast<int>(T / kBM);
    p.tiles_per_shard = static_cast<int>(cdiv(Fs, kBN));
    p.num_n_tiles = static_cast<int>(t * p.tiles_per_shard);
    p.num_kb = static_cast<int>(cdiv(H, kBK8));
    p.aux = static_cast<const __nv_bfloat16*>(Zsaved);
    p.out0 = dZ;
    p.amax_a = am + kAmaxDY;
    p.amax_b = am + kAmaxW2;
    p.amax_out = am + kAmaxDZ;
    p.colsum = bias ? part1 : nullptr;
    st = run_gemm_f8(h, h->swiglu ? GemmKind::DGRAD_SWIGLU : GemmKind::DGRAD_GELU, tdA, tdB,
                     p, s, h->swiglu ? "dgrad_swiglu_f8" : "dgrad_gelu_f8", 2.0 * T * F * H,
                     1.0 * (T * H + F * H) + 4.0 * T * F1 +
                         (bias ? 4.0 * ws_db1_parts(h) * F : 0.0));
  }
  // db2 = sum_t dY on the bf16 dY: the bf16 path's first pass (column sums over row
  // ranges, without the W2 transpose it shares a launch with there), so that both paths
  // give the same bits; the ranges are added with db1's partials below
  float* part2 = reinterpret_cast<float*>(ws + ws_db2_offset(h));
  const int splits2 = db2_splits(h);
  if (st == MLPB_OK && bias) {
    LaunchTimer lt(h, s, "colsum_db2", 0.0, 2.0 * T * H + 4.0 * splits2 * H);
    cudaError_t e = launch_transpose_w2(nullptr, nullptr, static_cast<int>(t), H, Fs, dY, T,
                                        splits2, part2, s);
    lt.done();
    st = from_cuda(e);
  }
  // ---- dX = sum_i dZ_i W1_i (f backward: the K loop runs over every shard's rows)
  if (st == MLPB_OK)
    st = f8_cast(h, dZ, 1, T, F1, L.dZq, L.dZt, am + kAmaxDZ, s, "fp8_cast_dz");
  if (st == MLPB_OK)
    st = f8_cast(h, W1, 1, F1, H, nullptr, L.W1t, am + kAmaxW1, s, "fp8_cast_w1t");
  if (st == MLPB_OK) {
    GemmParams p = base_params(h);
    p.M = static_cast<int>(T);
    p.num_m_tiles = static_cast<int>(T / kBM);
    p.num_n_tiles = static_cast<int>(cdiv(H, kBN));
    p.num_kb = static_cast<int>(cdiv(F1, kBK8));
    p.out0 = dX;
    p.out_bf16 = h->bf16_out ? 1 : 0;
    p.amax_a = am + kAmaxDZ;
    p.amax_b = am + kAmaxW1;
    st = run_gemm_f8(h, GemmKind::DX, txA, txB, p, s, "dgrad_x_f8", 2.0 * T * H * F1,
                     1.0 * (T * F1 + F1 * H) + (h->bf16_out ? 2.0 : 4.0) * T * H);
  }
  // ---- dW2_i = dY^T A_i  (M = H, N = F by shard, K = T)
  if (st == MLPB_OK)
    st = f8_cast(h, Asaved, 1, T, F, nullptr, L.At, am + kAmaxA, s, "fp8_cast_at");
  if (st == MLPB_OK) {
    GemmParams p = base_params(h);
    p.M = static_cast<int>(H);
    p.num_m_tiles = static_cast<int>(cdiv(H, kBM));
    p.tiles_per_shard = static_cast<int>(cdiv(Fs, kBN));
    p.num_n_tiles = static_cast<int>(t * p.tiles_per_shard);
    p.num_kb = static_cast<int>(T / kBK8);
    p.out0 = dW2;
    p.accumulate = acc;
    p.amax_a = am + kAmaxDY;
    p.amax_b = am + kAmaxA;
    st = run_gemm_f8(h, GemmKind::WGRAD_W2, tw2A, tw2B, p, s, "wgrad_w2_f8", 2.0 * H * F * T,
                     1.0 * (T * H + T * F) + 4.0 * (1 + acc) * H * F);
  }
  if (st == MLPB_OK && bias) {  // db1 and db2: the column partial sums, added in row order
    const int np = static_cast<int>(ws_db1_parts(h));
    LaunchTimer lt(h, s, "bias_sums", 0.0,
                   4.0 * np * F + 4.0 * splits2 * H + 4.0 * (1 + acc) * (F + H));
    cudaError_t e = launch_sum_partials_pair(part1, np, F, db1, part2, splits2, H, db2, s, acc);
    lt.done();
    st = from_cuda(e);
  }
  // ---- dW1 = dZ^T X  (M = F1, N = H, K = T)
  if (st == MLPB_OK) st = f8_cast(h, X, 1, T, H, nullptr, L.Xt, am + kAmaxX, s, "fp8_cast_xt");
  if (st == MLPB_OK) {
    GemmParams p = base_params(h);
    p.M = static_cast<int>(F1);
    p.num_m_tiles = static_cast<int>(cdiv(F1, kBM));
    p.num_n_tiles = static_cast<int>(cdiv(H, kBN));
    p.num_kb = static_cast<int>(T / kBK8);
    p.out0 = dW1;
    p.accumulate = acc;
    p.amax_a = am + kAmaxDZ;
    p.amax_b = am + kAmaxX;
    st = run_gemm_f8(h, GemmKind::WGRAD_W1, tw1A, tw1B, p, s, "wgrad_w1_f8", 2.0 * F1 * H * T,
                     1.0 * (T * F1 + T * H) + 4.0 * (1 + acc) * F1 * H);
  }
  return st;
}

mlpb_status mlpb_layernorm_sp_fwd(mlpb_handle* h, const void* X, const void* gamma,
                                  const void* beta, void* Xn, float* mean, float* rstd,
                                  mlpb_stream_t stream) {
  if (h == nullptr || !gamma || !beta) return MLPB_EINVAL;
  if (h->T > 0 && (!X || !Xn || !mean || !rstd)) return MLPB_EINVAL;  // T = 0: empty rows
  if (!h->cfg.seq_parallel_ln) return MLPB_EUNSUPPORTED;
  for (const void* p : {X, gamma, beta, static_cast<const void*>(Xn)})
    if (p && !aligned16(p)) return MLPB_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t T = h->T, H = h->H;
  if (T == 0) return MLPB_OK;
  LaunchTimer lt(h, s, "ln_fwd", 0.0, 4.0 * T * H + 8.0 * T + 4.0 * H);
  cudaError_t e = launch_ln_fwd(X, gamma, beta, Xn, mean, rstd, T, H, h->cfg.ln_eps,
                                h->num_sms, h->d_err, h->wait_ns, s);
  lt.done();
  return from_cuda(e);
}

mlpb_status mlpb_layernorm_sp_bwd(mlpb_handle* h, const void* X, const void* gamma,
                                  const float* mean, const float* rstd, const void* dXn,
                                  void* dX, float* dgamma, float* dbeta, void* workspace,
                                  mlpb_stream_t stream) {
  if (h == nullptr || !gamma || !dgamma || !dbeta) return MLPB_EINVAL;
  if (h->T > 0 && (!X || !mean || !rstd || !dXn || !dX || !workspace))
    return MLPB_EINVAL;  // T = 0: the row tensors are empty
  if (!h->cfg.seq_parallel_ln) return MLPB_EUNSUPPORTED;
  for (const void* p : {X, gamma, static_cast<const void*>(dXn), static_cast<const void*>(dX),
                        static_cast<const void*>(workspace)})
    if (p && !aligned16(p)) return MLPB_EINVAL;
  return ln_bwd_impl(h, X, gamma, mean, rstd, dXn, nullptr, dX, dgamma, dbeta, workspace,
                     reinterpret_cast<cudaStream_t>(stream));
}

// LayerNorm backward of validated arguments; `dres` (bf16 [T][H] or NULL) is added to dX.
static mlpb_status ln_bwd_impl(mlpb_handle* h, const void* X, const void* gamma,
                               const float* mean, const float* rstd, const void* dXn,
                               const void* dres, void* dX, float* dgamma, float* dbeta,
                               void* workspace, cudaStream_t s) {
  const int64_t T = h->T, H = h->H;
  const int nblk = h->t * h->ln_blocks_per_shard;
  float* pg = static_cast<float*>(workspace);
  float* pb = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                       align256(static_cast<size_t>(nblk) * H * 4));
  const int acc = h->accumulate ? 1 : 0;
  if (T == 0) {  // no rows: zero parameter gradients (adds nothing when accumulating)
    if (acc) return MLPB_OK;
    cudaError_t e = launch_fill_zero(dgamma, static_cast<size_t>(H * 4), s);
    if (e == cudaSuccess) e = launch_fill_zero(dbeta, static_cast<size_t>(H * 4), s);
    return from_cuda(e);
  }
  const double gb = h->bf16_out ? 2.0 : 4.0;  // bytes of a dXn / dX element
  LaunchTimer lt(h, s, "ln_bwd", 0.0,
                 (2.0 + 2.0 * gb + (dres ? 2.0 : 0.0)) * T * H + 8.0 * T + 10.0 * H);
  cudaError_t e = launch_ln_bwd(X, gamma, mean, rstd, dXn, dres, dX, h->bf16_out, pg, pb, T, H,
                                h->t, h->ln_blocks_per_shard, h->d_err, h->wait_ns, s);
  lt.done();
  if (e == cudaSuccess) {
    LaunchTimer lt2(h, s, "ln_bwd_param_reduce", 0.0, 8.0 * nblk * H + 8.0 * (1 + acc) * H, 1);
    e = launch_sum_partials2(pg, pb, nblk, H, dgamma, dbeta, s, acc);
    lt2.done();
  }
  return from_cuda(e);
}

mlpb_status mlpb_branch_forward(mlpb_handle* h, const void* X, const void* gamma,
                                const void* beta, const void* W1, const void* b1,
                                const void* W2, const void* b2, void* Y, void* Xn, float* mean,
                                float* rstd, void* Zsaved, void* Asaved, void* workspace,
                                mlpb_stream_t stream) {
  if (h == nullptr) return MLPB_EINVAL;
  const bool bias = h->cfg.has_bias != 0;
  if (!gamma || !beta || !W1 || !W2) return MLPB_EINVAL;
  if (h->T > 0 && (!X || !Xn || !mean || !rstd || !Y || !Zsaved || !Asaved)) return MLPB_EINVAL;
  if (bias != (b1 != nullptr) || bias != (b2 != nullptr)) return MLPB_EINVAL;
  if (!h->cfg.seq_parallel_ln) return MLPB_EUNSUPPORTED;
  for (const void* p : {X, gamma, beta, static_cast<const void*>(Xn), W1, W2,
                        static_cast<const void*>(Y), static_cast<const void*>(Zsaved),
                        static_cast<const void*>(Asaved), b1, b2})
    if (p && !aligned16(p)) return MLPB_EINVAL;
  if (h->T > 0 && (h->fp8 || h->emulate) && (!workspace || !aligned16(workspace)))
    return MLPB_EINVAL;
  if (h->T == 0) return MLPB_OK;
  mlpb_status st = mlpb_layernorm_sp_fwd(h, X, gamma, beta, Xn, mean, rstd, stream);
  if (st != MLPB_OK) return st;
  return forward_impl(h, Xn, W1, b1, W2, b2, Y, Zsaved, Asaved, X, workspace,
                      reinterpret_cast<cudaStream_t>(stream));
}

mlpb_status mlpb_branch_backward(mlpb_handle* h, const void* X, const void* gamma,
                                 const void* W1, const void* W2, const void* Xn,
                                 const float* mean, const float* rstd, const void* Zsaved,
                                 void* Asaved, const void* dY, void* dX, float* dW1,
                                 float* dW2, float* db1, float* db2, float* dgamma, float* dbeta,
                                 void* workspace, mlpb_stream_t stream) {
  if (h == nullptr) return MLPB_EINVAL;
  if (!h->cfg.seq_parallel_ln) return MLPB_EUNSUPPORTED;
  if (!gamma || !dgamma || !dbeta) return MLPB_EINVAL;
  if (h->T > 0 && (!X || !Xn || !mean || !rstd)) return MLPB_EINVAL;
  for (const void* p : {X, gamma})
    if (p && !aligned16(p)) return MLPB_EINVAL;
  // The MLP backward on the normalised input writes dXn into dX; the LayerNorm backward
  // then rewrites dX in place, row by row, as dY + LN'(dXn).  The parameter reductions of
  // both steps share the workspace one after the other (the first step's side stream has
  // joined the caller's stream when mlpb_backward returns).
  mlpb_status st = mlpb_backward(h, Xn, W1, W2, Zsaved, Asaved, dY, dX, dW1, dW2, db1, db2,
                                 workspace, stream);
  if (st != MLPB_OK) return st;
  return ln_bwd_impl(h, X, gamma, mean, rstd, dX, dY, dX, dgamma, dbeta, workspace,
                     reinterpret_cast<cudaStream_t>(stream));
}

mlpb_status mlpb_last_device_error(mlpb_handle* h, mlpb_stream_t stream) {
  if (h == nullptr) return MLPB_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLPB_ECUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, h->d_err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLPB_ECUDA;
  if (v != 0) {
    if (cudaMemset(h->d_err, 0, sizeof(uint32_t)) != cudaSuccess) return MLPB_ECUDA;
    return MLPB_ETIMEOUT;
  }
  return MLPB_OK;
}

mlpb_status mlpb_enable_timing(mlpb_handle* h, int enable) {
  if (h == nullptr) return MLPB_EINVAL;
  h->timing = enable != 0;
  return MLPB_OK;
}

mlpb_status mlpb_read_timings(mlpb_handle* h, mlpb_kernel_time* out, int capacity, int* count) {
  if (h == nullptr || count == nullptr || (capacity > 0 && out == nullptr)) return MLPB_EINVAL;
  int n = 0;
  mlpb_status st = MLPB_OK;
  for (auto& l : h->launches) {
    float ms = 0.f;
    if (cudaEventSynchronize(l.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, l.start, l.stop) != cudaSuccess)
      st = MLPB_ECUDA;
    if (n < capacity) {
      std::memcpy(out[n].name, l.name, sizeof(out[n].name));
      out[n].ms = ms;
      out[n].flops = l.flops;
      out[n].bytes = l.bytes;
      out[n].kernels = l.kernels;
      ++n;
    }
    h->event_pool.push_back(l.start);
    h->event_pool.push_back(l.stop);
  }
  h->launches.clear();
  *count = n;
  return st;
}

}  // extern "C"
