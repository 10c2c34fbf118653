// Persistent, warp-specialised tcgen05 GEMM for the MLP block's six contractions, run by
// CTA pairs (clusters of two CTAs on two SMs, tcgen05 cta_group::2).
//
// A pair computes a 256 x 256 output tile: M = 256 rows, 128 in each CTA's A tile and TMEM
// lanes; N = 256 columns, with each CTA's shared memory holding one 128-row half of the B
// tile, so every B byte in shared memory feeds both SMs' tensor cores.  Each CTA (192
// threads) has:
//   warp 0      TMA producer: a 7-stage ring of 128x64 A and 128x64 B-half bf16 tiles
//               (128-byte swizzle, 32 KB a stage).  Both CTAs' copies of a stage signal
//               the even CTA's full barrier (the odd CTA's through .cta_group::2), which
//               the even CTA's producer arms with both halves' byte count;
//   warp 1      with its peer, allocates 512 TMEM columns (two 256-column fp32
//               accumulators); in the even CTA it waits on that one barrier, issues the
//               pair's tcgen05.mma (M=256, N=256, K=16) and commits each consumed stage to
//               both CTAs' producers;
//   warps 2..5  epilogue: tcgen05.ld of this CTA's 128 accumulator rows (each warp owns the
//               32 TMEM lanes of its warp-id modulo 4), the fused pointwise op, stores to
//               HBM, then the accumulator is released to the even CTA's MMA issuer.
// Every wait is bounded (common.cuh): a wait that expires raises the CTA's abort flag
// and the device error word; all roles then drain what they issued and free TMEM.
//
// Pairs walk work units round robin: whole tiles, grouped 8 M-tile pairs at a time over
// all N tiles, and -- when the host asks for a tail split (FC2, DX, WGRAD_W1) -- the tiles of the
// last, partly filled wave cut into K-ranges whose raw partial sums go to a workspace for
// a fixup kernel (gemm_fwd.cu) to add up in a fixed order.
//
// The F8 instantiation runs the same pipeline on E4M3 operands (tcgen05 kind::f8f6f4, K = 32
// a call, 128-byte = 128-element K-major rows, every operand K-major from its own or its
// transposed E4M3 copy) and rescales each accumulator by 2^-(k_a + k_b) in the epilogue;
// FC1 and DGRAD also record the amax of the bf16 A / dZ they write.
//
// The contractions (T tokens, H hidden, F ffn, t shards, Fs = F/t, F1 = F or 2F):
//   FC1_GELU      Z = X W1^T + b1, A = gelu(Z)       M=T  N=F      K=H   A,B K-major
//   FC1_SWIGLU    [G|U] = X [Wg_i|Wu_i]^T, A = silu(G)U  (per shard i, 128 gate + 128 up
//                 columns per tile: the even CTA holds the gate rows, the odd the up rows)
//   FC2           Y = sum_i A_i W2_i^T + b2 (+ R)     M=T  N=H      K=t x Fs (walks shards)
//   DGRAD_GELU    dZ = (dY W2) * gelu'(Z)             M=T  N=F      K=H   B = W2's
//                 per-shard transpose [F][H] (K-major; a copy the backward makes first)
//   DGRAD_SWIGLU  dG = dA U silu'(G), dU = dA silu(G) M=T  N=F      K=H   B as DGRAD_GELU
//                 (both may also rewrite A = act(saved Z) for dW2: recomputation)
//   DX            dX = sum_i dZ_i W1_i                M=T  N=H      K=F1  B MN-major
//   WGRAD_W2T     dW2_i^T = A_i^T dY                  M=F  N=H      K=T   A,B MN-major
//                 (written into dW2's [t][H][Fs] layout: for each column h the 32 rows of
//                 a warp store 32 consecutive floats of one dW2 row)
//   WGRAD_W1      dW1 = dZ^T X                        M=F1 N=H      K=T   A,B MN-major
//   WGRAD_W2      dW2_i = dY^T A_i                    M=H  N=F      K=T   (E4M3 path only:
//                 both operands K-major copies; the bf16 path computes the transpose, which
//                 measured 11-20 % faster than this shape with MN-major operands)
#pragma once

#include "common.cuh"
#include "fp8.cuh"
#include "gemm_params.h"

namespace mlpb {

template <GemmKind K>
struct KindOf {
  // long K (F, F1 or T): a pair's whole tiles alternate the direction of their K loop
  static constexpr bool reverse_k = (K == GemmKind::FC2 || K == GemmKind::DX ||
                                     K == GemmKind::WGRAD_W1 || K == GemmKind::WGRAD_W2T ||
                                     K == GemmKind::WGRAD_W2);
  static constexpr bool a_mn = (K == GemmKind::WGRAD_W1 || K == GemmKind::WGRAD_W2T);
  static constexpr bool b_mn = (K == GemmKind::DX || K == GemmKind::WGRAD_W1 ||
                                K == GemmKind::WGRAD_W2T);
};

// Grouped rasterisation: `group` consecutive M tiles (or M-tile pairs; 0: 8) sweep all N
// tiles together, so that the B panels they share stay in L2 while the group's A panels
// are read once.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group, int& mt,
                                            int& nt) {
  const int G = group > 0 ? group : 8;
  const int span = G * num_n;
  const int g = tile / span;
  const int m0 = g * G;
  const int gm = min(num_m - m0, G);
  const int r = tile - g * span;
  mt = m0 + r % gm;
  nt = r / gm;
}

// Work unit u of a launch: a whole pair tile (part = -1) or, past split_start, one of the
// `split` K-ranges of a tail tile.
__device__ __forceinline__ void unit_range(int u, int split, int split_start, int num_kb, int& st,
                                           int& kb0, int& kb1, int& part) {
  if (u < split_start) {
    st = u;
    kb0 = 0;
    kb1 = num_kb;
    part = -1;
    return;
  }
  const int j = u - split_start;
  st = split_start + j / split;
  part = j - (j / split) * split;
  kb0 = num_kb * part / split;
  kb1 = num_kb * (part + 1) / split;
}

// ------------------------------------------------------------------ pointwise math
// tanh-form GELU written with s = sigmoid(2u), u = sqrt(2/pi) (z + 0.044715 z^3): since
// 1 + tanh(u) = 2 sigmoid(2u), gelu(z) = z s, the same function without cancellation for
// z << 0, and gelu'(z) = s + z s (1 - s) 2 sqrt(2/pi) (1 + 3 * 0.044715 z^2).  The
// constants are folded so that e^{-2u} = 2^{z (a + b z^2)} is one base-2 exponential:
//   a = -2k log2(e), b = -2k c log2(e),  k = sqrt(2/pi), c = 0.044715.
// For |z| past ~10 the exponential overflows to +inf (s = 0) or underflows to 0 (s = 1),
// and both forms then return their limits (0 and z; 0 and 1) with no inf * 0.
constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kGeluCubic = 0.044715f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kGeluA = -2.0f * kSqrt2OverPi * kLog2e;               // -2k log2(e)
constexpr float kGeluB = -2.0f * kSqrt2OverPi * kGeluCubic * kLog2e;  // -2kc log2(e)
constexpr float kGeluD0 = 2.0f * kSqrt2OverPi;                        // 2k
constexpr float kGeluD2 = 6.0f * kSqrt2OverPi * kGeluCubic;           // 6kc

__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// 2^x (the MUFU base-2 exponential; subnormal results flush to zero).
__device__ __forceinline__ float ex2_f(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Two fp32 values in one 64-bit register (lo in the low half) and the f32x2 arithmetic
// of the sm_100 family: one instruction for both lanes, each rounded as its fp32 form.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// e^{-2u} + 1 for two values of z (one MUFU exponential each), and its reciprocal s.
__device__ __forceinline__ uint64_t gelu_s_x2(uint64_t z, uint64_t z2) {
  float u0, u1, d0, d1;
  f2_unpack(f2_mul(z, f2_fma(z2, f2_pack(kGeluB, kGeluB), f2_pack(kGeluA, kGeluA))), u0, u1);
  f2_unpack(f2_add(f2_pack(ex2_f(u0), ex2_f(u1)), f2_pack(1.0f, 1.0f)), d0, d1);
  return f2_pack(__fdividef(1.0f, d0), __fdividef(1.0f, d1));
}

// gelu(z) = z s for two values.
__device__ __forceinline__ uint64_t gelu_x2(uint64_t z) { return f2_mul(z, gelu_s_x2(z, f2_mul(z, z))); }

// gelu'(z) = s + d s (1 - s), d = 2k z (1 + 3c z^2), for two values.
__device__ __forceinline__ uint64_t gelu_grad_x2(uint64_t z) {
  const uint64_t z2 = f2_mul(z, z);
  const uint64_t s = gelu_s_x2(z, z2);
  const uint64_t d = f2_mul(z, f2_fma(z2, f2_pack(kGeluD2, kGeluD2), f2_pack(kGeluD0, kGeluD0)));
  return f2_fma(d, f2_sub(s, f2_mul(s, s)), s);
}

// v[e] = gelu(v[e]) over 32 values, two at a time.
__device__ __forceinline__ void gelu_x32(float (&v)[32]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) f2_unpack(gelu_x2(f2_pack(v[e], v[e + 1])), v[e], v[e + 1]);
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* p, int nvalid, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u = make_uint4(0, 0, 0, 0);
    if (q * 8 < nvalid) u = ld_global_nc_v4(p + q * 8);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16x2(w[e]);
      v[q * 8 + 2 * e] = f.x;
      v[q * 8 + 2 * e + 1] = f.y;
    }
  }
}

// 32 values rounded to bf16 (nearest, ties to even), two to a word: w[e] = (v[2e], v[2e+1]).
__device__ __forceinline__ void pack_bf16x32(const float (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
}

__device__ __forceinline__ void store_packed_bf16x32(__nv_bfloat16* p, int nvalid,
                                                     const uint32_t (&w)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (q * 8 < nvalid)
      st_global_v4(p + q * 8, make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* p, int nvalid, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q * 8 < nvalid) {
      uint4 u;
      u.x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
      u.y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
      u.z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
      u.w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
      st_global_v4(p + q * 8, u);
    }
  }
}

__device__ __forceinline__ void store_f32x32(float* p, int nvalid, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q * 4 < nvalid) {
      uint4 u = make_uint4(__float_as_uint(v[q * 4 + 0]), __float_as_uint(v[q * 4 + 1]),
                           __float_as_uint(v[q * 4 + 2]), __float_as_uint(v[q * 4 + 3]));
      st_global_v4(p + q * 4, u);
    }
  }
}

// v += the nvalid (a multiple of 4) fp32 values at p (read-modify-write accumulation).
__device__ __forceinline__ void add_f32x32(const float* p, int nvalid, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q * 4 < nvalid) {
      const float4 o = __ldcg(reinterpret_cast<const float4*>(p + q * 4));
      v[q * 4 + 0] += o.x;
      v[q * 4 + 1] += o.y;
      v[q * 4 + 2] += o.z;
      v[q * 4 + 3] += o.w;
    }
  }
}

// Column sums over a warp's 32 rows: on entry lane l holds v[0..32) of its own row, on
// exit it returns the sum over the 32 lanes of column l.  Each of five exchange rounds
// halves the columns a lane keeps (16 + 8 + 4 + 2 + 1 shuffles); the order of the adds is
// fixed, so the sums are reproducible.  v is overwritten.
__device__ __forceinline__ float warp_column_sums(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = upper ? v[j] : v[j + w];
      const float keep = upper ? v[j + w] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

__device__ __forceinline__ void tmem_load_f32x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
}

// One 32-column accumulator chunk; FP8 sums are rescaled by 2^-(k_a + k_b) (sc, exact).
template <bool F8>
__device__ __forceinline__ void load_acc(uint32_t taddr, float (&v)[32], float sc) {
  tmem_load_f32x32(taddr, v);
  if constexpr (F8) {
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] *= sc;
  }
}

// am = max(am, |v[e]|) over the chunk's valid columns (FP8: amax of a written operand).
__device__ __forceinline__ void track_amax(const float (&v)[32], int nv, float& am) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (e < nv) am = fmaxf(am, fabsf(v[e]));
}

// Epilogue of one 128 x 256 tile for the calling thread's row.  `tacc` is the TMEM
// address of the accumulator at this warp's lane quarter.  All branches that skip
// tcgen05.ld are uniform across the warp.
template <GemmKind K, bool F8 = false>
__device__ __forceinline__ void epilogue_tile(uint32_t tacc, int row, int mt, int nt,
                                              const GemmParams& p, float sc, float& am) {
  const int m = mt * kBM + row;
  const bool row_ok = m < p.M;
  if constexpr (K == GemmKind::FC1_GELU) {
    const int n0 = nt * kBN;
    __nv_bfloat16* Z = static_cast<__nv_bfloat16*>(p.out0) + static_cast<size_t>(m) * p.F;
    __nv_bfloat16* A = static_cast<__nv_bfloat16*>(p.out1) + static_cast<size_t>(m) * p.F;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int col = n0 + c * 32;
      if (col >= p.F) break;
      float v[32];
      load_acc<F8>(tacc + c * 32, v, sc);
      const int nv = min(32, p.F - col);
      if (p.bias != nullptr) {
        float b[32];
        load_bf16x32(p.bias + col, nv, b);
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          f2_unpack(f2_add(f2_pack(v[e], v[e + 1]), f2_pack(b[e], b[e + 1])), v[e], v[e + 1]);
      }
      if (row_ok) store_bf16x32(Z + col, nv, v);
      gelu_x32(v);
      if (row_ok) {
        store_bf16x32(A + col, nv, v);
        if constexpr (F8) track_amax(v, nv, am);
      }
    }
  } else if constexpr (K == GemmKind::FC1_SWIGLU) {
    const int i = nt / p.tiles_per_shard;
    const int j0 = (nt - i * p.tiles_per_shard) * 128;
    __nv_bfloat16* GU = static_cast<__nv_bfloat16*>(p.out0) + static_cast<size_t>(m) * 2 * p.F +
                        static_cast<size_t>(i) * 2 * p.Fs;
    __nv_bfloat16* A = static_cast<__nv_bfloat16*>(p.out1) + static_cast<size_t>(m) * p.F +
                       static_cast<size_t>(i) * p.Fs;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int jc = j0 + c * 32;
      if (jc >= p.Fs) break;
      float g[32], u[32];
      load_acc<F8>(tacc + c * 32, g, sc);
      load_acc<F8>(tacc + 128 + c * 32, u, sc);
      const int nv = min(32, p.Fs - jc);
      if (row_ok) {
        store_bf16x32(GU + jc, nv, g);
        store_bf16x32(GU + p.Fs + jc, nv, u);
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) u[e] *= g[e] * sigmoid_f(g[e]);
      if (row_ok) {
        store_bf16x32(A + jc, nv, u);
        if constexpr (F8) track_amax(u, nv, am);
      }
    }
  } else if constexpr (K == GemmKind::FC2 || K == GemmKind::DX) {
    const int n0 = nt * kBN;
    const size_t yo = static_cast<size_t>(m) * p.H;  // row m of Y (fp32, or bf16 with out_bf16)
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int col = n0 + c * 32;
      if (col >= p.H) break;
      float v[32];
      load_acc<F8>(tacc + c * 32, v, sc);
      const int nv = min(32, p.H - col);
      if (K == GemmKind::FC2 && p.bias != nullptr) {
        float b[32];
        load_bf16x32(p.bias + col, nv, b);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] += b[e];
      }
      if (K == GemmKind::FC2 && p.aux != nullptr && row_ok) {  // residual, added after b2
        float r[32];
        load_bf16x32(p.aux + static_cast<size_t>(m) * p.H + col, nv, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] += r[e];
      }
      if (row_ok) {
        if (p.out_bf16)
          store_bf16x32(static_cast<__nv_bfloat16*>(p.out0) + yo + col, nv, v);
        else
          store_f32x32(static_cast<float*>(p.out0) + yo + col, nv, v);
      }
    }
  } else if constexpr (K == GemmKind::DGRAD_GELU || K == GemmKind::DGRAD_SWIGLU) {
    // The tile's dA columns f0.. (global indices into F) end at f_end: all of F when the N
    // tiles run across shard seams, else shard i's end.
    int f0 = nt * kBN, f_end = p.F;
    if (!p.flat_n) {
      const int i = nt / p.tiles_per_shard;
      f0 = i * p.Fs + (nt - i * p.tiles_per_shard) * kBN;
      f_end = (i + 1) * p.Fs;
    }
    // recomputation: A [T][F] rewritten from the saved Z (or G, U), for the dW2 GEMM that
    // follows
    __nv_bfloat16* A = p.out1 ? static_cast<__nv_bfloat16*>(p.out1) + static_cast<size_t>(m) * p.F
                              : nullptr;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int f = f0 + c * 32;
      if (f >= f_end) break;
      const int nv = min(32, f_end - f);
      float v[32];
      load_acc<F8>(tacc + c * 32, v, sc);
      if constexpr (K == GemmKind::DGRAD_GELU) {
        const size_t o = static_cast<size_t>(m) * p.F + f;  // Z, dZ [T][F]
        uint32_t w[16];  // the stored bf16 dZ, two to a word
        if (row_ok) {
          float z[32];
          load_bf16x32(p.aux + o, nv, z);
          if (A != nullptr) {
            float a[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = z[e];
            gelu_x32(a);
            store_bf16x32(A + f, nv, a);
          }
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            f2_unpack(f2_mul(f2_pack(v[e], v[e + 1]), gelu_grad_x2(f2_pack(z[e], z[e + 1]))),
                      v[e], v[e + 1]);
          pack_bf16x32(v, w);
          store_packed_bf16x32(static_cast<__nv_bfloat16*>(p.out0) + o, nv, w);
          if constexpr (F8) track_amax(v, nv, am);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = 0u;
        }
        if (p.colsum != nullptr) {  // db1 partials: column sums of the stored (bf16) dZ
#pragma unroll
          for (int e = 0; e < 16; ++e) {  // a bf16 is the high half of the float it equals
            v[2 * e] = __uint_as_float(w[e] << 16);
            v[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
          }
          const float cs = warp_column_sums(v);
          const int lane = threadIdx.x & 31;
          if (lane < nv) p.colsum[static_cast<size_t>(m >> 5) * p.F + f + lane] = cs;
        }
      } else if (row_ok) {
        // G|U, dG|dU [T][2F]: shard i's Fs gate columns, then its Fs up columns (the
        // chunk lies in one shard: Fs % 32 == 0 when tiles cross seams)
        const int i = f / p.Fs;
        const size_t o = static_cast<size_t>(m) * 2 * p.F + f + static_cast<size_t>(i) * p.Fs;
        float g[32], u[32];
        load_bf16x32(p.aux + o, nv, g);
        load_bf16x32(p.aux + o + p.Fs, nv, u);
        if (A != nullptr) {
          float a[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = u[e] * (g[e] * sigmoid_f(g[e]));
          store_bf16x32(A + f, nv, a);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float s = sigmoid_f(g[e]);
          const float dg = v[e] * u[e] * s * (1.0f + g[e] * (1.0f - s));
          u[e] = v[e] * g[e] * s;  // dU
          g[e] = dg;               // dG
        }
        __nv_bfloat16* dGU = static_cast<__nv_bfloat16*>(p.out0) + o;
        store_bf16x32(dGU, nv, g);
        store_bf16x32(dGU + p.Fs, nv, u);
        if constexpr (F8) {
          track_amax(g, nv, am);
          track_amax(u, nv, am);
        }
      }
    }
  } else if constexpr (K == GemmKind::WGRAD_W2) {
    const int i = nt / p.tiles_per_shard;
    const int j0 = (nt - i * p.tiles_per_shard) * kBN;
    float* dW = static_cast<float*>(p.out0) + (static_cast<size_t>(i) * p.H + m) * p.Fs;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int jc = j0 + c * 32;
      if (jc >= p.Fs) break;
      float v[32];
      load_acc<F8>(tacc + c * 32, v, sc);
      if (row_ok) {
        const int nv = min(32, p.Fs - jc);
        if (p.accumulate) add_f32x32(dW + jc, nv, v);
        store_f32x32(dW + jc, nv, v);
      }
    }
  } else if constexpr (K == GemmKind::WGRAD_W2T) {
    // row m is ffn feature f = i Fs + j of shard i; column h goes to dW2[i][h][j], so for
    // each h the warp's 32 rows write 32 consecutive floats of one dW2 row
    const int n0 = nt * kBN;
    const int i = row_ok ? m / p.Fs : 0;
    const int j = m - i * p.Fs;
    float* dW = static_cast<float*>(p.out0) + static_cast<size_t>(i) * p.H * p.Fs + j;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int col = n0 + c * 32;
      if (col >= p.H) break;
      float v[32];
      load_acc<F8>(tacc + c * 32, v, sc);
      if (row_ok) {
        const int nv = min(32, p.H - col);
        float* q = dW + static_cast<size_t>(col) * p.Fs;
        if (p.accumulate) {  // all 32 reads in flight before the first write
          float old[32];
#pragma unroll
          for (int e = 0; e < 32; ++e)
            old[e] = e < nv ? __ldcg(q + static_cast<size_t>(e) * p.Fs) : 0.0f;
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] += old[e];
        }
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e < nv) q[static_cast<size_t>(e) * p.Fs] = v[e];
      }
    }
  } else {  // WGRAD_W1
    const int n0 = nt * kBN;
    float* dW = static_cast<float*>(p.out0) + static_cast<size_t>(m) * p.H;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int col = n0 + c * 32;
      if (col >= p.H) break;
      float v[32];
      load_acc<F8>(tacc + c * 32, v, sc);
      if (row_ok) {
        const int nv = min(32, p.H - col);
        if (p.accumulate) add_f32x32(dW + col, nv, v);
        store_f32x32(dW + col, nv, v);
      }
    }
  }
}

// A stage's TMA loads land in the issuing CTA's shared memory.  The even CTA's signal its
// own full barrier; the odd CTA's (kPeer) signal the even CTA's, through .cta_group::2, so
// the pair's MMA issuer waits on one barrier for both halves of a stage.
template <bool kPeer>
__device__ __forceinline__ void ld2(uint32_t d, const CUtensorMap* m, uint32_t bar, int c0, int c1) {
  if constexpr (kPeer) tma_load_2d_pair(d, m, bar, c0, c1);
  else tma_load_2d(d, m, bar, c0, c1);
}

template <bool kPeer>
__device__ __forceinline__ void ld3(uint32_t d, const CUtensorMap* m, uint32_t bar, int c0, int c1,
                                    int c2) {
  if constexpr (kPeer) tma_load_3d_pair(d, m, bar, c0, c1, c2);
  else tma_load_3d(d, m, bar, c0, c1, c2);
}

template <bool kPeer>
__device__ __forceinline__ void ld4(uint32_t d, const CUtensorMap* m, uint32_t bar, int c0, int c1,
                                    int c2, int c3) {
  if constexpr (kPeer) tma_load_4d_pair(d, m, bar, c0, c1, c2, c3);
  else tma_load_4d(d, m, bar, c0, c1, c2, c3);
}

// The k-block a stage loads and, for FC2 (whose K loop walks the shards), its shard and
// its k-block within the shard; for the kinds whose N tiles lie in one shard, the tile's
// shard ts and its tile index tj within the shard.  The producer sets ts, tj once a tile
// and steps the rest with kb, so no stage divides.
struct KPos {
  int kb, sh, kr;
  int ts, tj;
};

template <GemmKind K>
__device__ __forceinline__ void step_kpos(KPos& kp, bool rev, const GemmParams& p) {
  if (rev) {
    --kp.kb;
    if constexpr (K == GemmKind::FC2) {
      if (--kp.kr < 0) {
        kp.kr = p.kb_per_shard - 1;
        --kp.sh;
      }
    }
  } else {
    ++kp.kb;
    if constexpr (K == GemmKind::FC2) {
      if (++kp.kr == p.kb_per_shard) {
        kp.kr = 0;
        ++kp.sh;
      }
    }
  }
}

// One stage of one CTA of the pair: its own 128 A rows, and its 128-row half of B (K-major:
// one box; MN-major: two 64-wide chunks, in one copy through a 3-D map when GemmParams.mn3d
// says so, else two).
// FP8: every operand is K-major (E4M3 copies, transposed where needed), one box each:
//   FC1  A Xq [T][H]            B W1q [F][H] / [t][2][Fs][H]
//   FC2  A Aq [T][t][Fs]        B W2q [t][H][Fs]             (K walks the shards)
//   DGRAD A dYq [T][H]          B W2t [t][Fs][H]
//   DX   A dZq [T][F1]          B W1t [H][F1]
//   WGRAD_W2 A dYt [H][T]       B At [t][Fs][T]
//   WGRAD_W1 A dZt [F1][T]      B Xt [H][T]
template <GemmKind K, bool kPeer>
__device__ __forceinline__ void issue_stage_f8(const CUtensorMap* tA, const CUtensorMap* tB,
                                               uint32_t sa, uint32_t sb, uint32_t bar, int mt,
                                               int nt, const KPos& kp, int rank,
                                               const GemmParams& p) {
  const int k0 = kp.kb * kBK8;
  const int nh = nt * kBN + 128 * rank;
  if constexpr (K == GemmKind::FC1_GELU || K == GemmKind::DX || K == GemmKind::WGRAD_W1) {
    ld2<kPeer>(sa, tA, bar, k0, mt * kBM);
    ld2<kPeer>(sb, tB, bar, k0, nh);
  } else if constexpr (K == GemmKind::FC1_SWIGLU) {
    ld2<kPeer>(sa, tA, bar, k0, mt * kBM);
    ld4<kPeer>(sb, tB, bar, k0, kp.tj * 128, rank, kp.ts);
  } else if constexpr (K == GemmKind::FC2) {
    const int j0 = kp.kr * kBK8;
    ld3<kPeer>(sa, tA, bar, j0, mt * kBM, kp.sh);
    ld3<kPeer>(sb, tB, bar, j0, nh, kp.sh);
  } else {  // DGRAD_*, WGRAD_W2: B rows are shard i's rows j0.. of a [t][Fs][K] operand
    ld2<kPeer>(sa, tA, bar, k0, mt * kBM);
    ld3<kPeer>(sb, tB, bar, k0, kp.tj * kBN + 128 * rank, kp.ts);
  }
}

template <GemmKind K, bool kPeer>
__device__ __forceinline__ void issue_stage_pair(const CUtensorMap* tA, const CUtensorMap* tB,
                                                 uint32_t sa, uint32_t sb, uint32_t bar, int mt,
                                                 int nt, const KPos& kp, int rank,
                                                 const GemmParams& p) {
  const int kb = kp.kb;
  static_assert(K != GemmKind::WGRAD_W2, "the bf16 dW2 is the transposed WGRAD_W2T");
  const int k0 = kb * kBK;
  const int nh = nt * kBN + 128 * rank;  // first B row (N index) of this CTA's half
  if constexpr (K == GemmKind::FC1_GELU) {
    ld2<kPeer>(sa, tA, bar, k0, mt * kBM);
    ld2<kPeer>(sb, tB, bar, k0, nh);
  } else if constexpr (K == GemmKind::FC1_SWIGLU) {
    // W1 as [2F][H]: shard i's gate rows (even CTA) or up rows (odd CTA) j0..
    ld2<kPeer>(sa, tA, bar, k0, mt * kBM);
    ld2<kPeer>(sb, tB, bar, k0, (2 * kp.ts + rank) * p.Fs + kp.tj * 128);
  } else if constexpr (K == GemmKind::FC2) {
    // K walks the shards: A [T][F] at shard i's columns, W2 as [tH][Fs] at shard i's rows
    const int i = kp.sh;
    const int j0 = kp.kr * kBK;
    ld2<kPeer>(sa, tA, bar, i * p.Fs + j0, mt * kBM);
    ld2<kPeer>(sb, tB, bar, j0, i * p.H + nh);
  } else if constexpr (K == GemmKind::DGRAD_GELU || K == GemmKind::DGRAD_SWIGLU) {
    // B = W2's transposed copy [F][H] (K-major): rows nh.. over all of F, or shard i's
    // rows j0..
    const int row = p.flat_n ? nh : kp.ts * p.Fs + kp.tj * kBN + 128 * rank;
    ld2<kPeer>(sa, tA, bar, k0, mt * kBM);
    ld2<kPeer>(sb, tB, bar, k0, row);
  } else if constexpr (K == GemmKind::DX) {
    ld2<kPeer>(sa, tA, bar, k0, mt * kBM);
    if (p.mn3d & 2) {
      ld3<kPeer>(sb, tB, bar, 0, k0, nh >> 6);
    } else {
#pragma unroll
      for (int q = 0; q < 2; ++q) ld2<kPeer>(sb + q * kChunk, tB, bar, nh + 64 * q, k0);
    }
  } else {  // WGRAD_W1, WGRAD_W2T
    if (p.mn3d & 1) {
      ld3<kPeer>(sa, tA, bar, 0, k0, (mt * kBM) >> 6);
    } else {
#pragma unroll
      for (int q = 0; q < 2; ++q) ld2<kPeer>(sa + q * kChunk, tA, bar, mt * kBM + 64 * q, k0);
    }
    if (p.mn3d & 2) {
      ld3<kPeer>(sb, tB, bar, 0, k0, nh >> 6);
    } else {
#pragma unroll
      for (int q = 0; q < 2; ++q) ld2<kPeer>(sb + q * kChunk, tB, bar, nh + 64 * q, k0);
    }
  }
}

template <GemmKind K, bool F8 = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  constexpr int S = kPairStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sA0 = base;
  const uint32_t sB0 = base + S * kPairAStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * kPairStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const uint32_t full0 = smem_u32(bars);            // even CTA: both CTAs' halves of stage s landed
  const uint32_t empty0 = smem_u32(bars + S);       // the pair's MMAs have read stage s
  const uint32_t tfull0 = smem_u32(bars + 2 * S);
  const uint32_t tempty0 = smem_u32(bars + 2 * S + 2);
  const uint32_t drain = smem_u32(bars + 2 * S + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int cid = blockIdx.x / 2;
  const int nclusters = gridDim.x / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);  // the even CTA's producer arms it for both halves
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 8);  // four epilogue warps in each CTA
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t full_lead = mapa_shared(full0, 0);
  const uint32_t tempty_lead = mapa_shared(tempty0, 0);

  const WaitCtx wc{abort_flag, p.err, p.wait_ns};
  const int num_pm = (p.num_m_tiles + 1) / 2;
  const int num_super = num_pm * p.num_n_tiles;
  const int split = p.split > 1 ? p.split : 1;
  const int split_start = split > 1 ? p.split_start : num_super;
  const int num_units = split_start + (num_super - split_start) * split;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;
      bool skip_once = p.fault_inject != 0 && cid == 0 && leader;
      int it = 0;
      for (int u = cid; u < num_units; u += nclusters, ++it) {
        int st, kb0, kb1, part;
        unit_range(u, split, split_start, p.num_kb, st, kb0, kb1, part);
        int mp, nt;
        tile_coords(st, num_pm, p.num_n_tiles, p.raster_group, mp, nt);
        const int mt = mp * 2 + rank;
        // long-K GEMMs: whole tiles of odd iterations walk K backwards.  The pair's next
        // tile shares an operand panel with this one (the grouped raster), and it starts
        // on the k-blocks just read, which are still in L2 (5-10 % less DRAM traffic)
        const bool rev = KindOf<K>::reverse_k && part < 0 && (it & 1) != 0;
        KPos kp{rev ? kb1 - 1 : kb0, 0, 0, 0, 0};
        if constexpr (K == GemmKind::FC2) {  // one division a tile; then stepped
          kp.sh = kp.kb / p.kb_per_shard;
          kp.kr = kp.kb - kp.sh * p.kb_per_shard;
        }
        if constexpr (K == GemmKind::FC1_SWIGLU || K == GemmKind::DGRAD_GELU ||
                      K == GemmKind::DGRAD_SWIGLU || K == GemmKind::WGRAD_W2) {
          kp.ts = nt / p.tiles_per_shard;
          kp.tj = nt - kp.ts * p.tiles_per_shard;
        }
        bool ok = true;
        for (int i = kb0; i < kb1; ++i) {
          if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, wc, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t sa = sA0 + stage * kPairAStage, sb = sB0 + stage * kPairBStage;
          if (skip_once) {
            skip_once = false;  // fault injection: this stage is never armed
          } else if (leader) {
            // one arrival with both CTAs' bytes; the odd CTA's copies may land first (the
            // barrier's transaction count goes below zero until this expect-tx)
            const uint32_t fb = full0 + 8 * stage;
            mbar_arrive_expect_tx(fb, 2 * kPairStageBytes);
            if constexpr (F8)
              issue_stage_f8<K, false>(&tmA, &tmB, sa, sb, fb, mt, nt, kp, rank, p);
            else
              issue_stage_pair<K, false>(&tmA, &tmB, sa, sb, fb, mt, nt, kp, rank, p);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          } else {
            const uint32_t fb = full_lead + 8 * stage;
            if constexpr (F8)
              issue_stage_f8<K, true>(&tmA, &tmB, sa, sb, fb, mt, nt, kp, rank, p);
            else
              issue_stage_pair<K, true>(&tmA, &tmB, sa, sb, fb, mt, nt, kp, rank, p);
            armed = 1u;  // issued copies that nothing in this CTA observes
          }
          step_kpos<K>(kp, rev, p);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (leader) {
        // every armed stage's bytes, the odd CTA's included, have landed
        for (int s = 0; s < S; ++s)
          if (armed & (1u << s)) wait_drain(full0 + 8 * s, (armed_par >> s) & 1u, wc);
      } else if (armed != 0u && *abort_flag) {
        // The odd CTA's copies signal the even CTA's barriers.  Without an abort every copy
        // it issued is consumed by an MMA that waited for it before the final cluster
        // barrier.  After one, its last copies were issued before a bounded wait expired
        // (a second at the default limit) and have long landed; settle a little longer
        // before the shared memory they write can be released.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 20000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA issuer (pair)
      // FP8 reads every operand K-major; bf16 reads some MN-major (KindOf)
      constexpr bool a_mn = !F8 && KindOf<K>::a_mn;
      constexpr bool b_mn = !F8 && KindOf<K>::b_mn;
      constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(2 * kBM, kBN)
                                    : idesc_bf16_f32(2 * kBM, kBN, a_mn, b_mn);
      // Shared-memory descriptors of stage 0; a stage's and an MMA's are these plus an
      // offset in the 14-bit address field (byte address / 16), which cannot carry out of
      // the field: shared memory ends below 256 KB.
      static_assert(kPairSmem < 256 * 1024, "descriptor address field");
      const uint64_t adesc0 = a_mn ? sdesc(sA0, kChunk, 1024, 2u) : sdesc(sA0, 16, 1024, 2u);
      const uint64_t bdesc0 = b_mn ? sdesc(sB0, kChunk, 1024, 2u) : sdesc(sB0, 16, 1024, 2u);
      constexpr uint32_t kAk = (a_mn ? 2048u : 32u) >> 4, kBk = (b_mn ? 2048u : 32u) >> 4;
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int u = cid; u < num_units; u += nclusters, ++it) {
        int st, kb0, kb1, part;
        unit_range(u, split, split_start, p.num_kb, st, kb0, kb1, part);
        const int buf = it & 1;
        const uint32_t acc_par = (it >> 1) & 1;
        if (!wait_bounded(tempty0 + 8 * buf, acc_par ^ 1u, wc, kSiteMmaAccEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kBN;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {  // stage order; the producer chose the k-blocks
          if (!wait_bounded(full0 + 8 * stage, phase, wc, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t as = adesc0 + static_cast<uint32_t>(stage) * (kPairAStage >> 4);
          const uint64_t bs = bdesc0 + static_cast<uint32_t>(stage) * (kPairBStage >> 4);
          // four MMAs a stage: K = 16 bf16 or 32 E4M3 each, 32 bytes of every K-major row
          // (MN-major: the next 8-row group of K, 2 KB on)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = as + kk * kAk;
            const uint64_t bd = bs + kk * kBk;
            const uint32_t accumulate = (kb != kb0 || kk != 0) ? 1u : 0u;
            if constexpr (F8)
              umma_f8_pair(d, ad, bd, idesc, accumulate);
            else
              umma_bf16_pair(d, ad, bd, idesc, accumulate);
          }
          umma_commit_pair_mc(empty0 + 8 * stage, 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(tfull0 + 8 * buf, 0x3);
      }
      umma_commit_pair(drain);
      wait_drain(drain, 0, wc);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    float sc = 1.0f;  // FP8: 2^-(k_a + k_b), exact
    if constexpr (F8) sc = ldexpf(1.0f, -(e4m3_scale_exp(*p.amax_a) + e4m3_scale_exp(*p.amax_b)));
    int it = 0;
    for (int u = cid; u < num_units; u += nclusters, ++it) {
      int st, kb0, kb1, part;
      unit_range(u, split, split_start, p.num_kb, st, kb0, kb1, part);
      const int buf = it & 1;
      const uint32_t acc_par = (it >> 1) & 1;
      int ok = 1;
      if (lane == 0)
        ok = wait_bounded(tfull0 + 8 * buf, acc_par, wc, kSiteEpiAccFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      int mp, nt;
      tile_coords(st, num_pm, p.num_n_tiles, p.raster_group, mp, nt);
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * kBN;
      float am = 0.0f;
      if (part >= 0) {  // a K-range of a tail tile: raw partial sums, summed by the fixup
        float* P = p.partial +
                   ((static_cast<size_t>(st - split_start) * split + part) * 2 + rank) * (kBM * kBN) +
                   static_cast<size_t>(row) * kBN;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          float v[32];
          load_acc<F8>(tacc + c * 32, v, sc);
          store_f32x32(P + c * 32, 32, v);
        }
      } else {
        epilogue_tile<K, F8>(tacc, row, mp * 2 + rank, nt, p, sc, am);
      }
      if constexpr (F8) {
        if (p.amax_out != nullptr) {  // non-negative floats order like their bit patterns
          const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(am));
          if (lane == 0 && m != 0u) atomicMax(p.amax_out, m);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty0 + 8 * buf);
        else mbar_arrive_remote(tempty_lead + 8 * buf);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // no remote arrive or MMA of the pair is still outstanding
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace mlpb
