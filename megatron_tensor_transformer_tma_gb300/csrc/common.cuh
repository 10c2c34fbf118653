// Shared device helpers: the device error word, bounded mbarrier waits, bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "ptx.cuh"

namespace mlpb {

// Device error word values (first error wins).  The low byte names the wait site.
constexpr uint32_t kDevErrTimeout = 0x100u;
enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaFull = 2,
  kSiteMmaAccEmpty = 3,
  kSiteEpiAccFull = 4,
  kSiteDrain = 5,
  kSiteLnFull = 6,
};

// Default limit of one bounded wait: 1 s of wall time (globaltimer).
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

struct WaitCtx {
  volatile uint32_t* abort_flag;  // shared memory, set by the first waiter that gives up
  uint32_t* err;                  // global device error word
  uint64_t limit_ns;
};

// Spins on an mbarrier phase.  Gives up (returns false) when the CTA's abort flag is
// raised or the limit expires; on expiry it raises the abort flag and records the site.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                             uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        *w.abort_flag = 1u;
        atomicCAS(w.err, 0u, kDevErrTimeout | site);
        return false;
      }
    }
  }
}

// Waits for copies or MMAs that were already issued (they always complete); ignores the
// abort flag but still gives up after the limit.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > w.limit_ns) {
      atomicCAS(w.err, 0u, kDevErrTimeout | kSiteDrain);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Read-only 16-byte load (ld.global.nc).  Not an asm volatile: the compiler must be free
// to hoist a batch of these ahead of their uses so that they are in flight together.
__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  return __ldg(static_cast<const uint4*>(p));
}

}  // namespace mlpb
