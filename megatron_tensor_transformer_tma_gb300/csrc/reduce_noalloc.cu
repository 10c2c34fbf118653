// mlpb_bias_grad_noalloc: the bias-gradient column sum with its scratch in a fixed,
// file-scope device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot obtain device memory at the point where they need a
// bias gradient -- for example code running under a memory manager that owns every byte
// of the GPU (a framework pool or a fixed budget reserved at start-up) and has no
// temporary buffer to hand out there, or code running inside such a manager's own
// callbacks, where calling cudaMalloc could fail or re-enter the manager.  This entry
// point needs no handle (creating one allocates its error word) and no workspace.
//
// The scratch holds the first pass's per-split partial sums, at most kScratchFloats
// fp32 values (4 MiB); every GPU that loads the library keeps it until the process exits.
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/mlpb.h"
#include "kernels.h"

namespace {

constexpr int64_t kScratchFloats = int64_t(1) << 20;  // 4 MiB of fp32 partials

static __device__ __align__(256) float g_colsum_scratch[kScratchFloats];

// The device address of g_colsum_scratch on the current device.  The host-side name
// g_colsum_scratch is only a stand-in for the device array; its device address comes
// from cudaGetSymbolAddress, which the first call on a device also uses to load the
// library's device code there.  The address is resolved again on every call (a host
// lookup once the code is loaded), so it stays valid if the caller resets the device or
// releases and re-creates its context: a cached address could then name memory that
// no longer holds the array.
mlpb_status current_scratch(float** scratch, int* num_sms) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLPB_ECUDA;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_colsum_scratch) != cudaSuccess || ptr == nullptr)
    return MLPB_ECUDA;
  if (cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return MLPB_ECUDA;
  *scratch = static_cast<float*>(ptr);
  return MLPB_OK;
}

}  // namespace

extern "C" mlpb_status mlpb_bias_grad_noalloc(const void* in, int64_t rows, int64_t cols,
                                              float* out, mlpb_stream_t stream) {
  if (in == nullptr && rows > 0) return MLPB_EINVAL;
  if (out == nullptr || rows < 0 || cols <= 0) return MLPB_EINVAL;
  if (cols % 8 != 0) return MLPB_EUNSUPPORTED;  // 16-byte rows of 8 bf16
  if (cols > kScratchFloats) return MLPB_EUNSUPPORTED;  // one split of partials must fit
  if ((reinterpret_cast<uintptr_t>(in) & 15u) != 0 || (reinterpret_cast<uintptr_t>(out) & 15u) != 0)
    return MLPB_EINVAL;
  float* scratch = nullptr;
  int num_sms = 0;
  const mlpb_status st = current_scratch(&scratch, &num_sms);
  if (st != MLPB_OK) return st;

  // Row splits: about four CTAs per SM over the 512-column chunks, at least 16 rows per
  // split, and no more splits than the scratch holds.
  const int64_t chunks = (cols + 511) / 512;
  int64_t splits = std::max<int64_t>(1, (4 * num_sms + chunks - 1) / chunks);
  splits = std::min<int64_t>(splits, std::max<int64_t>(1, rows / 16));
  splits = std::min<int64_t>(splits, kScratchFloats / cols);
  const int64_t rows_per_split = std::max<int64_t>(1, (rows + splits - 1) / splits);
  splits = std::max<int64_t>(1, (rows + rows_per_split - 1) / rows_per_split);
  // Pass 1 writes every partial pass 2 reads, so earlier calls' leftovers need no clearing.
  const cudaError_t e = mlpb::launch_colsum_bf16(in, rows, cols, static_cast<int>(splits),
                                                 rows_per_split, scratch, out,
                                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLPB_OK : MLPB_ECUDA;
}
