// moe_permute_noalloc: the stable counting-sort permutation without a caller-supplied
// workspace.
//
// Who needs this: code that cannot hand the library device memory for scratch.
// Examples are a plugin running inside a host framework that owns the device memory
// pool and gives plugins no scratch, or a serving loop whose device-memory budget is
// fixed at start-up and may not grow.  Those callers still pass their inputs and
// outputs; the per-chunk count table lives in the file-scope array below instead of
// a workspace.
//
// The array is a static __device__ symbol: every GPU that loads this library holds
// its 128 KiB until the process exits.  Host code must not pass the symbol itself
// to a kernel (on the host it is only a stand-in, not a device address); the device
// address is looked up once per device with cudaGetSymbolAddress and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "moe_gb300.h"

namespace moe {
namespace {

// The count table: at most kMaxCountEntries int32.
constexpr size_t kNoAllocScratchInts = (size_t)kMaxCountEntries;
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

// Device address of g_permute_scratch on the current device, looked up on the first
// call made on that device (with it current) and cached; nullptr on failure.  The
// address belongs to the device's context as it was then: a cudaDeviceReset would
// leave it stale, which is why the header rules out use of the library after one.
int32_t* scratch_on_current_device() {
  static int32_t* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    int32_t* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_permute_scratch) != cudaSuccess)
      return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_permute_noalloc(const moe_shape_t* shape, const int32_t* idx,
                                            int32_t* offsets, int32_t* perm_tok,
                                            int32_t* inv_pos, void* stream) {
  // The same validation, in the same order, as moe_permute.
  const moe_status_t st = check_shape(shape);
  if (st) return st;
  if (!idx || !offsets || !perm_tok || !inv_pos) return MOE_ERR_INVALID_ARG;
  const int ct = permute_chunk_tokens(shape->T, shape->E);
  const int chunks = (shape->T + ct - 1) / ct;
  const size_t table = (size_t)chunks * shape->E;
  if (table > kNoAllocScratchInts) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
  int32_t* scratch = scratch_on_current_device();
  if (!scratch) return MOE_ERR_CUDA;
  int32_t* counts = scratch;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the count table must start at zero.
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * table, s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e = launch_count(idx, shape->T, shape->k, shape->E, ct, counts, s);
  if (e == cudaSuccess)
    e = launch_scatter(idx, counts, shape->T, shape->k, shape->E, ct, offsets, nullptr, nullptr,
                       0.f, 0, perm_tok, inv_pos, nullptr, 0, shape->d, nullptr, nullptr, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
