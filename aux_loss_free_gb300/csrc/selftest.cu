// Self-test of the failure path: the library's kernels never trap; a wait that cannot
// complete gives up after a wall-clock limit, records the timeout in the device status
// word and returns.  This kernel makes one wait run out on purpose -- a counter that
// nothing raises -- through the same helper the chained GEMM launch waits with, so a
// test can check that the limit holds, that the host reads the timeout, and that the
// context stays usable.  Nothing faults: no trap, no bad address, no endless loop.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__device__ int g_never_raised;  // zero-initialised, never written
__device__ int g_gave_up;

__global__ void bounded_wait_selftest_kernel(unsigned long long limit_ns, int* status) {
  if (threadIdx.x == 0 && blockIdx.x == 0)
    g_gave_up = wait_counter_geq(&g_never_raised, 1, status, limit_ns) ? 0 : 1;
}

}  // namespace

cudaError_t run_bounded_wait_selftest(unsigned long long limit_ns, int* gave_up, cudaStream_t s) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevicePointer;
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(gave_up, g_gave_up, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

}  // namespace moe
