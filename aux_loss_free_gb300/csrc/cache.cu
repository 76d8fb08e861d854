// GPU-side residency cache of the int4 routed experts.
//
// Relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B de
// NanoColibri por $200"), opening section, second paragraph: the int4 experts are
// streamed from NVMe through an LRU cache under a memory budget; section
// "Entrenamiento por relevos", top-2 paragraph: the skew left after balancing is what
// such a cache likes.  Here every expert's int4 weights live in pinned host memory,
// HBM holds `slots` of them, and each serving step brings in what its routing uses,
// with no host round trip: one block plans the step (least recently used: hits
// stamped first, then the misses in ascending expert order each take the slot with the
// smallest stamp among those not used in the step, ties to the lowest slot), and a
// grid copies the missing experts' codes and scales from host memory over the
// CPU-GPU link straight into their slots.  The expert kernels then read the weights
// through the expert -> slot table.
#include <cuda_runtime.h>

#include "cache_plan.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// The plan runs in one warp (cache_plan_warp): every load it needs (the counters, the
// slot tables, the routing result) is issued up front.
__global__ void __launch_bounds__(32) cache_plan_kernel(const int32_t* __restrict__ idx, int pairs, int E,
                                                        int slots, CacheState* st,
                                                        int32_t* __restrict__ slot_expert,
                                                        int32_t* __restrict__ stamp,
                                                        int32_t* __restrict__ expert_slot,
                                                        int2* __restrict__ jobs, long long expert_bytes,
                                                        int* status) {
  __shared__ CachePlanScratch sc;
  cache_plan_warp(idx, pairs, E, slots, st, slot_expert, stamp, expert_slot, jobs, expert_bytes, status, sc,
                  (int)threadIdx.x, [] {
                    pdl_wait();  // idx comes from the router
                    pdl_trigger();
                  });
  cache_plan_write_back(sc, E, slots, st, slot_expert, stamp, expert_slot, (int)threadIdx.x);
}

// Copies the planned experts' weights from host memory into their slots: one block
// per SM (cache_copy_range).
__global__ void __launch_bounds__(256) cache_copy_kernel(const CacheState* st, const int2* __restrict__ jobs,
                                                         CacheSegments src, CacheSegments dst) {
  pdl_wait();  // the plan
  pdl_trigger();
  const int njobs = st->njobs;
  if (njobs == 0) return;
  cache_copy_range(njobs, jobs, src, dst, (long long)blockIdx.x * blockDim.x + threadIdx.x,
                   (long long)gridDim.x * blockDim.x);
}

}  // namespace

cudaError_t launch_cache_fetch(const int32_t* idx, int pairs, int E, int slots, const CacheView& v,
                               const CacheSegments& host_src, long long expert_bytes, cudaStream_t s) {
  if (slots < 1 || slots > kMaxCacheSlots || E > kMaxE) return cudaErrorInvalidValue;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevicePointer;
  cudaError_t e = launch_pdl(cache_plan_kernel, dim3(1), dim3(32), 0, s, idx, pairs, E, slots, v.state,
                             v.slot_expert, v.stamp, v.expert_slot, v.jobs, expert_bytes, status);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_pdl(cache_copy_kernel, dim3(sms), dim3(256), 0, s, static_cast<const CacheState*>(v.state),
                    static_cast<const int2*>(v.jobs), host_src, v.slots_w);
}

}  // namespace moe
