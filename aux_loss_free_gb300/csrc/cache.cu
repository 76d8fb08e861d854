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

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// The plan runs in one warp: every load it needs (the counters, the slot tables, the
// routing result) is issued up front, and no block-wide barrier is needed.
__global__ void __launch_bounds__(32) cache_plan_kernel(const int32_t* __restrict__ idx, int pairs, int E,
                                                        int slots, CacheState* st,
                                                        int32_t* __restrict__ slot_expert,
                                                        int32_t* __restrict__ stamp,
                                                        int32_t* __restrict__ expert_slot,
                                                        int2* __restrict__ jobs, long long expert_bytes,
                                                        int* status) {
  __shared__ unsigned used[kMaxE / 32];
  __shared__ int s_stamp[kMaxCacheSlots], s_se[kMaxCacheSlots], s_es[kMaxE];
  const int lane = threadIdx.x;
  if (lane < kMaxE / 32) used[lane] = 0u;
  // State first (independent of the router), then the routing result.
  const CacheState h = *st;
  for (int c = lane; c < slots; c += 32) {
    s_stamp[c] = stamp[c];
    s_se[c] = slot_expert[c];
  }
  for (int e = lane; e < E; e += 32) s_es[e] = expert_slot[e];
  pdl_wait();  // idx comes from the router
  pdl_trigger();
  __syncwarp();
  for (int i = lane; i < pairs; i += 32) {
    const int e = idx[i];
    if (e >= 0 && e < E) atomicOr(&used[e >> 5], 1u << (e & 31));
  }
  __syncwarp();
  const int step = h.step;
  // Hits: stamped first, so that nothing this step uses can be chosen as a victim.
  int hits = 0;
  for (int e = lane; e < E; e += 32)
    if (((used[e >> 5] >> (e & 31)) & 1u) && s_es[e] >= 0) {
      s_stamp[s_es[e]] = step;
      ++hits;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) hits += __shfl_xor_sync(0xFFFFFFFFu, hits, o);
  __syncwarp();
  // Misses in ascending expert order, one at a time; the victim is the lexicographic
  // minimum of (stamp, slot) over the slots with stamp < step.
  int njobs = 0, evictions = 0, failed = 0;
  for (int e = 0; e < E; ++e) {
    if (!((used[e >> 5] >> (e & 31)) & 1u) || s_es[e] >= 0) continue;  // warp-uniform
    int best_st = 0x7FFFFFFF, best_c = -1;
    for (int c = lane; c < slots; c += 32) {
      const int sc = s_stamp[c];
      if (sc < step && (best_c < 0 || sc < best_st)) {  // c ascends within a lane
        best_st = sc;
        best_c = c;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int ost = __shfl_xor_sync(0xFFFFFFFFu, best_st, o);
      const int oc = __shfl_xor_sync(0xFFFFFFFFu, best_c, o);
      if (oc >= 0 && (best_c < 0 || ost < best_st || (ost == best_st && oc < best_c))) {
        best_st = ost;
        best_c = oc;
      }
    }
    if (best_c < 0) {  // more experts in this step than slots
      failed = 1;
      break;
    }
    const int old = s_se[best_c];
    if (old >= 0) ++evictions;
    __syncwarp();
    if (lane == 0) {
      if (old >= 0) s_es[old] = -1;
      s_se[best_c] = e;
      s_es[e] = best_c;
      s_stamp[best_c] = step;
      jobs[njobs] = make_int2(e, best_c);
    }
    ++njobs;
    __syncwarp();
  }
  for (int c = lane; c < slots; c += 32) {
    stamp[c] = s_stamp[c];
    slot_expert[c] = s_se[c];
  }
  for (int e = lane; e < E; e += 32) expert_slot[e] = s_es[e];
  if (lane == 0) {
    CacheState n = h;
    n.njobs = failed ? 0 : njobs;
    n.step = step + 1;
    n.hits += hits;
    n.misses += njobs;
    n.evictions += evictions;
    n.bytes += (long long)njobs * expert_bytes;
    if (failed) {
      n.overflow += 1;
      atomicOr(status, kDevCheck);
    }
    *st = n;
  }
}

// Copies the planned experts' four weight segments from host memory into their slots:
// one block per SM, four 16-byte loads in flight per thread (the CPU-GPU link wants
// many bytes in flight); one grid-stride pass per segment.
constexpr int COPY_UNROLL = 4;

__global__ void __launch_bounds__(256) cache_copy_kernel(const CacheState* st, const int2* __restrict__ jobs,
                                                         CacheSegments src, CacheSegments dst) {
  pdl_wait();  // the plan
  pdl_trigger();
  const int njobs = st->njobs;
  if (njobs == 0) return;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long first = (long long)blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll
  for (int sg = 0; sg < 4; ++sg) {
    const long long per = src.bytes[sg] / 16;
    const long long total = (long long)njobs * per;
    for (long long u0 = first; u0 < total; u0 += COPY_UNROLL * stride) {
      uint4 v[COPY_UNROLL];
#pragma unroll
      for (int r = 0; r < COPY_UNROLL; ++r) {
        const long long u = u0 + r * stride;
        if (u < total) {
          const int2 job = jobs[u / per];
          v[r] = __ldcs(reinterpret_cast<const uint4*>(src.base[sg] + (long long)job.x * src.bytes[sg]) + u % per);
        }
      }
#pragma unroll
      for (int r = 0; r < COPY_UNROLL; ++r) {
        const long long u = u0 + r * stride;
        if (u < total) {
          const int2 job = jobs[u / per];
          reinterpret_cast<uint4*>(dst.base[sg] + (long long)job.y * dst.bytes[sg])[u % per] = v[r];
        }
      }
    }
  }
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
