// The residency cache's step plan and expert copies as device functions, shared by the
// cache's own kernels and the single-launch serving kernel.
//
// Relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B de
// NanoColibri por $200"), opening section, second paragraph: int4 experts streamed
// through an LRU cache under a memory budget.  Policy (least recently used): the step's
// hits are stamped first, then its misses, in ascending expert order, each take the slot
// with the smallest stamp among those not used in the step, ties to the lowest slot.
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace moe {

// Scratch of the plan (shared memory of the calling block): the step's new tables, and
// what cache_plan_write_back stores.
struct CachePlanScratch {
  unsigned used[kMaxE / 32];
  int stamp[kMaxCacheSlots], slot_expert[kMaxCacheSlots], expert_slot[kMaxE];
  CacheState next;  // the counters after the step (written by lane 0)
  int failed;
};

// One warp plans the step from the routing result idx [pairs] (after `ready_wait`, a
// callable the warp runs between loading the cache's state and reading idx): the new
// slot tables, stamps and counters in the scratch, the copies listed in jobs (global,
// jobs[0 .. next.njobs)).  The tables and counters are written back to global memory
// by cache_plan_write_back, which the caller may defer until nothing reads the old
// tables any more.  Every load the plan needs is issued up front; no block-wide barrier.
template <typename ReadyWait>
__device__ __forceinline__ void cache_plan_warp(const int32_t* idx, int pairs, int E, int slots, CacheState* st,
                                                int32_t* slot_expert, int32_t* stamp, int32_t* expert_slot,
                                                int2* jobs, long long expert_bytes, int* status,
                                                CachePlanScratch& sc, int lane, ReadyWait ready_wait) {
  if (lane < kMaxE / 32) sc.used[lane] = 0u;
  // State first (independent of the router), then the routing result.
  const CacheState h = *st;
  for (int c = lane; c < slots; c += 32) {
    sc.stamp[c] = stamp[c];
    sc.slot_expert[c] = slot_expert[c];
  }
  for (int e = lane; e < E; e += 32) sc.expert_slot[e] = expert_slot[e];
  ready_wait();
  __syncwarp();
  for (int i = lane; i < pairs; i += 32) {
    const int e = idx[i];
    if (e >= 0 && e < E) atomicOr(&sc.used[e >> 5], 1u << (e & 31));
  }
  __syncwarp();
  const int step = h.step;
  // Hits: stamped first, so that nothing this step uses can be chosen as a victim.
  int hits = 0;
  for (int e = lane; e < E; e += 32)
    if (((sc.used[e >> 5] >> (e & 31)) & 1u) && sc.expert_slot[e] >= 0) {
      sc.stamp[sc.expert_slot[e]] = step;
      ++hits;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) hits += __shfl_xor_sync(0xFFFFFFFFu, hits, o);
  __syncwarp();
  // Misses in ascending expert order, one at a time; the victim is the lexicographic
  // minimum of (stamp, slot) over the slots with stamp < step.
  int njobs = 0, evictions = 0, failed = 0;
  for (int e = 0; e < E; ++e) {
    if (!((sc.used[e >> 5] >> (e & 31)) & 1u) || sc.expert_slot[e] >= 0) continue;  // warp-uniform
    int best_st = 0x7FFFFFFF, best_c = -1;
    for (int c = lane; c < slots; c += 32) {
      const int s = sc.stamp[c];
      if (s < step && (best_c < 0 || s < best_st)) {  // c ascends within a lane
        best_st = s;
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
    const int old = sc.slot_expert[best_c];
    if (old >= 0) ++evictions;
    __syncwarp();
    if (lane == 0) {
      if (old >= 0) sc.expert_slot[old] = -1;
      sc.slot_expert[best_c] = e;
      sc.expert_slot[e] = best_c;
      sc.stamp[best_c] = step;
      jobs[njobs] = make_int2(e, best_c);
    }
    ++njobs;
    __syncwarp();
  }
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
    sc.next = n;
    sc.failed = failed;
  }
  __syncwarp();
}

// The plan's new tables and counters, from the scratch to global memory (one warp).
__device__ __forceinline__ void cache_plan_write_back(const CachePlanScratch& sc, int E, int slots, CacheState* st,
                                                      int32_t* slot_expert, int32_t* stamp, int32_t* expert_slot,
                                                      int lane) {
  for (int c = lane; c < slots; c += 32) {
    stamp[c] = sc.stamp[c];
    slot_expert[c] = sc.slot_expert[c];
  }
  for (int e = lane; e < E; e += 32) expert_slot[e] = sc.expert_slot[e];
  if (lane == 0) *st = sc.next;
}

// Copies the planned experts' four weight segments from host memory into their slots:
// thread `first` of `stride` threads, four 16-byte loads in flight per thread (the
// CPU-GPU link wants many bytes in flight); one pass per segment.
constexpr int kCacheCopyUnroll = 4;
__device__ __forceinline__ void cache_copy_range(int njobs, const int2* jobs, const CacheSegments& src,
                                                 const CacheSegments& dst, long long first, long long stride) {
#pragma unroll
  for (int sg = 0; sg < 4; ++sg) {
    const long long per = src.bytes[sg] / 16;
    const long long total = (long long)njobs * per;
    for (long long u0 = first; u0 < total; u0 += kCacheCopyUnroll * stride) {
      uint4 v[kCacheCopyUnroll];
#pragma unroll
      for (int r = 0; r < kCacheCopyUnroll; ++r) {
        const long long u = u0 + r * stride;
        if (u < total) {
          const int2 job = jobs[u / per];
          v[r] = __ldcs(reinterpret_cast<const uint4*>(src.base[sg] + (long long)job.x * src.bytes[sg]) + u % per);
        }
      }
#pragma unroll
      for (int r = 0; r < kCacheCopyUnroll; ++r) {
        const long long u = u0 + r * stride;
        if (u < total) {
          const int2 job = jobs[u / per];
          reinterpret_cast<uint4*>(dst.base[sg] + (long long)job.y * dst.bytes[sg])[u % per] = v[r];
        }
      }
    }
  }
}

}  // namespace moe
