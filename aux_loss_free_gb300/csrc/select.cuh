// Routing helpers shared by the router kernels, the permutation launch and the fused
// serving kernel: the per-token selection, the balance statistics of a load vector and
// the aux-loss-free bias step.
//
// Relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B de
// NanoColibri por $200"), opening section, architecture paragraph: sigmoid-plus-bias
// router, top-k routing, the bias moved by the sign of (target - load); section
// "Entrenamiento por relevos": the dashboard's expert balance, the top-2 paragraph's
// renormalised gates and dead-expert fraction.
#pragma once
#include <math.h>

#include "internal.h"

namespace moe {

constexpr int kSelMaxC = kMaxE / 32;  // experts per lane in the selection

// Selection for one token by one warp, from its E logits (offset included): scores,
// the biased top-k (k rounds of a warp-shuffle arg-max under key descending, expert
// index ascending), gates, and the pair counts (into the block histogram `hist`, or
// straight into the global load and chunk table when `hist` is null).
__device__ __forceinline__ void select_token(const RouterArgs& a, const float* lg, int t, int lane,
                                             int* hist) {
  const unsigned FULL = 0xFFFFFFFFu;
  constexpr int NONE = 0x7FFFFFFF;
  const int E = a.E;
  float sc[kSelMaxC], key[kSelMaxC];
#pragma unroll
  for (int i = 0; i < kSelMaxC; ++i) {
    const int e = lane + 32 * i;
    sc[i] = 0.f;
    key[i] = -INFINITY;
    if (e < E) {
      const float z = lg[e];
      const float s = 1.0f / (1.0f + expf(-z));
      sc[i] = s;
      key[i] = __fadd_rn(s, a.bias[e]);  // selection key: one fp32 addition
      if (a.scores) a.scores[(size_t)t * E + e] = s;
    }
  }
  unsigned taken = 0;
  float sel_s[kMaxK];
  int sel_e[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    sel_s[j] = 0.f;
    sel_e[j] = 0;
    if (j < a.k) {
      float bk = -INFINITY;
      int be = NONE;
#pragma unroll
      for (int i = 0; i < kSelMaxC; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (be == NONE || key[i] > bk)) {
          bk = key[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ok = __shfl_xor_sync(FULL, bk, off);
        const int oe = __shfl_xor_sync(FULL, be, off);
        if (oe != NONE && (be == NONE || ok > bk || (ok == bk && oe < be))) {
          bk = ok;
          be = oe;
        }
      }
      float sw = 0.f;
      if ((be & 31) == lane) {
        taken |= 1u << (be >> 5);
#pragma unroll
        for (int i = 0; i < kSelMaxC; ++i)
          if (i == (be >> 5)) sw = sc[i];
      }
      sel_s[j] = __shfl_sync(FULL, sw, be & 31);
      sel_e[j] = be;
    }
  }
  float denom = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j)
    if (j < a.k) denom += sel_s[j];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < a.k && lane == j) {
      a.idx[(size_t)t * a.k + j] = sel_e[j];
      a.gate[(size_t)t * a.k + j] = a.renorm ? __fdiv_rn(sel_s[j], denom) : sel_s[j];
      if (!hist) {
        if (a.load) atomicAdd(&a.load[sel_e[j]], 1);
        if (a.counts) atomicAdd(&a.counts[(size_t)(t / a.chunk_tokens) * E + sel_e[j]], 1);
      }
    }
  }
  if (hist && lane == 0) {
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < a.k) atomicAdd(&hist[sel_e[j]], 1);
  }
}

// Balance statistics of load[0..E) (moe_balance_t) by one warp; lane 0 writes them.
// The ratios are the fp32 values nearest to the exact rationals: the fp64 quotient of
// the two exact integers is correctly rounded, and rounding it again to fp32 gives the
// nearest fp32 for denominators below 2^28 (the exact quotient then never lies within
// half an fp64 ulp of an fp32 rounding boundary unless it is one).
__device__ __forceinline__ void warp_balance(const int32_t* load, int E, moe_balance_t* out, int lane) {
  int mx = 0, mn = 0x7FFFFFFF, dead = 0;
  long long sum = 0;
  for (int e = lane; e < E; e += 32) {
    const int v = load[e];
    mx = max(mx, v);
    mn = min(mn, v);
    dead += v == 0;
    sum += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
    dead += __shfl_xor_sync(0xFFFFFFFFu, dead, o);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  }
  if (lane == 0) {
    out->pairs = sum;
    out->max_load = mx;
    out->min_load = mn;
    out->dead_experts = dead;
    const double pe = (double)sum;
    out->max_over_mean = sum > 0 ? __double2float_rn(__ddiv_rn((double)mx * E, pe)) : 0.f;
    out->min_over_mean = sum > 0 ? __double2float_rn(__ddiv_rn((double)mn * E, pe)) : 0.f;
    out->dead_fraction = __double2float_rn(__ddiv_rn((double)dead, (double)E));
  }
}

// b + gamma * sign(T*k - E * load): one fp32 addition (sign taken on the exact
// integer difference, so the target T*k / E is never rounded).
__device__ __forceinline__ float biased_step(float b, long long tokens_times_k, int E, int load, float gamma) {
  const long long diff = tokens_times_k - (long long)E * load;
  const float step = diff > 0 ? gamma : (diff < 0 ? -gamma : 0.f);
  return __fadd_rn(b, step);
}

}  // namespace moe
