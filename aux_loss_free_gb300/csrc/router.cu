// Router: fp32 logits, sigmoid scores, biased top-k selection, gates and loads.
//
// Relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B de
// NanoColibri por $200"), opening section, architecture paragraph: sigmoid-plus-bias
// router with top-2 routing; section "Entrenamiento por relevos", top-2 paragraph:
// gates are the winners' scores renormalised over the k winners.
//
// One block handles 32 tokens.  Phase 1 is an fp32 tile product (32 tokens x 64
// experts per pass, each thread a 4 x 4 register tile) with x and W_r staged in shared
// memory; phase 2 gives each warp whole tokens: every lane holds E/32 experts'
// scores in registers, the top-k is k rounds of a warp-shuffle arg-max under the
// order (key descending, expert index ascending), and the gate normalisation is a
// register sum.  Per-block expert counts go to shared memory, then one atomic per
// expert to the global load (and to the permutation's chunk table when asked).
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"
#include "select.cuh"

namespace moe {
namespace {

constexpr int RT = kRouterTokens;  // tokens per block
constexpr int KC = 64;             // K chunk staged in shared memory
constexpr int EB = 64;             // experts per pass
constexpr int NTHR = 128;
constexpr int XS_LD = RT + 4;
constexpr int WS_LD = EB + 4;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

template <bool XF32>
__global__ void __launch_bounds__(NTHR) router_kernel(RouterArgs a) {
  __shared__ __align__(16) float xs[KC][XS_LD];
  __shared__ __align__(16) float ws[KC][WS_LD];
  __shared__ int hist[kMaxE];
  extern __shared__ float logits[];  // [RT][E + 1]

  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * RT;
  const int E = a.E, d = a.d, LD = a.E + 1;
  for (int e = tid; e < E; e += NTHR) hist[e] = 0;

  const int tx = tid % 16, ty = tid / 16;
  for (int e0 = 0; e0 < E; e0 += EB) {
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += KC) {
      __syncthreads();
#pragma unroll
      for (int pass = 0; pass < RT * KC / 4 / NTHR; ++pass) {
        const int li = pass * NTHR + tid;
        const int tok = li / 16, kq = (li % 16) * 4;
        const int t = t0 + tok;
        float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
        if (t < a.T) {
          if (XF32) {
            const float4 f =
                *reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)t * d + k0 + kq);
            v0 = f.x; v1 = f.y; v2 = f.z; v3 = f.w;
          } else {
            const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) +
                                                            (size_t)t * d + k0 + kq);
            v0 = bf16_bits_to_f32(u.x & 0xFFFFu); v1 = bf16_bits_to_f32(u.x >> 16);
            v2 = bf16_bits_to_f32(u.y & 0xFFFFu); v3 = bf16_bits_to_f32(u.y >> 16);
          }
        }
        xs[kq + 0][tok] = v0; xs[kq + 1][tok] = v1; xs[kq + 2][tok] = v2; xs[kq + 3][tok] = v3;
      }
#pragma unroll
      for (int pass = 0; pass < EB * KC / 4 / NTHR; ++pass) {
        const int li = pass * NTHR + tid;
        const int el = li / 16, kq = (li % 16) * 4;
        const int e = e0 + el;
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < E) f = *reinterpret_cast<const float4*>(a.w_router + (size_t)e * d + k0 + kq);
        ws[kq + 0][el] = f.x; ws[kq + 1][el] = f.y; ws[kq + 2][el] = f.z; ws[kq + 3][el] = f.w;
      }
      __syncthreads();
#pragma unroll 16
      for (int kk = 0; kk < KC; ++kk) {
        const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][ty * 4]);
        const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
        const float xr[4] = {xv.x, xv.y, xv.z, xv.w};
        const float wr[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xr[i], wr[j], acc[i][j]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = e0 + tx * 4 + j;
        if (e < E) {
          const float off = a.logit_offset ? a.logit_offset[e] : 0.f;
          logits[(ty * 4 + i) * LD + e] = acc[i][j] + off;
        }
      }
  }
  __syncthreads();

  const int warp = tid / 32, lane = tid % 32;
  for (int tok = warp; tok < RT; tok += NTHR / 32) {
    const int t = t0 + tok;
    if (t >= a.T) break;  // warp-uniform
    select_token(a, &logits[tok * LD], t, lane, hist);
  }
  __syncthreads();
  for (int e = tid; e < E; e += NTHR) {
    const int h = hist[e];
    if (h) {
      if (a.load) atomicAdd(&a.load[e], h);
      if (a.counts) atomicAdd(&a.counts[(size_t)(t0 / a.chunk_tokens) * E + e], h);
    }
  }
}


// Small-T router: a cluster of CL CTAs per CTPB tokens.  CTA r of the cluster computes
// the logits of experts [r*EPC, (r+1)*EPC) for the cluster's tokens, one warp per
// expert row of W_r (read once, coalesced float4) against the tokens staged in shared
// memory; CTA 0 then gathers all E logits over distributed shared memory and runs the
// selection, one warp per token.  At T = 1 this spreads the 256 KB of W_r over
// 64 warps on 8 SMs instead of one block.
constexpr int CL = 8;
constexpr int CTPB = 4;
constexpr int CTHR = 256;

template <bool XF32>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(CTHR) router_cluster_kernel(RouterArgs a) {
  extern __shared__ __align__(16) float csm[];
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int E = a.E, d = a.d;
  const int EPC = (E + CL - 1) / CL;
  const int t0 = (blockIdx.x / CL) * CTPB;
  float* xs = csm;                 // [CTPB][d]
  float* lg = xs + CTPB * d;       // [CTPB][EPC] this CTA's logits
  float* all = lg + CTPB * EPC;    // [CTPB][E] (CTA 0)
  for (int i = tid; i < CTPB * d; i += CTHR) {
    const int tok = i / d, kk = i % d, t = t0 + tok;
    float v = 0.f;
    if (t < a.T) {
      if (XF32)
        v = static_cast<const float*>(a.x)[(size_t)t * d + kk];
      else
        v = bf16_bits_to_f32(static_cast<const uint16_t*>(a.x)[(size_t)t * d + kk]);
    }
    xs[i] = v;
  }
  __syncthreads();
  const int e_begin = (int)rank * EPC, e_end = min(E, e_begin + EPC);
  for (int e = e_begin + warp; e < e_end; e += CTHR / 32) {
    float acc[CTPB];
#pragma unroll
    for (int tok = 0; tok < CTPB; ++tok) acc[tok] = 0.f;
    const float* wr = a.w_router + (size_t)e * d;
    // Eight float4 of the row in flight per lane before any is used.
    for (int k0 = lane * 4; k0 < d; k0 += 128 * 8) {
      float4 w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int kk = k0 + u * 128;
        w[u] = kk < d ? *reinterpret_cast<const float4*>(wr + kk) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int kk = k0 + u * 128;
        if (kk < d) {
#pragma unroll
          for (int tok = 0; tok < CTPB; ++tok) {
            const float4 xv = *reinterpret_cast<const float4*>(xs + tok * d + kk);
            acc[tok] = fmaf(w[u].x, xv.x, fmaf(w[u].y, xv.y, fmaf(w[u].z, xv.z, fmaf(w[u].w, xv.w, acc[tok]))));
          }
        }
      }
    }
    const float off = a.logit_offset ? a.logit_offset[e] : 0.f;
#pragma unroll
    for (int tok = 0; tok < CTPB; ++tok) {
      float v = acc[tok];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      if (lane == 0) lg[tok * EPC + (e - e_begin)] = v + off;
    }
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (rank == 0) {
    const uint32_t lg_base = static_cast<uint32_t>(__cvta_generic_to_shared(lg));
    for (int i = tid; i < CTPB * E; i += CTHR) {
      const int tok = i / E, e = i % E;
      const uint32_t src = (uint32_t)(e / EPC);
      uint32_t remote;
      const uint32_t local = lg_base + 4u * (uint32_t)(tok * EPC + e % EPC);
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(src));
      float v;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
      all[i] = v;
    }
    __syncthreads();
    if (warp < CTPB && t0 + warp < a.T) select_token(a, all + warp * E, t0 + warp, lane, nullptr);
  }
  // No CTA leaves while CTA 0 may still read its logits.
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Router of the permutation-free serving path (at most 64 tokens, bf16 tokens).  CTA
// (eb, tb) computes the logits of experts [4 eb, 4 eb + 4) for tokens [8 tb, 8 tb + 8),
// two warps per expert row of W_r, each against 4 tokens staged in shared memory, in
// the cluster router's summation order (the logits are the same bits), and writes them
// to scratch.  The last CTA of each token block (an atomic count per block) runs the
// selection for the block's tokens, one warp per token, and publishes the block's
// histogram; the last of those (a second count) adds the histograms into the loads,
// written outright, so they need no clearing.  The launcher zeroes the counters in the
// same stream.
constexpr int SR_EB = 4;   // experts per CTA (two warps each)
constexpr int SR_TB = 8;   // tokens per CTA (four per warp)
constexpr int SR_THR = 256;

__global__ void __launch_bounds__(SR_THR, 1) router_small_kernel(RouterArgs a, float* lgs, int* bhist,
                                                                unsigned* ctr) {
  extern __shared__ __align__(16) float ssm[];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int E = a.E, d = a.d, T = a.T;
  const int neb = (E + SR_EB - 1) / SR_EB;
  const int eb = (int)blockIdx.x % neb, t0 = ((int)blockIdx.x / neb) * SR_TB;
  const int e = eb * SR_EB + warp / 2, tq = (warp & 1) * 4;
  // The first 1024 inputs of this warp's W_r row, before the dependency wait: no
  // kernel writes the router weight.
  float4 w[8];
  const float* wr = a.w_router + (size_t)min(e, E - 1) * d;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int kk = lane * 4 + u * 128;
    w[u] = kk < d ? *reinterpret_cast<const float4*>(wr + kk) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();
  pdl_trigger();
  float* xs = ssm;  // [SR_TB][d]
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  for (int kk = tid * 8; kk < d; kk += SR_THR * 8) {
    uint4 u[SR_TB];  // every token's chunk in flight before any is stored
#pragma unroll
    for (int tok = 0; tok < SR_TB; ++tok)
      u[tok] = t0 + tok < T ? *reinterpret_cast<const uint4*>(x + (size_t)(t0 + tok) * d + kk) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int tok = 0; tok < SR_TB; ++tok) {
      float4* o = reinterpret_cast<float4*>(xs + tok * d + kk);
      o[0] = make_float4(bf16_bits_to_f32(u[tok].x & 0xFFFFu), bf16_bits_to_f32(u[tok].x >> 16),
                         bf16_bits_to_f32(u[tok].y & 0xFFFFu), bf16_bits_to_f32(u[tok].y >> 16));
      o[1] = make_float4(bf16_bits_to_f32(u[tok].z & 0xFFFFu), bf16_bits_to_f32(u[tok].z >> 16),
                         bf16_bits_to_f32(u[tok].w & 0xFFFFu), bf16_bits_to_f32(u[tok].w >> 16));
    }
  }
  __syncthreads();
  if (e < E) {  // warp-uniform
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = lane * 4; k0 < d; k0 += 128 * 8) {
      if (k0 != lane * 4) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int kk = k0 + u * 128;
          w[u] = kk < d ? *reinterpret_cast<const float4*>(wr + kk) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int kk = k0 + u * 128;
        if (kk < d) {
#pragma unroll
          for (int tok = 0; tok < 4; ++tok) {
            const float4 xv = *reinterpret_cast<const float4*>(xs + (tq + tok) * d + kk);
            acc[tok] = fmaf(w[u].x, xv.x, fmaf(w[u].y, xv.y, fmaf(w[u].z, xv.z, fmaf(w[u].w, xv.w, acc[tok]))));
          }
        }
      }
    }
    const float off = a.logit_offset ? a.logit_offset[e] : 0.f;
#pragma unroll
    for (int tok = 0; tok < 4; ++tok) {
      float v = acc[tok];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      const int t = t0 + tq + tok;
      if (lane == 0 && t < T) lgs[(size_t)t * E + e] = v + off;
    }
  }
  __syncthreads();
  const int ntb = (T + SR_TB - 1) / SR_TB, tb = t0 / SR_TB;
  if (tid == 0) {
    __threadfence();  // the CTA's logits, ordered before this thread by the barrier
    s_last = atomicAdd(&ctr[tb], 1u) == (unsigned)neb - 1;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  // The block's last CTA: its tokens' logits (one load per thread in flight), then one
  // warp per token.
  float* lb = ssm;  // [SR_TB][E]
  int* hist = reinterpret_cast<int*>(lb + SR_TB * E);
  const int nt = min(SR_TB, T - t0);
  {
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = tid + j * SR_THR;
      v[j] = i < nt * E ? __ldcg(lgs + (size_t)t0 * E + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (tid + j * SR_THR < nt * E) lb[tid + j * SR_THR] = v[j];
    for (int i = tid + 4 * SR_THR; i < nt * E; i += SR_THR) lb[i] = __ldcg(lgs + (size_t)t0 * E + i);
  }
  for (int i = tid; i < E; i += SR_THR) hist[i] = 0;
  __syncthreads();
  if (warp < nt) select_token(a, lb + (size_t)warp * E, t0 + warp, lane, hist);
  if (!a.load) return;  // the same for the whole CTA
  __syncthreads();
  for (int i = tid; i < E; i += SR_THR) bhist[(size_t)tb * E + i] = hist[i];
  __syncthreads();
  if (tid == 0) {
    __threadfence();  // the CTA's writes, ordered before this thread by the barrier
    s_last = atomicAdd(&ctr[ntb], 1u) == (unsigned)ntb - 1;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  for (int i = tid; i < E; i += SR_THR) {
    int sum = 0;
    for (int b = 0; b < ntb; ++b) sum += __ldcg(bhist + (size_t)b * E + i);
    a.load[i] = sum;
  }
}

size_t router_small_smem(int T, int E, int d) {
  (void)T;
  return std::max((size_t)SR_TB * d * 4, (size_t)SR_TB * E * 4 + (size_t)E * 4);
}
}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  if (a.T <= kRouterClusterMaxT) {
    // Few tokens: spread W_r over a cluster per CTPB tokens.
    const int clusters = (a.T + CTPB - 1) / CTPB;
    const int epc = (a.E + CL - 1) / CL;
    const size_t dyn = sizeof(float) * ((size_t)CTPB * a.d + (size_t)CTPB * epc + (size_t)CTPB * a.E);
    if (a.x_is_f32) {
      cudaError_t e = cudaFuncSetAttribute(router_cluster_kernel<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
      if (e != cudaSuccess) return e;
      router_cluster_kernel<true><<<clusters * CL, CTHR, dyn, s>>>(a);
    } else {
      cudaError_t e = cudaFuncSetAttribute(router_cluster_kernel<false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
      if (e != cudaSuccess) return e;
      router_cluster_kernel<false><<<clusters * CL, CTHR, dyn, s>>>(a);
    }
    return cudaGetLastError();
  }
  const int blocks = (a.T + RT - 1) / RT;
  const size_t dyn = sizeof(float) * RT * (a.E + 1);
  if (a.x_is_f32) {
    cudaError_t e = cudaFuncSetAttribute(router_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    router_kernel<true><<<blocks, NTHR, dyn, s>>>(a);
  } else {
    cudaError_t e = cudaFuncSetAttribute(router_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    router_kernel<false><<<blocks, NTHR, dyn, s>>>(a);
  }
  return cudaGetLastError();
}


bool router_small_supported(const RouterArgs& a) {
  return !a.x_is_f32 && !a.counts && a.T >= 1 && a.T <= kDirectMaxPairs && a.E >= 1 && a.E <= kMaxE &&
         a.k >= 1 && a.k <= kMaxK && a.d % 8 == 0 && router_small_smem(a.T, a.E, a.d) <= 48 * 1024 &&
         (reinterpret_cast<uintptr_t>(a.x) & 15u) == 0 && (reinterpret_cast<uintptr_t>(a.w_router) & 15u) == 0;
}

// Scratch: logits [T][E] fp32, block histograms [T/8][E] int32, counters [T/8 + 1].
size_t router_small_scratch_bytes(int T, int E) {
  const size_t ntb = (T + SR_TB - 1) / SR_TB;
  return ((size_t)T * E * 4 + 15) / 16 * 16 + (ntb * E * 4 + 15) / 16 * 16 + ((ntb + 1) * 4 + 15) / 16 * 16;
}

cudaError_t launch_router_small(const RouterArgs& a, void* scratch, cudaStream_t s) {
  if (!router_small_supported(a)) return cudaErrorInvalidValue;
  const size_t ntb = (a.T + SR_TB - 1) / SR_TB;
  uint8_t* p = static_cast<uint8_t*>(scratch);
  float* lgs = reinterpret_cast<float*>(p);
  int* bhist = reinterpret_cast<int*>(p + ((size_t)a.T * a.E * 4 + 15) / 16 * 16);
  auto* ctr = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(bhist) + (ntb * a.E * 4 + 15) / 16 * 16);
  cudaError_t e = cudaMemsetAsync(ctr, 0, (ntb + 1) * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const int grid = ((a.E + SR_EB - 1) / SR_EB) * (int)ntb;
  return launch_pdl(router_small_kernel, dim3(grid), dim3(SR_THR), router_small_smem(a.T, a.E, a.d), s, a, lgs, bhist,
                    ctr);
}

}  // namespace moe
