// Top-1 serving of a few tokens in one persistent launch (sm_103a): router, expert
// selection, bias update and balance statistics, the shared expert, the int4 routed
// experts and the combine.
//
// Relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B de
// NanoColibri por $200"), opening section: experts ship in an int4 container, a
// sigmoid-plus-bias router, one always-resident shared expert; section "Entrenamiento
// por relevos", top-2 paragraph: serving runs one expert per token.
//
// With at most kServeMaxPairs token-expert pairs the layer is a chain of small products
// whose cost is latency (launches, dependency waits, DRAM round trips), not bytes.  One
// launch with one CTA per SM does all of it:
//   0. every CTA starts bulk copies of its slices of the weights (W_r for the router
//      CTAs, gate/up rows of the shared expert for the shared CTAs, the shared down
//      rows of its output rows for every CTA) before waiting for the previous kernel,
//      then the copy of the tokens x; CTA 0 zeroes the call's counters and publishes
//      the call's id, which every CTA waits for before it counts;
//   1. the router CTAs (the first R) compute the fp32 logits of their experts for every
//      token and count themselves;
//   2. the shared CTAs compute their hidden units of the shared expert's SwiGLU for
//      every token (hs, bf16);
//   3. once every router CTA has counted, every CTA selects the experts of every token
//      from the logits (biased top-k, ties to the lower index; the same deterministic
//      result in every CTA), and starts copying its rows of the selected experts' down
//      projections; CTA 0 writes idx, gates, scores, loads and the balance statistics;
//   4. every CTA takes (expert, hidden unit) items of the routed experts' gate/up,
//      decoding the int4 codes in registers (h by pair, bf16);
//   5. after every CTA has finished 2 and 4 (a counted grid barrier) CTA 0 applies the
//      bias update (no CTA reads the bias any more) and each CTA writes its output rows:
//      out = residual + S + sum_j gate_j * y_j, with S the shared down projection in
//      fp32 and y_j the routed down projection rounded to bf16, as the multi-launch path
//      stores it.
// The launch needs every CTA resident at once (one per SM, grid = SM count); every wait
// on a flag, a counter or a copy is bounded: on a timeout the status word is set and the
// CTA goes on to the end (its outputs are then unspecified).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>
#include <atomic>

#include "cache_plan.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "select.cuh"

namespace moe {
namespace {

constexpr int SV_THREADS = 256;
constexpr int SV_WARPS = SV_THREADS / 32;
constexpr int SV_ROUTER_CTAS = 16;
constexpr int SV_MAXT = kServeMaxPairs;  // tokens (k >= 1)
constexpr unsigned FULLM = 0xFFFFFFFFu;

struct ServeParams {
  const uint16_t* x;          // [T][d] bf16
  const float* w_router;      // [E][d]
  const float* logit_offset;  // [E] or null
  float* bias;                // [E], updated in place when update_bias
  const uint8_t* gu_q;        // [E][2f][d/2] int4 codes (gate/up interleaved by block bf)
  const uint16_t* gu_s;       // [E][2f][d/32] fp16 scales
  const uint8_t* dn_q;        // [E][d][f/2]
  const uint16_t* dn_s;       // [E][d][f/32]
  const uint16_t* s_gu;       // [2F][d] bf16 (interleaved by block bF)
  const uint16_t* s_dn;       // [d][F] bf16
  const uint16_t* residual;   // [T][d] or null
  uint16_t* out;              // [T][d]
  float* scores;              // [T][E] or null
  int32_t* idx;               // [T][k]
  float* gate;                // [T][k]
  int32_t* load;              // [E] or null
  moe_balance_t* balance;     // or null
  float* logits;              // scratch [T][E]
  uint16_t* hs;               // scratch [T][F]
  uint16_t* h;                // scratch [T*k][f]
  int* sync;                  // [8]: router count, done count, the 64-bit id of the call that zeroed
                              // them, the cache's plan flag and fill count
  // Expert cache (cached != 0): the routed weights above are the slots' arrays, read
  // through expert_slot once this launch has planned the step and copied its misses.
  int cached, slots;
  CacheState* cstate;
  int32_t* slot_expert;
  int32_t* cstamp;
  int32_t* expert_slot;
  int2* jobs;
  CacheSegments host_src, slots_w;
  long long expert_bytes;
  unsigned long long call_id; // unique per call
  int* status;
  int T, d, E, f, F, k, renorm, update_bias, bf, bF;
  float gamma;
  int R, epc;                 // router CTAs and experts per router CTA
  int U, nSG;                 // shared hidden units per shared CTA, shared CTAs
  int RD;                     // output rows per CTA
  int MT;                     // 16-row tiles of a shared CTA's 2U gate/up rows
  int SX, SR, SD, SH;         // padded row strides (bf16) of x, shared gate/up rows, shared down rows, hs
  int o_x, o_w, o_sdn, o_hs, o_h, o_lg, o_hist, o_rd, o_b, o_red;  // shared-memory offsets (bytes)
};

// One bulk copy global -> shared (16-byte aligned, size a multiple of 16), counted on bar.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULLM, v, o);
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The kernel runs each of its phases once per SM and call, so its code is fetched
// more than it is reused: the larger helpers are kept out of line (one copy each).
//
// sum_i q_i * v_i over one group: q_i the 32 integer codes in `codes` (16 bytes of
// two's-complement nibbles, the even index in the low nibble: (c ^ 8) is q + 8 in
// [0, 15], and 2^23 + (q + 8) - (2^23 + 8) is q exactly in fp32), v the group's 32 bf16
// values in shared memory.
__device__ __noinline__ float group_qdot(const uint4 codes, const uint16_t* v) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
  const uint4* p = reinterpret_cast<const uint4*>(v);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = p[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float q0 = __uint_as_float(0x4B000000u | (((cw[i] >> (8 * j)) & 0xFu) ^ 0x8u)) - 8388616.0f;
      const float q1 = __uint_as_float(0x4B000000u | (((cw[i] >> (8 * j + 4)) & 0xFu) ^ 0x8u)) - 8388616.0f;
      acc = fmaf(q0, bf_lo(w[j]), acc);
      acc = fmaf(q1, bf_hi(w[j]), acc);
    }
  }
  return acc;
}

__device__ __forceinline__ uint16_t bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Acquire-spins (GPU scope, no sleep between reads) until *ctr >= target; bounded like
// every wait here (sets the timeout bit and returns false).
__device__ __forceinline__ bool spin_geq(const int* ctr, int target, int* status) {
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
}

// Acquire-spins until the 64-bit word at p equals want (bounded).
__device__ __forceinline__ bool spin_eq64(const unsigned long long* w, unsigned long long want, int* status) {
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(w) : "memory");
    if (v == want) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t ld_pair(const uint16_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// This warp's share of C[m][n] = sum_k A[m][k] B[n][k] for m < 16 * MT (rows past `rows_a`
// read as zero), n < 8 (columns past `cols_b` zero), k < K: the 16-deep K steps w, w + 8,
// ... of warp w, partial sums written to red[w][tile][16][8] for a reduction over warps.
// A rows `lda` bf16 apart, B columns `ldb` apart (both padded so the 32-bit fragment
// loads of a warp fall in distinct banks).
template <int MT>
__device__ __noinline__ void mma_rows_x_tokens(const uint16_t* A, int lda, int rows_a, const uint16_t* B, int ldb,
                                               int cols_b, int K, float* red, int warp, int lane) {
  const int g = lane >> 2, tg = lane & 3;
  float c[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) c[mt][0] = c[mt][1] = c[mt][2] = c[mt][3] = 0.f;
  const bool bn = g < cols_b;
#pragma unroll 1
  for (int k0 = warp * 16; k0 < K; k0 += SV_WARPS * 16) {
    const uint32_t b0 = bn ? ld_pair(B + (long long)g * ldb + k0 + 2 * tg) : 0u;
    const uint32_t b1 = bn ? ld_pair(B + (long long)g * ldb + k0 + 8 + 2 * tg) : 0u;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int r0 = mt * 16 + g, r1 = r0 + 8;
      const uint16_t* p0 = A + (long long)r0 * lda + k0 + 2 * tg;
      const uint16_t* p1 = A + (long long)r1 * lda + k0 + 2 * tg;
      const uint32_t a0 = r0 < rows_a ? ld_pair(p0) : 0u, a2 = r0 < rows_a ? ld_pair(p0 + 8) : 0u;
      const uint32_t a1 = r1 < rows_a ? ld_pair(p1) : 0u, a3 = r1 < rows_a ? ld_pair(p1 + 8) : 0u;
      mma16816(c[mt], a0, a1, a2, a3, b0, b1);
    }
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    float* t = red + ((long long)warp * MT + mt) * 128;
    t[g * 8 + 2 * tg] = c[mt][0];
    t[g * 8 + 2 * tg + 1] = c[mt][1];
    t[(g + 8) * 8 + 2 * tg] = c[mt][2];
    t[(g + 8) * 8 + 2 * tg + 1] = c[mt][3];
  }
}

__global__ void __launch_bounds__(SV_THREADS, 1) serve_kernel(const __grid_constant__ ServeParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  // Copies: the CTA's W_r rows or shared gate/up rows (a), its shared down rows (d), the
  // tokens (x), its rows of the routed experts' down projections (r).
  __shared__ __align__(8) uint64_t bar_a, bar_d, bar_x, bar_r, bar_g;
  __shared__ int s_ok, s_nu, s_rarmed, s_garmed, s_allhit;
  __shared__ int s_idx[SV_MAXT], s_ue[SV_MAXT], s_pu[SV_MAXT];  // selection; distinct experts; pair -> distinct
  __shared__ int s_we[SV_MAXT];  // where each distinct expert's weights are: the expert, or its cache slot
  __shared__ CachePlanScratch plan_sc;
  __shared__ float s_gate[SV_MAXT];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int c = blockIdx.x, G = gridDim.x;
  const int T = p.T, d = p.d, E = p.E, f = p.f, F = p.F, k = p.k, P = p.T * p.k;
  const bool router = c < p.R;
  const int e0 = c * p.epc, e1 = router ? min(E, e0 + p.epc) : e0;
  const bool shared = F > 0 && c >= p.R && c < p.R + p.nSG;
  const int j0 = (c - p.R) * p.U;  // first shared hidden unit of a shared CTA
  const int i0 = min(d, c * p.RD), i1 = min(d, i0 + p.RD);
  uint16_t* const xs = reinterpret_cast<uint16_t*>(sm + p.o_x);
  float* const bs = reinterpret_cast<float*>(sm + p.o_b);      // the bias as the call found it
  float* const sc = reinterpret_cast<float*>(sm + p.o_lg);     // [T][E] scores
  float* const key = sc + T * E;                                // [T][E] selection keys
  int* const hist = reinterpret_cast<int*>(sm + p.o_hist);
  int* const cnt_router = p.sync;
  int* const cnt_done = p.sync + 1;
  unsigned long long* const ready = reinterpret_cast<unsigned long long*>(p.sync + 2);
  int* const planned = p.sync + 4;
  int* const cnt_filled = p.sync + 5;
  int* const plan_njobs = p.sync + 6;
  const uint32_t rd_codes = (uint32_t)(i1 - i0) * (f / 2), rd_bytes = rd_codes + (uint32_t)(i1 - i0) * (f / 16);
  const uint32_t item_bytes = (uint32_t)d + (uint32_t)d / 8;  // gate and up codes (d / 2 each), scales (d / 16 each)

  if (tid == 0) {
    s_rarmed = 0;
    s_garmed = 0;
    mbar_init(smem_u32(&bar_a), 1);
    mbar_init(smem_u32(&bar_d), 1);
    mbar_init(smem_u32(&bar_x), 1);
    mbar_init(smem_u32(&bar_r), 1);
    mbar_init(smem_u32(&bar_g), 1);
    fence_mbar_init();
  }
  __syncthreads();
  {
    // Weights are inputs no earlier kernel of the call writes: copied before the wait.
    // One copy per thread (a copy takes tens of ns to issue); thread 0 alone arrives on
    // each barrier, with the byte count of all its copies (completions may come first).
    const uint32_t ab = smem_u32(&bar_a), db = smem_u32(&bar_d), wa = smem_u32(sm + p.o_w);
    const uint32_t rbytes = router ? (uint32_t)(e1 - e0) * d * 4u : 0u;
    const int srows = shared ? 2 * p.U : 0, drows = F > 0 ? i1 - i0 : 0;
    if (tid == 0) {
      mbar_arrive_expect_tx(ab, rbytes + (uint32_t)srows * d * 2u);
      mbar_arrive_expect_tx(db, (uint32_t)drows * F * 2u);
      if (rbytes) bulk_load(wa, p.w_router + (long long)e0 * d, rbytes, ab);
    }
    if (tid < srows) {
      // Rows SR apart: U gate rows, then the U matching up rows.
      const long long rg = (long long)(j0 / p.bF) * 2 * p.bF + j0 % p.bF;
      const long long src = tid < p.U ? rg + tid : rg + p.bF + (tid - p.U);
      bulk_load(wa + (uint32_t)tid * p.SR * 2u, p.s_gu + src * d, (uint32_t)d * 2u, ab);
    }
    if (tid >= 64 && tid - 64 < drows)
      bulk_load(smem_u32(sm + p.o_sdn) + (uint32_t)(tid - 64) * p.SD * 2u, p.s_dn + (long long)(i0 + tid - 64) * F,
                (uint32_t)F * 2u, db);
  }
  pdl_wait();  // x, the bias, the residual and the workspace's last use come before
  pdl_trigger();
  if (c == 0 && tid == 0) {
    // The call's counters start at zero; `ready` = this call's id publishes that.
    *cnt_router = 0;
    *cnt_done = 0;
    *planned = 0;
    *cnt_filled = 0;
    __threadfence();
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(ready), "l"(p.call_id) : "memory");
  }
  if (tid == 0) mbar_arrive_expect_tx(smem_u32(&bar_x), (uint32_t)T * d * 2u);
  if (tid >= 96 && tid - 96 < T)
    bulk_load(smem_u32(xs) + (uint32_t)(tid - 96) * p.SX * 2u, p.x + (long long)(tid - 96) * d, (uint32_t)d * 2u,
              smem_u32(&bar_x));
  for (int e = tid; e < E; e += SV_THREADS) bs[e] = p.bias[e];
  if (tid == 0)
    s_ok = mbar_wait(smem_u32(&bar_x), 0, p.status) && mbar_wait(smem_u32(&bar_a), 0, p.status) ? 1 : 0;
  __syncthreads();
  int ok = s_ok;

  // ---------------------------------------------------------------- 1. router logits
  if (router && ok) {
    // The cluster router's per-lane order (lane l: elements 4l + 128i, i ascending) and
    // reduction, so both paths give the same logits.
    const float* wr = reinterpret_cast<const float*>(sm + p.o_w);
    // (expert, token) pairs dealt over the warps.
    for (int task = warp; task < (e1 - e0) * T; task += SV_WARPS) {
      const int el = task / T, t = task % T;
      const float off = p.logit_offset ? p.logit_offset[e0 + el] : 0.f;
      {
        float acc = 0.f;
#pragma unroll 1
        for (int c4 = lane; c4 < d / 4; c4 += 32) {
          const float4 w = reinterpret_cast<const float4*>(wr + (long long)el * d)[c4];
          const uint2 xv = reinterpret_cast<const uint2*>(xs + (long long)t * p.SX)[c4];
          acc = fmaf(w.x, bf_lo(xv.x), fmaf(w.y, bf_hi(xv.x), fmaf(w.z, bf_lo(xv.y), fmaf(w.w, bf_hi(xv.y), acc))));
        }
        acc = warp_sum(acc);
        if (lane == 0) p.logits[(long long)t * E + e0 + el] = acc + off;
      }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      ok = spin_eq64(ready, p.call_id, p.status);
      if (ok) atomicAdd(cnt_router, 1);
      s_ok = ok;
    }
    __syncthreads();
    ok = s_ok;
  }

  // ---------------------------------------------------------------- 2. shared gate/up
  if (shared && ok) {
    // [2U rows] x [T tokens] over d on the tensor cores (mma.sync, K split over the
    // warps), then the SwiGLU of each (gate row, up row) pair.
    const uint16_t* rows = reinterpret_cast<const uint16_t*>(sm + p.o_w);
    float* red = reinterpret_cast<float*>(sm + p.o_red);
    switch (p.MT) {
      case 1: mma_rows_x_tokens<1>(rows, p.SR, 2 * p.U, xs, p.SX, T, d, red, warp, lane); break;
      case 2: mma_rows_x_tokens<2>(rows, p.SR, 2 * p.U, xs, p.SX, T, d, red, warp, lane); break;
      case 3: mma_rows_x_tokens<3>(rows, p.SR, 2 * p.U, xs, p.SX, T, d, red, warp, lane); break;
      default: mma_rows_x_tokens<4>(rows, p.SR, 2 * p.U, xs, p.SX, T, d, red, warp, lane); break;
    }
    __syncthreads();
    for (int i = tid; i < p.U * T; i += SV_THREADS) {
      const int ju = i / T, t = i % T, mu = p.U + ju;
      float g = 0.f, u = 0.f;
      for (int w = 0; w < SV_WARPS; ++w) {
        g += red[((w * p.MT) + ju / 16) * 128 + (ju % 16) * 8 + t];
        u += red[((w * p.MT) + mu / 16) * 128 + (mu % 16) * 8 + t];
      }
      p.hs[(long long)t * F + j0 + ju] = bf16_bits(swiglu(g, u));
    }
  }

  // ---------------------------------------------------------------- 3. selection
  // Every CTA selects for itself from the logits all router CTAs wrote (the same
  // deterministic result everywhere); CTA 0 writes the routing outputs.
  if (tid == 0) s_ok = ok && spin_eq64(ready, p.call_id, p.status) && spin_geq(cnt_router, p.R, p.status);
  __syncthreads();
  ok = s_ok;
  if (ok) {
    for (int i = tid; i < T * E; i += SV_THREADS) {
      const float z = __ldcg(p.logits + i);
      const float sv = 1.0f / (1.0f + expf(-z));
      sc[i] = sv;
      key[i] = __fadd_rn(sv, bs[i % E]);  // the selection key: one fp32 addition
      if (c == 0 && p.scores) p.scores[i] = sv;
    }
    for (int e = tid; e < E; e += SV_THREADS) hist[e] = 0;
    __syncthreads();
    if (warp < T) {
      // Token `warp`: k rounds of a warp arg-max under (key descending, expert index
      // ascending); lane l holds experts l, l + 32, ...
      const int t = warp;
      constexpr int NONE = 0x7FFFFFFF;
      unsigned taken = 0;
      float denom = 0.f;
#pragma unroll 1
      for (int j = 0; j < k; ++j) {
        float bk = -INFINITY;
        int be = NONE;
#pragma unroll 1
        for (int i = 0, e = lane; e < E; ++i, e += 32) {
          const float kv = key[t * E + e];
          if (!((taken >> i) & 1u) && (be == NONE || kv > bk)) {
            bk = kv;
            be = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float okv = __shfl_xor_sync(FULLM, bk, o);
          const int oe = __shfl_xor_sync(FULLM, be, o);
          if (oe != NONE && (be == NONE || okv > bk || (okv == bk && oe < be))) {
            bk = okv;
            be = oe;
          }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        const float sv = sc[t * E + be];
        denom += sv;
        if (lane == 0) {
          s_idx[t * k + j] = be;
          s_gate[t * k + j] = sv;
          atomicAdd(&hist[be], 1);
        }
      }
      __syncwarp();
      if (lane < k && p.renorm) s_gate[t * k + lane] = __fdiv_rn(s_gate[t * k + lane], denom);
    }
    __syncthreads();
    if (warp == 0) {
      // Distinct experts in order of first appearance; each pair's distinct index (pair q
      // in lane q, P <= 32; every lane takes part in the match and the ballot).
      const int e = lane < P ? s_idx[lane] : -1 - lane;
      const unsigned same = __match_any_sync(FULLM, e);
      const int first = __ffs(same) - 1;  // the first pair with this lane's expert
      const unsigned firsts = __ballot_sync(FULLM, lane < P && first == lane);
      const int u = __popc(firsts & ((1u << first) - 1u));
      if (lane < P) s_pu[lane] = u;
      if (lane < P && first == lane) s_ue[u] = s_we[u] = e;
      if (lane == 0) s_nu = __popc(firsts);
    }
    __syncthreads();
    if (c == 0) {
      for (int q = tid; q < P; q += SV_THREADS) {
        p.idx[q] = s_idx[q];
        p.gate[q] = s_gate[q];
      }
      for (int e = tid; e < E; e += SV_THREADS)
        if (p.load) p.load[e] = hist[e];
      if (p.balance && warp == SV_WARPS - 1) warp_balance(hist, E, p.balance, lane);
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- 3b. expert cache
  // Every CTA reads where the step's experts are in the tables as the call found them:
  // CTA 0 writes the step's new tables back only after the last grid barrier, so all
  // CTAs see the same table and take the same branch.  A hit's slot cannot change in its
  // own step.  When every expert of the step is resident nothing waits for the plan;
  // otherwise CTA 0 publishes the plan's copies, every CTA copies its share of the
  // missing experts from host memory into their slots, and a counted barrier ends the
  // phase.
  if (p.cached && ok) {
    if (tid == 0) {
      int all = 1;
      for (int u = 0; u < s_nu; ++u) {
        s_we[u] = __ldcg(p.expert_slot + s_ue[u]);
        if (s_we[u] < 0 || s_we[u] >= p.slots) all = 0;
      }
      s_allhit = all;
    }
    __syncthreads();
    const bool all_hit = s_allhit != 0;
    if (c == 0) {
      if (warp == 0)
        cache_plan_warp(s_idx, P, E, p.slots, p.cstate, p.slot_expert, p.cstamp, p.expert_slot, p.jobs,
                        p.expert_bytes, p.status, plan_sc, lane, [] {});
      if (!all_hit) {
        __syncthreads();
        if (tid == 0) {
          *plan_njobs = plan_sc.next.njobs;
          __threadfence();
          asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(planned), "r"(1) : "memory");
        }
      }
    }
    if (!all_hit) {
      if (tid == 0) s_ok = spin_geq(planned, 1, p.status) ? 1 : 0;
      __syncthreads();
      ok = s_ok;
      if (ok) {
        const int njobs = __ldcg(plan_njobs);
        cache_copy_range(njobs, p.jobs, p.host_src, p.slots_w, (long long)c * SV_THREADS + tid,
                         (long long)G * SV_THREADS);
        // The copies are read next by bulk copies (the async proxy) of other CTAs.
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        __syncthreads();
        if (tid == 0) {
          atomicAdd(cnt_filled, 1);
          s_ok = spin_geq(cnt_filled, G, p.status) ? 1 : 0;
          asm volatile("fence.proxy.async.global;" ::: "memory");
          // The missing experts' slots, from the plan's copies.
          for (int u = 0; u < s_nu; ++u) {
            if (s_we[u] >= 0 && s_we[u] < p.slots) continue;
            s_we[u] = -1;
            for (int jb = 0; jb < njobs; ++jb) {
              const int2 job = p.jobs[jb];
              if (job.x == s_ue[u]) s_we[u] = job.y;
            }
            if (s_we[u] < 0 || s_we[u] >= p.slots) {  // not served (the plan ran out of slots)
              atomicOr(p.status, kDevCheck);
              s_ok = 0;
            }
          }
        }
        __syncthreads();
        ok = s_ok;
      }
    }
  }

  // ---------------------------------------------------------------- prefetch of the
  // routed weights this CTA needs: its routed gate/up items (into the now idle weight
  // slice region) and its output rows of the experts' down projections
  if (ok) {
    if (tid == 0) {
      mbar_arrive_expect_tx(smem_u32(&bar_r), i1 > i0 ? (uint32_t)s_nu * rd_bytes : 0u);
      s_rarmed = 1;
      const long long items = (long long)s_nu * f;
      const int mine = items > c ? (int)((items - c + G - 1) / G) : 0;
      mbar_arrive_expect_tx(smem_u32(&bar_g), (uint32_t)mine * (uint32_t)item_bytes);
      s_garmed = 1;
    }
    // The region was last read by generic loads; the copies write it through the async proxy.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    {
      // Item m of this CTA is global item c + G m; thread i issues copy i % 4 of item i / 4.
      const long long items = (long long)s_nu * f;
      const int mine = items > c ? (int)((items - c + G - 1) / G) : 0;
      for (int i = tid; i < 4 * mine; i += SV_THREADS) {
        const int m = i >> 2, part = i & 3;
        const long long it = c + (long long)G * m;
        const int u = (int)(it / f), j = (int)(it % f);
        const long long rg = (long long)s_we[u] * 2 * f + (j / p.bf) * 2 * p.bf + j % p.bf;
        const long long row = (part & 1) ? rg + p.bf : rg;  // gate, up
        // Codes of gate, up at 0, d / 2; scales of gate, up at d, d + d / 16.
        const uint32_t off = (part & 2) ? (uint32_t)d + (part & 1) * (uint32_t)(d / 16) : (part & 1) * (uint32_t)(d / 2);
        const uint32_t dst = smem_u32(sm + p.o_w) + (uint32_t)m * item_bytes + off;
        if (part & 2)
          bulk_load(dst, p.gu_s + row * (d / 32), (uint32_t)d / 16, smem_u32(&bar_g));
        else
          bulk_load(dst, p.gu_q + row * (d / 2), (uint32_t)d / 2, smem_u32(&bar_g));
      }
    }
    if (warp == 0 && i1 > i0 && lane < 2 * s_nu) {
      const int u = lane >> 1;
      const long long row = (long long)s_we[u] * d + i0;
      const uint32_t dst = smem_u32(sm + p.o_rd) + (uint32_t)u * rd_bytes;
      if (lane & 1)
        bulk_load(dst + rd_codes, p.dn_s + row * (f / 32), rd_bytes - rd_codes, smem_u32(&bar_r));
      else
        bulk_load(dst, p.dn_q + row * (f / 2), rd_codes, smem_u32(&bar_r));
    }
  }

  // ---------------------------------------------------------------- 4. routed gate/up
  if (ok) {
    if (tid == 0) s_ok = mbar_wait(smem_u32(&bar_g), 0, p.status) ? 1 : 0;
    __syncthreads();
    ok = s_ok;
  }
  if (ok) {
    const int ng = d / 32;
    const long long items = (long long)s_nu * f;
    const int mine = items > c ? (int)((items - c + G - 1) / G) : 0;
    // Item m (global item c + G m: hidden unit j of distinct expert u), for each of the
    // expert's pairs, from its rows in shared memory: gate codes, up codes, gate
    // scales, up scales.
    for (int m = warp; m < mine; m += SV_WARPS) {
      const long long it = c + (long long)G * m;
      const int u = (int)(it / f), j = (int)(it % f);
      const uint8_t* base = sm + p.o_w + (long long)m * item_bytes;
      const uint16_t* sgs = reinterpret_cast<const uint16_t*>(base + d);
      const uint16_t* sus = sgs + ng;
#pragma unroll 1
      for (int q = 0; q < P; ++q) {
        if (s_pu[q] != u) continue;
        const uint16_t* xt = xs + (long long)(q / k) * p.SX;
        float ag = 0.f, au = 0.f;
#pragma unroll 1
        for (int g = lane; g < ng; g += 32) {
          const uint4 cg = *reinterpret_cast<const uint4*>(base + g * 16);
          const uint4 cu = *reinterpret_cast<const uint4*>(base + d / 2 + g * 16);
          ag = fmaf(__half2float(__ushort_as_half(sgs[g])), group_qdot(cg, xt + g * 32), ag);
          au = fmaf(__half2float(__ushort_as_half(sus[g])), group_qdot(cu, xt + g * 32), au);
        }
        ag = warp_sum(ag);
        au = warp_sum(au);
        if (lane == 0) p.h[(long long)q * f + j] = bf16_bits(swiglu(ag, au));
      }
    }
  }

  // ---------------------------------------------------------------- grid barrier
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const bool mine = ok;
    if (mine) atomicAdd(cnt_done, 1);
    s_ok = mine && spin_geq(cnt_done, G, p.status);
    if (s_ok && i1 > i0)
      s_ok = mbar_wait(smem_u32(&bar_d), 0, p.status) && mbar_wait(smem_u32(&bar_r), 0, p.status) ? 1 : 0;
  }
  __syncthreads();
  ok = s_ok;
  // Every CTA has read the cache's tables for this step: the plan's tables can go in.
  if (ok && c == 0 && p.cached && warp == 0)
    cache_plan_write_back(plan_sc, E, p.slots, p.cstate, p.slot_expert, p.cstamp, p.expert_slot, lane);
  // Every CTA has read the bias for its selection: the update can go in.
  if (ok && c == 0 && p.update_bias)
    for (int e = tid; e < E; e += SV_THREADS) p.bias[e] = biased_step(bs[e], (long long)T * k, E, hist[e], p.gamma);

  // ---------------------------------------------------------------- 5. output rows
  if (ok && i1 > i0) {
    uint16_t* hss = reinterpret_cast<uint16_t*>(sm + p.o_hs);  // [T] rows SH apart
    uint16_t* hh = reinterpret_cast<uint16_t*>(sm + p.o_h);
    float* red = reinterpret_cast<float*>(sm + p.o_red);
    const int nr = i1 - i0;
    for (int i = tid; i < T * F / 8; i += SV_THREADS) {
      const int t = i / (F / 8), c8 = i % (F / 8);
      reinterpret_cast<uint4*>(hss + (long long)t * p.SH)[c8] = __ldcg(reinterpret_cast<const uint4*>(p.hs) + i);
    }
    for (int i = tid; i < P * f / 8; i += SV_THREADS)
      reinterpret_cast<uint4*>(hh)[i] = __ldcg(reinterpret_cast<const uint4*>(p.h) + i);
    __syncthreads();
    // S = the shared down rows [nr <= 16] x hs [T] over F, on the tensor cores.
    if (F > 0)
      mma_rows_x_tokens<1>(reinterpret_cast<const uint16_t*>(sm + p.o_sdn), p.SD, nr, hss, p.SH, T, F, red, warp,
                           lane);
    __syncthreads();
    const int ng = f / 32;
    // Each half-warp takes one token of the row at a time (two in flight per warp): its 16
    // lanes share the row's groups and reduce among themselves.  The token loop is the
    // same for the whole warp, so every lane reaches each shuffle.
    const int half = lane >> 4, hl = lane & 15;
    for (int r = i0 + warp; r < i1; r += SV_WARPS) {
#pragma unroll 1
      for (int t0 = 0; t0 < T; t0 += 2) {
        const int t = t0 + half;
        const bool tv = t < T;
        float o = 0.f;
        if (F > 0 && tv)
          for (int w = 0; w < SV_WARPS; ++w) o += red[w * 128 + (r - i0) * 8 + t];
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
          const int q = (tv ? t : 0) * k + j;
          const uint8_t* rows = sm + p.o_rd + s_pu[q] * rd_bytes;  // this expert's prefetched rows
          const uint8_t* codes = rows + (r - i0) * (f / 2);
          const uint16_t* scales = reinterpret_cast<const uint16_t*>(rows + rd_codes) + (r - i0) * ng;
          float acc = 0.f;
#pragma unroll 1
          for (int g = hl; g < ng; g += 16)
            if (tv)
              acc = fmaf(__half2float(__ushort_as_half(scales[g])),
                         group_qdot(*reinterpret_cast<const uint4*>(codes + g * 16), hh + (long long)q * f + g * 32),
                         acc);
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(FULLM, acc, off);
          const float y = bf16_round(acc);  // the routed output is stored in bf16
          o = fmaf(s_gate[q], y, o);
        }
        if (hl == 0 && tv) {
          if (p.residual) o += __bfloat162float(__ushort_as_bfloat16(p.residual[(long long)t * d + r]));
          p.out[(long long)t * d + r] = bf16_bits(o);
        }
      }
    }
  }
  // After a timeout: no copy may still be landing when the CTA exits (bounded waits).
  if (tid == 0 && !ok) {
    mbar_wait(smem_u32(&bar_d), 0, p.status);
    if (s_rarmed) mbar_wait(smem_u32(&bar_r), 0, p.status);
    if (s_garmed) mbar_wait(smem_u32(&bar_g), 0, p.status);
  }
}

// SM count of the current device, queried once per device.
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

struct ServePlan {
  int G, R, epc, U, nSG, RD, bF;
  int MT, SX, SR, SD, SH;
  int o_x, o_w, o_sdn, o_hs, o_h, o_lg, o_hist, o_rd, o_b, o_red, smem;
};

size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }

bool plan_serve(const moe_shape_t* s, ServePlan* pl) {
  const long long P = (long long)s->T * s->k;
  if (s->w_format != MOE_W_INT4_G32 || s->x_dtype != MOE_X_BF16 || P < 1 || P > kServeMaxPairs) return false;
  // d % 256, f % 256: a row's fp16 scales are a multiple of 16 bytes (bulk copies).
  if (s->d % 256 || s->f % 256 || (s->F && s->F % 8) || s->E > kMaxE) return false;
  const int sms = sm_count();
  if (sms < 8) return false;
  ServePlan q{};
  q.G = sms;
  q.R = std::min(SV_ROUTER_CTAS, s->E);
  q.epc = (s->E + q.R - 1) / q.R;
  q.R = (s->E + q.epc - 1) / q.epc;  // every router CTA has experts
  q.bF = s->F ? moe_gate_up_block(s->F) : 1;
  q.U = 0;
  q.nSG = 0;
  if (s->F) {
    const int avail = q.G - q.R;
    int u = 1;
    while ((long long)u * avail < s->F) u *= 2;
    if (u > q.bF || q.bF % u || 2 * u > 64) return false;  // at most four 16-row tiles
    q.U = u;
    q.nSG = s->F / u;
  }
  q.MT = std::max(1, (2 * q.U + 15) / 16);
  q.RD = (s->d + q.G - 1) / q.G;
  if (q.RD > 16) return false;  // one 16-row tile of output rows per CTA
  // Rows 16 bytes longer than their data: a warp's fragment loads hit distinct banks.
  q.SX = s->d + 8;
  q.SR = s->d + 8;
  q.SD = s->F + 8;
  q.SH = s->F + 8;
  size_t off = 0;
  q.o_x = (int)off;
  off += align16((size_t)s->T * q.SX * 2);
  q.o_w = (int)off;
  {
    // The weight slice region: W_r rows or shared gate/up rows, later the CTA's routed
    // gate/up items (at most ceil(P f / G), d + d / 8 bytes each).
    const size_t items = ((size_t)P * s->f + q.G - 1) / q.G;
    off += align16(std::max({(size_t)q.epc * s->d * 4, (size_t)2 * q.U * q.SR * 2, items * (s->d + s->d / 8)}));
  }
  q.o_sdn = (int)off;
  off += align16((size_t)q.RD * q.SD * 2);
  q.o_hs = (int)off;
  off += align16((size_t)s->T * q.SH * 2);
  q.o_red = (int)off;  // per warp and 16-row tile, a 16 x 8 fp32 partial product
  off += (size_t)SV_WARPS * q.MT * 128 * 4;
  q.o_h = (int)off;
  off += align16((size_t)P * s->f * 2);
  q.o_lg = (int)off;
  off += align16((size_t)2 * s->T * s->E * 4);  // scores, then keys
  q.o_hist = (int)off;
  off += align16((size_t)s->E * 4);
  q.o_b = (int)off;
  off += align16((size_t)s->E * 4);
  q.o_rd = (int)off;  // per distinct expert: the CTA's down rows (codes, then scales)
  off += (size_t)P * q.RD * (s->f / 2 + s->f / 16);
  if (off > kServeMaxSmem) return false;
  q.smem = (int)off;
  *pl = q;
  return true;
}

}  // namespace

bool serve_fused_supported(const moe_shape_t* s, const void* x, const float* w_router, const moe_weights_t* w) {
  ServePlan pl;
  if (!plan_serve(s, &pl)) return false;
  // The bulk copies read x, W_r and the shared expert's rows from 16-byte boundaries.
  auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  return a16(x) && a16(w_router) && a16(w->w_gate_up) && a16(w->scale_gate_up) && a16(w->w_down) &&
         a16(w->scale_down) &&
         (s->F == 0 || (a16(w->shared_gate_up) && a16(w->shared_down)));
}

size_t serve_fused_scratch_bytes(const moe_shape_t* s) {
  // logits [T][E] fp32, then the eight sync words.
  return align16((size_t)s->T * s->E * 4) + 32;
}

cudaError_t launch_serve_fused(const moe_shape_t* s, const ServeArgs& a, cudaStream_t st) {
  ServePlan pl;
  if (!plan_serve(s, &pl)) return cudaErrorInvalidValue;
  ServeParams p{};
  p.x = static_cast<const uint16_t*>(a.x);
  p.w_router = a.w_router;
  p.logit_offset = a.logit_offset;
  p.bias = a.bias;
  p.gu_q = static_cast<const uint8_t*>(a.w->w_gate_up);
  p.gu_s = static_cast<const uint16_t*>(a.w->scale_gate_up);
  p.dn_q = static_cast<const uint8_t*>(a.w->w_down);
  p.dn_s = static_cast<const uint16_t*>(a.w->scale_down);
  p.s_gu = static_cast<const uint16_t*>(a.w->shared_gate_up);
  p.s_dn = static_cast<const uint16_t*>(a.w->shared_down);
  p.residual = static_cast<const uint16_t*>(a.residual);
  p.out = a.out;
  p.scores = a.scores;
  p.idx = a.idx;
  p.gate = a.gate;
  p.load = a.load;
  p.balance = a.balance;
  p.logits = static_cast<float*>(a.scratch);
  p.sync = reinterpret_cast<int*>(static_cast<uint8_t*>(a.scratch) + align16((size_t)s->T * s->E * 4));
  p.hs = a.hs;
  p.h = a.h;
  if (a.cache_view) {
    p.cached = 1;
    p.slots = a.cache_slots;
    p.cstate = a.cache_view->state;
    p.slot_expert = a.cache_view->slot_expert;
    p.cstamp = a.cache_view->stamp;
    p.expert_slot = a.cache_view->expert_slot;
    p.jobs = a.cache_view->jobs;
    p.slots_w = a.cache_view->slots_w;
    p.host_src = *a.cache_src;
    p.expert_bytes = a.cache_expert_bytes;
  }
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;
  p.T = s->T;
  p.d = s->d;
  p.E = s->E;
  p.f = s->f;
  p.F = s->F;
  p.k = s->k;
  p.renorm = s->renorm;
  p.update_bias = a.update_bias;
  p.bf = moe_gate_up_block(s->f);
  p.bF = pl.bF;
  p.gamma = a.gamma;
  p.R = pl.R;
  p.epc = pl.epc;
  p.U = pl.U;
  p.nSG = pl.nSG;
  p.RD = pl.RD;
  p.o_x = pl.o_x;
  p.o_w = pl.o_w;
  p.o_sdn = pl.o_sdn;
  p.o_hs = pl.o_hs;
  p.o_h = pl.o_h;
  p.o_lg = pl.o_lg;
  p.o_hist = pl.o_hist;
  p.o_rd = pl.o_rd;
  p.o_b = pl.o_b;
  p.o_red = pl.o_red;
  p.MT = pl.MT;
  p.SX = pl.SX;
  p.SR = pl.SR;
  p.SD = pl.SD;
  p.SH = pl.SH;
  // A different id for every call in the process: the counters' zeroing by CTA 0 is
  // recognised by it, so the workspace needs no clearing between calls.
  static std::atomic<unsigned long long> next_id{0x5e7a11c0de000001ull};
  p.call_id = next_id.fetch_add(1);
  // The kernel's shared-memory limit, raised once per device to the largest plan.
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(serve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kServeMaxSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  return launch_pdl(serve_kernel, dim3((unsigned)pl.G), dim3(SV_THREADS), (size_t)pl.smem, st, p);
}

}  // namespace moe
