// Router on tcgen05 tensor cores for bf16 tokens.
//
// Relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B de
// NanoColibri por $200"), opening section, architecture paragraph: sigmoid-plus-bias
// router with top-k routing; section "Entrenamiento por relevos", top-2 paragraph:
// gates renormalised over the winners.
//
// The router weight is fp32.  It is split exactly into three bf16 parts,
// W = W_hi + W_mid + W_lo (each part the bf16 rounding of what the previous parts
// left), stored as one [3E][d] matrix.  Token values are bf16, so every product
// x * W_part is exact in fp32 and the tensor core accumulates in fp32: the logits
// carry fp32 accuracy (no reduced-precision weights, no TF32).  One CTA owns 128
// tokens: a TMA producer streams 128-wide k-blocks of the tokens (128 x 128) and of
// the weights (3E x 128), one 3-D copy of two 64-column swizzle atoms per operand,
// through a 2-stage ring (the CTA's whole token slab is prefetched into L2 first;
// copies of 32-48 KB cost far less TMA issue time per byte than 16-24 KB ones),
// one thread issues tcgen05.mma (M = 128, N = 3E, K = 16) into TMEM, and then two
// threads per token read its 3E accumulator columns (one half of the experts
// each), form the logits, apply the sigmoid, keep their best k by fl32(score +
// bias) with ties to the lower index, and merge the two lists; the gates and the
// per-warp shared-memory histogram follow.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int RBM = 128;
constexpr int RAT = 64;           // K width of one 128-byte swizzle atom
constexpr int RBK = 2 * RAT;      // K per stage: two atoms in one copy per operand
constexpr int RSTAGES = 2;
constexpr int A_ATOM = RBM * RAT * 2;
constexpr int A_BYTES = 2 * A_ATOM;
constexpr int RTHREADS = 256;  // 8 warps: two threads per token in the epilogue
constexpr unsigned FULL = 0xFFFFFFFFu;

struct RouterTcParams {
  CUtensorMap x_map;  // [T][d] bf16 as (64, T, d / 64), box (64, 128, 2)
  CUtensorMap w_map;  // [3E][d] bf16 as (64, 3E, d / 64), box (64, 3E, 2)
  const float* logit_offset;
  const float* bias;
  float* scores;
  int32_t* idx;
  float* gate;
  int32_t* load;
  int32_t* counts;
  int* status;
  int chunk_tokens, T, d, k, renorm, stage_bytes;
};

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

template <int E>
__global__ void __launch_bounds__(RTHREADS, 1) router_tc_kernel(const __grid_constant__ RouterTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[RSTAGES];
  __shared__ __align__(8) uint64_t empty_bar[RSTAGES];
  __shared__ __align__(8) uint64_t tfull_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ float s_bias[E];
  __shared__ float s_off[E];
  __shared__ int hist[4][E];
  __shared__ float cand_key[2][RBM][kMaxK];
  __shared__ int cand_e[2][RBM][kMaxK];
  __shared__ float cand_s[2][RBM][kMaxK];

  constexpr int N = 3 * E;
  constexpr uint32_t TCOLS = N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256));
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t0 = blockIdx.x * RBM;

  for (int i = threadIdx.x; i < 4 * E; i += RTHREADS) (&hist[0][0])[i] = 0;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < RSTAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&tfull_bar), 1);
    fence_mbar_init();
    tma_prefetch_desc(&p.x_map);
    tma_prefetch_desc(&p.w_map);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), TCOLS);
    tmem_relinquish();
  }
  // Everything above is CTA-local; from here on the kernel reads the bias (updated
  // by the previous forward), the split weights and the tokens.
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += RTHREADS) {
    s_bias[e] = p.bias[e];
    s_off[e] = p.logit_offset ? p.logit_offset[e] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;
  const int nkb = (p.d + RBK - 1) / RBK;  // a ragged last atom arrives zero-filled
  constexpr uint32_t W_ATOM = (uint32_t)N * RAT * 2;

  if (warp == 0 && lane == 0) {
    // The token slab is read once, from DRAM: ask for all of it up front so the
    // ring below is fed from L2 instead of paying DRAM latency per stage.
    for (int kb = 0; kb < nkb; ++kb) tma_prefetch_l2_3d(&p.x_map, 0, t0, 2 * kb);
    const uint32_t bytes = A_BYTES + 2 * W_ATOM;
    uint32_t issued = 0, last_par = 0;
    int stage = 0;
    uint32_t phase = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      if (!mbar_wait_spin(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) break;
      const uint32_t sa = ring + stage * p.stage_bytes;
      const uint32_t fb = smem_u32(&full_bar[stage]);
      mbar_arrive_expect_tx(fb, bytes);
      tma_load_3d(sa, &p.x_map, fb, 0, t0, 2 * kb);
      tma_load_3d(sa + A_BYTES, &p.w_map, fb, 0, 0, 2 * kb);
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == RSTAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    for (int s = 0; s < RSTAGES; ++s)
      if ((issued >> s) & 1u) mbar_wait_spin(smem_u32(&full_bar[s]), (last_par >> s) & 1u, p.status);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(RBM, N);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int kb = 0; kb < nkb && ok; ++kb) {
      if (!mbar_wait_spin(smem_u32(&full_bar[stage]), phase, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sa = ring + stage * p.stage_bytes;
      const uint64_t adesc = sw128_kmajor_desc(sa);
      const uint64_t bdesc = sw128_kmajor_desc(sa + A_BYTES);
#pragma unroll
      for (int kk = 0; kk < RBK / 16; ++kk)  // atom kk / 4, 32 bytes per K step inside it
        tc_mma_bf16(tmem_base, adesc + (kk >> 2) * (A_ATOM >> 4) + 2 * (kk & 3),
                    bdesc + (kk >> 2) * (W_ATOM >> 4) + 2 * (kk & 3), idesc, (kb | kk) != 0);
      tc_commit(smem_u32(&empty_bar[stage]));
      if (++stage == RSTAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    tc_commit(smem_u32(&tfull_bar));  // also fires after a partial (timed-out) loop
  }
  __syncwarp();

  // ------------------------------------------------------------ per-token epilogue
  // Warps w and w + 4 own the same 32 TMEM lanes (tokens); warp w takes experts
  // [0, EH), warp w + 4 experts [EH, E).  Each thread forms its experts' scores,
  // keeps its best k by (key desc, index asc), and the two lists are merged.
  int ok = 1;
  if (lane == 0) ok = mbar_wait(smem_u32(&tfull_bar), 0, p.status) ? 1 : 0;
  ok = __shfl_sync(FULL, ok, 0);
  tc_fence_after();
  constexpr int EH = ((E / 2 + 15) / 16) * 16;
  const int q = warp & 3, h = warp >> 2;
  const int row = q * 32 + lane;
  const int t = t0 + row;
  const bool valid = ok && t < p.T;
  const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  const int e_lo = h ? EH : 0, e_hi = h ? E : EH;
  float s[EH];
#pragma unroll
  for (int c = 0; c < EH; c += 16) {
    if (e_lo + c < e_hi) {  // warp-uniform
      uint32_t hv[16], mv[16], lv[16];
      tmem_ld16(tl + e_lo + c, hv);
      tmem_ld16(tl + E + e_lo + c, mv);
      tmem_ld16(tl + 2 * E + e_lo + c, lv);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float z = (__uint_as_float(hv[i]) + __uint_as_float(mv[i])) + __uint_as_float(lv[i]) +
                        s_off[e_lo + c + i];
        // Branch-free sigmoid; saturates to exactly 0 / 1 for extreme logits.
        s[c + i] = __fdividef(1.0f, 1.0f + __expf(-z));
      }
    }
  }
  const int nmine = e_hi - e_lo;
  const int kk = min(p.k, nmine);
  if (valid) {
    if (p.scores) {
      float4* dst = reinterpret_cast<float4*>(p.scores + (size_t)t * E + e_lo);
#pragma unroll
      for (int i = 0; i < EH / 4; ++i)
        if (4 * i < nmine) dst[i] = make_float4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
    }
    uint64_t taken = 0;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < kk) {
        float bk = -INFINITY, bs = 0.f;
        int be = -1;
#pragma unroll
        for (int i = 0; i < EH; ++i) {
          if (i < nmine && !((taken >> i) & 1ull)) {
            const float key = __fadd_rn(s[i], s_bias[e_lo + i]);
            if (be < 0 || key > bk) {
              bk = key;
              be = i;
              bs = s[i];
            }
          }
        }
        taken |= 1ull << be;
        cand_key[h][row][j] = bk;
        cand_e[h][row][j] = e_lo + be;
        cand_s[h][row][j] = bs;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (valid && h == 0) {
    const int na = min(p.k, EH), nb = min(p.k, E - EH);
    int ia = 0, ib = 0;
    float sel_s[kMaxK];
    int sel_e[kMaxK];
    float denom = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      sel_s[j] = 0.f;
      sel_e[j] = 0;
      if (j < p.k) {
        bool take_a;
        if (ia >= na) take_a = false;
        else if (ib >= nb) take_a = true;
        else {
          const float ka = cand_key[0][row][ia], kb = cand_key[1][row][ib];
          take_a = ka > kb || (ka == kb && cand_e[0][row][ia] < cand_e[1][row][ib]);
        }
        if (take_a) {
          sel_e[j] = cand_e[0][row][ia];
          sel_s[j] = cand_s[0][row][ia];
          ++ia;
        } else {
          sel_e[j] = cand_e[1][row][ib];
          sel_s[j] = cand_s[1][row][ib];
          ++ib;
        }
        denom += sel_s[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < p.k) {
        p.idx[(size_t)t * p.k + j] = sel_e[j];
        p.gate[(size_t)t * p.k + j] = p.renorm ? __fdiv_rn(sel_s[j], denom) : sel_s[j];
        atomicAdd(&hist[q][sel_e[j]], 1);
      }
    }
  }
  __syncthreads();
  // Each warp's 32 tokens lie in one permutation chunk (chunks are multiples of 32).
  for (int i = threadIdx.x; i < 4 * E; i += RTHREADS) {
    const int w = i / E, e = i % E;
    const int v = hist[w][e];
    if (v) {
      atomicAdd(&p.load[e], v);
      if (p.counts) atomicAdd(&p.counts[(size_t)((t0 + 32 * w) / p.chunk_tokens) * E + e], v);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TCOLS);
  }
}

// W (fp32 [E][d]) -> W3 (bf16 [3E][d]): rows [0,E) W_hi, [E,2E) W_mid, [2E,3E) W_lo with
// W_hi = bf16(W), W_mid = bf16(W - W_hi), W_lo = bf16(W - W_hi - W_mid); each
// difference is exact in fp32.
__global__ void split_router_kernel(const float* __restrict__ w, long long n, uint16_t* __restrict__ w3,
                                    int32_t* __restrict__ zero_a, int na, int32_t* __restrict__ zero_b,
                                    int nb) {
  pdl_wait();
  pdl_trigger();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < na) zero_a[i] = 0;
  if (i < nb) zero_b[i] = 0;
  if (i >= n) return;
  const float v = w[i];
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(mid);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
  w3[i] = __bfloat16_as_ushort(hi);
  w3[n + i] = __bfloat16_as_ushort(mid);
  w3[2 * n + i] = __bfloat16_as_ushort(lo);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// bf16 [outer][inner] viewed as (64 columns, outer rows, inner / 64 atoms), box (64,
// box_outer, 2): one copy = two consecutive 128-byte-swizzled atoms, box_outer * 128
// bytes apart (an atom past `inner` is zero-filled).
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn || inner % RAT != 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(RAT), outer, inner / RAT};
  const cuuint64_t strides[2] = {inner * 2, static_cast<cuuint64_t>(RAT) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(RAT), box_outer, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int E>
cudaError_t launch_e(RouterTcParams& p, int blocks, cudaStream_t s) {
  const int dyn = RSTAGES * p.stage_bytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<E>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  return launch_pdl(router_tc_kernel<E>, dim3(blocks), dim3(RTHREADS), dyn, s, p);
}

}  // namespace

bool router_tc_supported(int T, int E, int x_is_f32) {
  // One CTA per 128 tokens: below that the CUDA-core router (fp32 weights read
  // directly, no split launch) finishes sooner.
  return !x_is_f32 && T >= 128 && (E == 16 || E == 32 || E == 48 || E == 64 || E == 80);
}

size_t router_tc_scratch_bytes(int E, int d) { return (size_t)3 * E * d * sizeof(uint16_t); }

cudaError_t launch_router_tc(const RouterArgs& a, void* w3_scratch, cudaStream_t s) {
  const long long n = (long long)a.E * a.d;
  uint16_t* w3 = static_cast<uint16_t*>(w3_scratch);
  const int nb = a.counts ? ((a.T + a.chunk_tokens - 1) / a.chunk_tokens) * a.E : 0;
  const long long nthreads = std::max<long long>(n, std::max(a.E, nb));
  cudaError_t e = launch_pdl(split_router_kernel, dim3((unsigned)((nthreads + 255) / 256)), dim3(256), 0,
                             s, a.w_router, n, w3, a.load, a.E, a.counts, nb);
  if (e != cudaSuccess) return e;
  RouterTcParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_map(&p.x_map, a.x, a.d, a.T, RBM) || !make_map(&p.w_map, w3, a.d, 3 * a.E, 3 * a.E))
    return cudaErrorInvalidValue;
  p.logit_offset = a.logit_offset;
  p.bias = a.bias;
  p.scores = a.scores;
  p.idx = a.idx;
  p.gate = a.gate;
  p.load = a.load;
  p.counts = a.counts;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;
  p.chunk_tokens = a.chunk_tokens;
  p.T = a.T;
  p.d = a.d;
  p.k = a.k;
  p.renorm = a.renorm;
  p.stage_bytes = A_BYTES + 2 * 3 * a.E * RAT * 2;  // multiples of 1024 for E % 16 == 0
  const int blocks = (a.T + RBM - 1) / RBM;
  switch (a.E) {
    case 16: return launch_e<16>(p, blocks, s);
    case 32: return launch_e<32>(p, blocks, s);
    case 48: return launch_e<48>(p, blocks, s);
    case 64: return launch_e<64>(p, blocks, s);
    case 80: return launch_e<80>(p, blocks, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
