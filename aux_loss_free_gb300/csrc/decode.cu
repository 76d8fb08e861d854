// int4 container support for the top-1 serving path.
//
// Relay article, opening section, second paragraph: experts ship in an int4
// container.  Format (this library's reading): symmetric, groups of 32 consecutive
// input elements, fp16 scale = fp16(fl32(max|w| / 7)), code = clamp(rint(fl32(w /
// scale)), -7, 7) (0 where the scale is 0), two's-complement nibbles with the even
// index in the low nibble.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// One thread per group of 32 weights: 64 bytes in, 16 bytes of codes + 2 bytes out.
__global__ void quantize_int4_kernel(long long groups, const uint16_t* __restrict__ w,
                                     uint8_t* __restrict__ q, uint16_t* __restrict__ scale) {
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const uint4* src = reinterpret_cast<const uint4*>(w + g * 32);
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = src[i];
    const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(ws[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const __half sh = __float2half_rn(__fdiv_rn(amax, 7.0f));
  const float s = __half2float(sh);
  uint32_t packed[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    int c = 0;
    if (s > 0.f) c = (int)fminf(7.f, fmaxf(-7.f, rintf(__fdiv_rn(v[i], s))));
    packed[i / 8] |= (static_cast<uint32_t>(c) & 0xFu) << (4 * (i % 8));
  }
  reinterpret_cast<uint4*>(q + g * 16)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  scale[g] = __half_as_ushort(sh);
}

}  // namespace

cudaError_t launch_quantize_int4(long long rows, int K, const uint16_t* w, uint8_t* q,
                                 uint16_t* scale, cudaStream_t s) {
  const long long groups = rows * (K / 32);
  quantize_int4_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, s>>>(groups, w, q, scale);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------------
// Top-1 serving path: routed experts with int4 weights, dequantised in registers.
//
// Relay article, "Entrenamiento por relevos", top-2 paragraph: at serving time the
// engine runs one expert per token; opening section: experts ship as int4.  Only
// the experts actually hit are read (the permutation's compact active list), each
// weight row once, which makes the step bound by weight bytes.  A row's 32-input
// groups are spread over the lanes; each lane turns its group's nibbles into the
// integers q (exact in fp32), forms sum_i q_i * x_i for up to DEC_TOK tokens of the
// expert at a time and scales the sum once by the group's fp16 scale, so a group is
// dequantised once per pass over the expert's tokens.  A lane-group reduction gives
// the row's dot products.
namespace moe {
namespace {

constexpr int DEC_WARPS = 8;
constexpr int DEC_TOK = 4;  // tokens of one expert per pass

// Integer codes of one group: 16 bytes of two's-complement nibbles (even index in the
// low nibble) -> 32 floats.  (c ^ 8) is q + 8 in [0, 15]; 2^23 + (q + 8) is exact in
// fp32, so subtracting 2^23 + 8 gives q exactly.
__device__ __forceinline__ void int4_codes(const uint8_t* codes, float (&q)[32]) {
  const uint4 u = *reinterpret_cast<const uint4*>(codes);
  const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const uint32_t c = ((words[i] >> (4 * n)) & 0xFu) ^ 0x8u;
      q[8 * i + n] = __uint_as_float(0x4B000000u | c) - 8388616.0f;
    }
}

__device__ __forceinline__ float scale_of(const uint16_t* ws, long long i) {
  return __half2float(__ushort_as_half(ws[i]));
}

// sum_i q_i * x_i over the 32 bf16 values at p.
__device__ __forceinline__ float dot32(const float (&q)[32], const uint16_t* p) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = v[i];
    const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc = fmaf(q[8 * i + 2 * j], __uint_as_float(ws[j] << 16), acc);
      acc = fmaf(q[8 * i + 2 * j + 1], __uint_as_float(ws[j] & 0xFFFF0000u), acc);
    }
  }
  return acc;
}

// Sum over the `width` lanes of this lane's group (width a power of two <= 32).
__device__ __forceinline__ float group_sum(float v, int width) {
  for (int o = width / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ uint16_t to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Lanes per weight row: the row's groups spread over 32 lanes, or over fewer (and
// several rows per warp) when the row has fewer than 32 groups.
__device__ __forceinline__ int lanes_per_row(int ngroups) {
  int w = 32;
  while (w > 1 && w / 2 >= ngroups) w /= 2;
  return w;
}

// Gate/up of the routed experts: unit (active expert a, hidden unit j) computes
// h[p][j] = silu(Wg_e[j] . xp[p]) * (Wu_e[j] . xp[p]) for the expert's rows p.
__global__ void __launch_bounds__(DEC_WARPS * 32) int4_gate_up_kernel(
    const int32_t* __restrict__ active, const int32_t* __restrict__ offsets,
    const uint8_t* __restrict__ wq, const uint16_t* __restrict__ ws, const uint16_t* __restrict__ xp,
    uint16_t* __restrict__ h, int d, int f, int block, const int32_t* __restrict__ slot) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x % 32;
  const int ngroups = d / 32;
  const int lpr = lanes_per_row(ngroups), rpw = 32 / lpr;
  const int sub = lane / lpr, gl = lane % lpr;
  const long long per_expert = (f + rpw - 1) / rpw;
  const long long units = (long long)active[kMaxE] * per_expert;  // active[kMaxE]: count
  const long long stride = (long long)gridDim.x * DEC_WARPS;
  for (long long u = (long long)blockIdx.x * DEC_WARPS + threadIdx.x / 32; u < units; u += stride) {
    const int e = active[u / per_expert];
    const int j = (int)(u % per_expert) * rpw + sub;
    const bool row_ok = j < f;
    const int jj = row_ok ? j : f - 1;
    const long long we = slot ? slot[e] : e;  // the weights' position (a cache slot)
    const long long grow = we * 2 * f + (jj / block) * 2 * block + jj % block;
    const long long urow = grow + block;
    const int p0 = offsets[e], p1 = offsets[e + 1];
    for (int pc = p0; pc < p1; pc += DEC_TOK) {
      float ag[DEC_TOK], au[DEC_TOK];
#pragma unroll
      for (int m = 0; m < DEC_TOK; ++m) ag[m] = au[m] = 0.f;
      for (int g = gl; g < ngroups; g += lpr) {
        float qg[32], qu[32];
        int4_codes(wq + grow * (d / 2) + g * 16, qg);
        int4_codes(wq + urow * (d / 2) + g * 16, qu);
        const float sg = scale_of(ws, grow * ngroups + g), su = scale_of(ws, urow * ngroups + g);
#pragma unroll
        for (int m = 0; m < DEC_TOK; ++m)
          if (pc + m < p1) {
            const uint16_t* xr = xp + (long long)(pc + m) * d + g * 32;
            ag[m] = fmaf(sg, dot32(qg, xr), ag[m]);
            au[m] = fmaf(su, dot32(qu, xr), au[m]);
          }
      }
#pragma unroll
      for (int m = 0; m < DEC_TOK; ++m) {
        const float gs = group_sum(ag[m], lpr), us = group_sum(au[m], lpr);
        if (gl == 0 && row_ok && pc + m < p1)
          h[(long long)(pc + m) * f + j] = to_bf16_bits(gs / (1.0f + __expf(-gs)) * us);
      }
    }
  }
}

// Down projection of the routed experts: unit (active expert a, output row i)
// computes y[p][i] = Wd_e[i] . h[p] for the expert's rows p.
__global__ void __launch_bounds__(DEC_WARPS * 32) int4_down_kernel(
    const int32_t* __restrict__ active, const int32_t* __restrict__ offsets,
    const uint8_t* __restrict__ wq, const uint16_t* __restrict__ ws, const uint16_t* __restrict__ h,
    uint16_t* __restrict__ y, int d, int f, const int32_t* __restrict__ slot) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x % 32;
  const int ngroups = f / 32;
  const int lpr = lanes_per_row(ngroups), rpw = 32 / lpr;
  const int sub = lane / lpr, gl = lane % lpr;
  const long long per_expert = (d + rpw - 1) / rpw;
  const long long units = (long long)active[kMaxE] * per_expert;
  const long long stride = (long long)gridDim.x * DEC_WARPS;
  for (long long u = (long long)blockIdx.x * DEC_WARPS + threadIdx.x / 32; u < units; u += stride) {
    const int e = active[u / per_expert];
    const int i = (int)(u % per_expert) * rpw + sub;
    const bool row_ok = i < d;
    const long long row = (long long)(slot ? slot[e] : e) * d + (row_ok ? i : d - 1);
    const int p0 = offsets[e], p1 = offsets[e + 1];
    for (int pc = p0; pc < p1; pc += DEC_TOK) {
      float acc[DEC_TOK];
#pragma unroll
      for (int m = 0; m < DEC_TOK; ++m) acc[m] = 0.f;
      for (int g = gl; g < ngroups; g += lpr) {
        float q[32];
        int4_codes(wq + row * (f / 2) + g * 16, q);
        const float sc = scale_of(ws, row * ngroups + g);
#pragma unroll
        for (int m = 0; m < DEC_TOK; ++m)
          if (pc + m < p1) acc[m] = fmaf(sc, dot32(q, h + (long long)(pc + m) * f + g * 32), acc[m]);
      }
#pragma unroll
      for (int m = 0; m < DEC_TOK; ++m) {
        const float v = group_sum(acc[m], lpr);
        if (gl == 0 && row_ok && pc + m < p1) y[(long long)(pc + m) * d + i] = to_bf16_bits(v);
      }
    }
  }
}

// Serving with few (token, expert) pairs: the same products straight from the routing
// result, with no permutation.  Pairs p (= t * k + j) keep their order; a warp's unit
// is (pair, DIR_RPU row slots) and only the first pair routed to an expert does the
// work, for all of that expert's pairs (found by a ballot over idx), so each expert's
// rows are still read once.  Per pass over up to DIR_TOK of the expert's pairs, a lane
// decodes each of its row groups once (integer codes, exact in fp32), unpacks each
// pair's inputs once, and accumulates the products; the scale multiplies each group's
// sum once.  h and y are indexed by pair.
constexpr int DIR_RPU = 2;
constexpr int DIR_TOK = 2;

template <bool GATE_UP>
__global__ void __launch_bounds__(DEC_WARPS * 32, 2) int4_direct_kernel(
    const int32_t* __restrict__ idx, int P, int k, const uint8_t* __restrict__ wq,
    const uint16_t* __restrict__ ws, const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
    int d, int f, int block, const int32_t* __restrict__ slot) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int NM = GATE_UP ? 2 : 1;  // gate and up rows, or the down row
  const int lane = threadIdx.x % 32;
  const int K = GATE_UP ? d : f, rows = GATE_UP ? f : d;  // inputs, outputs per expert
  const int ngroups = K / 32;
  const int lpr = lanes_per_row(ngroups), rpw = 32 / lpr;
  const int sub = lane / lpr, gl = lane % lpr;
  const int ea = lane < P ? idx[lane] : -1, eb = lane + 32 < P ? idx[lane + 32] : -1;
  // Fewer pairs leave more warps idle: then each unit covers fewer rows.
  const int rpu = P >= 16 ? DIR_RPU : 1;
  const int rows_per_unit = rpw * rpu;
  const long long per_pair = (rows + rows_per_unit - 1) / rows_per_unit;
  const long long units = (long long)P * per_pair;
  const long long stride = (long long)gridDim.x * DEC_WARPS;
  for (long long u = (long long)blockIdx.x * DEC_WARPS + threadIdx.x / 32; u < units; u += stride) {
    const int p = (int)(u / per_pair);
    const int e = __shfl_sync(0xFFFFFFFFu, p < 32 ? ea : eb, p & 31);
    const unsigned ma = __ballot_sync(0xFFFFFFFFu, ea == e), mb = __ballot_sync(0xFFFFFFFFu, eb == e);
    const int first = ma ? __ffs(ma) - 1 : 32 + __ffs(mb) - 1;
    if (first != p) continue;  // warp-uniform: another unit covers this expert's pairs
    const int r_base = (int)(u % per_pair) * rows_per_unit + sub;
    const long long we = slot ? slot[e] : e;  // the weights' position (a cache slot)
    unsigned long long mask = (unsigned long long)ma | ((unsigned long long)mb << 32);
    while (mask) {
      int pp[DIR_TOK], cnt = 0;
#pragma unroll
      for (int m = 0; m < DIR_TOK; ++m) {
        pp[m] = 0;
        if (mask) {
          pp[m] = __ffsll((long long)mask) - 1;
          mask &= mask - 1;
          cnt = m + 1;
        }
      }
      for (int i = 0; i < rpu; ++i) {
        const int r = r_base + i * rpw;
        const int rr = min(r, rows - 1);
        long long wrow[NM];
        if (GATE_UP) {
          wrow[0] = we * 2 * f + (rr / block) * 2 * block + rr % block;
          wrow[NM - 1] = wrow[0] + block;
        } else {
          wrow[0] = we * d + rr;
        }
        float acc[NM][DIR_TOK];
#pragma unroll
        for (int mm = 0; mm < NM; ++mm)
#pragma unroll
          for (int m = 0; m < DIR_TOK; ++m) acc[mm][m] = 0.f;
        for (int g = gl; g < ngroups; g += lpr) {
#pragma unroll
          for (int mm = 0; mm < NM; ++mm) {
            float q[32];
            int4_codes(wq + wrow[mm] * (K / 2) + g * 16, q);
            const float sc = scale_of(ws, wrow[mm] * ngroups + g);
            // Each pair's inputs are read inside its product (gate/up: token pp / k of
            // x; down: pair pp of h), so only the decoded codes stay live.
#pragma unroll
            for (int m = 0; m < DIR_TOK; ++m)
              if (m < cnt)
                acc[mm][m] = fmaf(sc, dot32(q, src + (long long)(GATE_UP ? pp[m] / k : pp[m]) * K + g * 32),
                                  acc[mm][m]);
          }
        }
#pragma unroll
        for (int m = 0; m < DIR_TOK; ++m)
          if (m < cnt) {
            const float va = group_sum(acc[0][m], lpr);
            const float vb = GATE_UP ? group_sum(acc[NM - 1][m], lpr) : 0.f;
            if (gl == 0 && r < rows)
              dst[(long long)pp[m] * rows + r] = to_bf16_bits(GATE_UP ? va / (1.0f + __expf(-va)) * vb : va);
          }
      }
    }
  }
}

// The same permutation-free products on the tensor cores (mma.sync m16n8k16: bf16
// inputs, fp32 sums): weights in M, the expert's pairs in N (8 per pass).  A unit is
// (expert, row tile); the experts are the distinct ones of the routing result, in the
// order of their first pair.  The CTA's 8 warps share a unit: gate/up, 16 gate rows and
// the 16 matching up rows with K split 8 ways; down, two 16-row tiles with K split 4
// ways.  Each CTA walks its units through a ring of shared-memory stages (two for gate/up,
// four for down) filled by cp.async (a unit's code rows and scale rows, each row padded
// by 16 bytes so the fragment reads below fall in distinct banks), so the next units'
// weights stream in while one is multiplied.  Per 32-input group a lane reads one 32-bit word of 8
// codes (word l%4) of each of its rows l/4 and l/4 + 8 and forms bf16 pairs of nibbles
// (i, i + 4) (`q_pair`).  The sum over k may run in any order as long as both operands
// follow it, so the lane's B fragment holds the inputs at those same positions: its 8
// consecutive bf16 of the pair's row, re-paired (`input_pairs`).  A group's two 16-deep
// steps accumulate from zero and its fp16 scale multiplies that partial once (every
// product q * x exact, as in the CUDA-core path); the warps' partials are summed in a
// fixed order through shared memory.  With one expert per token the down projection can
// end with the combine: out = bf16(s + gate * y), y still in fp32 (`comb_s`, `comb_gate`).
constexpr int TCD_WARPS = 8;
// Ring depth: two stages let four gate/up CTAs share an SM (more warps to hide latency
// beat a deeper ring); four for the down projection, also four CTAs per SM.
template <bool GATE_UP>
__host__ __device__ constexpr int tcd_stages() { return GATE_UP ? 2 : 4; }

template <bool GATE_UP>
struct TcdShape {
  static constexpr int NM = GATE_UP ? 2 : 1;  // row sets: gate and up, or the down rows
  static constexpr int RT = GATE_UP ? 1 : 2;  // 16-row tiles per unit
  static constexpr int KS = TCD_WARPS / RT;   // K parts per tile, one warp each
  static constexpr int ROWS = 16 * RT * NM;   // weight rows per unit
};

// Nibbles i and i + 4 of a code word as a bf16 pair of the integers q.  Each half of
// (w >> 4i) & 0x000F000F ^ 0x43084308 is the bf16 bit pattern of 128 + (q + 8) (the
// nibble ^ 8 is q + 8 in [0, 15], and the unit in the last place of 128 is 1), so
// subtracting 136 leaves q, exactly.
__device__ __forceinline__ uint32_t q_pair(uint32_t w, int i) {
  const uint32_t v = ((w >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u;
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x43084308u));
  return r;
}

// 8 consecutive bf16 inputs x0..x7 as the pairs (x0, x4), (x1, x5), (x2, x6), (x3, x7).
__device__ __forceinline__ void input_pairs(const uint4& u, uint32_t (&b)[4]) {
  b[0] = __byte_perm(u.x, u.z, 0x5410);
  b[1] = __byte_perm(u.x, u.z, 0x7632);
  b[2] = __byte_perm(u.y, u.w, 0x5410);
  b[3] = __byte_perm(u.y, u.w, 0x7632);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <bool GATE_UP>
__global__ void __launch_bounds__(TCD_WARPS * 32, 4) int4_tc_direct_kernel(
    const int32_t* __restrict__ idx, int P, int k, const uint8_t* __restrict__ wq,
    const uint16_t* __restrict__ ws, const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
    int d, int f, int block, const int32_t* __restrict__ slot, const uint16_t* __restrict__ comb_s,
    const float* __restrict__ comb_gate) {
  using S = TcdShape<GATE_UP>;
  extern __shared__ __align__(16) uint8_t tcd_smem[];
  const int K = GATE_UP ? d : f, rows = GATE_UP ? f : d;
  const int ngroups = K / 32, gpw = ngroups / S::KS;
  const int cstride = K / 2 + 16, sstride = ngroups * 2 + 16;  // padded row strides (bytes)
  const int stage_bytes = S::ROWS * (cstride + sstride);
  float(*red)[S::NM][4][32] = reinterpret_cast<float(*)[S::NM][4][32]>(tcd_smem + tcd_stages<GATE_UP>() * stage_bytes);
  int(*plist)[kDirectMaxPairs] = reinterpret_cast<int(*)[kDirectMaxPairs]>(red + TCD_WARPS);
  int* dexp = plist[TCD_WARPS];  // the distinct experts, in the order of their first pair
  int* goff = dexp + kDirectMaxPairs;  // gate/up: each tile's first gate row within an expert
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int rt = warp / S::KS, kp = warp % S::KS;
  const int tiles = rows / (16 * S::RT);
  // The distinct experts: pairs whose expert no earlier pair has (every warp alike).
  const bool va = lane < P, vb = lane + 32 < P;
  const int ea = va ? idx[lane] : -1 - lane, eb = vb ? idx[lane + 32] : -1 - lane;
  const unsigned below = (1u << lane) - 1u;
  bool b_seen_in_a = false;
  for (int q = 0; q < 32; ++q) b_seen_in_a |= __shfl_sync(0xFFFFFFFFu, ea, q) == eb;
  // Every lane takes part in both matches (full-mask warp primitives; none of them may
  // sit behind a short-circuit test that some lanes skip).
  const unsigned same_a = __match_any_sync(0xFFFFFFFFu, ea), same_b = __match_any_sync(0xFFFFFFFFu, eb);
  const unsigned first_lo = __ballot_sync(0xFFFFFFFFu, va && !(same_a & below));
  const unsigned first_hi = __ballot_sync(0xFFFFFFFFu, vb && !b_seen_in_a && !(same_b & below));
  if (warp == 0) {
    if ((first_lo >> lane) & 1u) dexp[__popc(first_lo & below)] = ea;
    if ((first_hi >> lane) & 1u) dexp[__popc(first_lo) + __popc(first_hi & below)] = eb;
  }
  if (GATE_UP)
    for (int tl = tid; tl < tiles; tl += TCD_WARPS * 32) goff[tl] = (tl * 16 / block) * 2 * block + tl * 16 % block;
  __syncthreads();
  const int nunits = (__popc(first_lo) + __popc(first_hi)) * tiles;
  const int mine = (int)blockIdx.x < nunits ? (nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const uint32_t smem0 = smem_u32(tcd_smem);
  // Global row (in the code and scale tensors) of row r of a unit (the tile's 16 gate rows
  // sit inside one interleave block: block is a multiple of 16).
  auto weight_row = [&](long long we, int tile, int r) -> long long {
    if (GATE_UP) return we * 2 * f + goff[tile] + (r & 15) + (r >= 16 ? block : 0);
    return we * d + tile * 32 + r;
  };
  // A CTA's units are blockIdx.x + i * gridDim.x; walk their (expert, tile) without
  // dividing per unit.
  const int step_q = (int)gridDim.x / tiles, step_r = (int)gridDim.x % tiles;
  auto advance = [&](int& ue, int& tl) {
    tl += step_r;
    ue += step_q;
    if (tl >= tiles) {
      tl -= tiles;
      ++ue;
    }
  };
  // All threads: copy unit `unit`'s code and scale rows into stage `st`, 8 threads per
  // row (each row's address computed once), 16-byte chunks.
  static_assert(S::ROWS * 8 == TCD_WARPS * 32, "8 copying threads per row");
  const int crow_r = tid >> 3, csub = tid & 7;
  auto issue = [&](int ue, int tile, int st) {
    const int e = dexp[ue];
    const long long row = weight_row(slot ? slot[e] : e, tile, crow_r);
    const uint8_t* cs = wq + row * (K / 2) + csub * 16;
    uint32_t cd = smem0 + st * stage_bytes + crow_r * cstride + csub * 16;
    for (int q = csub; q < K / 32; q += 8, cs += 128, cd += 128) cp_async16(cd, cs);
    const uint8_t* ss = reinterpret_cast<const uint8_t*>(ws) + row * (K / 16) + csub * 16;
    uint32_t sd = smem0 + st * stage_bytes + S::ROWS * cstride + crow_r * sstride + csub * 16;
    for (int q = csub; q < K / 256; q += 8, ss += 128, sd += 128) cp_async16(sd, ss);
  };
  int cur_ue = (int)blockIdx.x / tiles, cur_tl = (int)blockIdx.x % tiles;  // unit i
  int nxt_ue = cur_ue, nxt_tl = cur_tl;                                      // unit i + stages - 1
#pragma unroll 1
  for (int i = 0; i < tcd_stages<GATE_UP>() - 1; ++i) {
    if (i < mine) issue(nxt_ue, nxt_tl, i);
    cp_async_commit();
    advance(nxt_ue, nxt_tl);
  }
  int* pl = plist[warp];
#pragma unroll 1
  for (int i = 0; i < mine; ++i) {
    if (i + tcd_stages<GATE_UP>() - 1 < mine) issue(nxt_ue, nxt_tl, (i + tcd_stages<GATE_UP>() - 1) % tcd_stages<GATE_UP>());
    cp_async_commit();
    advance(nxt_ue, nxt_tl);
    const int e = dexp[cur_ue], tile = cur_tl;
    advance(cur_ue, cur_tl);
    const unsigned ma = __ballot_sync(0xFFFFFFFFu, ea == e), mb = __ballot_sync(0xFFFFFFFFu, eb == e);
    const int cnt = __popc(ma) + __popc(mb);
    // The expert's pairs in order (each warp keeps its own copy).
    if ((ma >> lane) & 1u) pl[__popc(ma & below)] = lane;
    if ((mb >> lane) & 1u) pl[__popc(ma) + __popc(mb & below)] = lane + 32;
    __syncwarp();
    const uint8_t* stage = tcd_smem + (i % tcd_stages<GATE_UP>()) * stage_bytes;
    const int g0 = kp * gpw;
    // This lane's rows r0 = m*16 + rt*16 + l/4 and r0 + 8 of each set, at group g0.
    const uint8_t* cp0 = stage + (rt * 16 + g) * cstride + g0 * 16 + 4 * t;
    const uint8_t* sp0 = stage + S::ROWS * cstride + (rt * 16 + g) * sstride + g0 * 2;
    bool waited = false;
#pragma unroll 1
    for (int n0 = 0; n0 < cnt; n0 += 8) {
      const int pn = n0 + g;  // this lane's column of B
      const bool col_ok = pn < cnt;
      const int srow = col_ok ? (GATE_UP && k != 1 ? pl[pn] / k : pl[pn]) : 0;
      const uint16_t* xr = src + (long long)srow * K + g0 * 32 + 8 * t;
      float acc[S::NM][4];
#pragma unroll
      for (int m = 0; m < S::NM; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
#pragma unroll 1
      for (int j0 = 0; j0 < gpw; j0 += 4) {
        uint4 xv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          xv[j] = (col_ok && j0 + j < gpw) ? *reinterpret_cast<const uint4*>(xr + (j0 + j) * 32)
                                           : make_uint4(0, 0, 0, 0);
        if (!waited) {  // the unit's rows have landed (this thread's copies, then everyone's)
          cp_async_wait<tcd_stages<GATE_UP>() - 1>();
          __syncthreads();
          waited = true;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j0 + j >= gpw) break;
          const int jj = j0 + j;
          uint32_t b[4];
          input_pairs(xv[j], b);
#pragma unroll
          for (int m = 0; m < S::NM; ++m) {
            const uint8_t* c0 = cp0 + m * 16 * cstride + jj * 16;
            const uint8_t* s0p = sp0 + m * 16 * sstride + jj * 2;
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(c0);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(c0 + 8 * cstride);
            const float s0 = __half2float(*reinterpret_cast<const __half*>(s0p));
            const float s1 = __half2float(*reinterpret_cast<const __half*>(s0p + 8 * sstride));
            float part[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(part, q_pair(w0, 0), q_pair(w1, 0), q_pair(w0, 1), q_pair(w1, 1), b[0], b[1]);
            mma16816(part, q_pair(w0, 2), q_pair(w1, 2), q_pair(w0, 3), q_pair(w1, 3), b[2], b[3]);
            acc[m][0] = fmaf(s0, part[0], acc[m][0]);
            acc[m][1] = fmaf(s0, part[1], acc[m][1]);
            acc[m][2] = fmaf(s1, part[2], acc[m][2]);
            acc[m][3] = fmaf(s1, part[3], acc[m][3]);
          }
        }
      }
      if (n0 > 0) __syncthreads();  // the previous pass's sums have been read
#pragma unroll
      for (int m = 0; m < S::NM; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) red[warp][m][c][lane] = acc[m][c];
      __syncthreads();
      // Cells (tile row r, column n) summed over the K parts in order.  Lane l/4 holds
      // rows l/4 and l/4 + 8 (c / 2), columns 2(l%4) + c%2.
      constexpr int CELLS = 16 * S::RT * 8;
      for (int cell = tid; cell < CELLS; cell += TCD_WARPS * 32) {
        const int n = cell / (16 * S::RT), rr = cell % (16 * S::RT);
        const int tt = rr / 16, r = rr % 16;
        const int cl = (r % 8) * 4 + n / 2, cc = (r / 8) * 2 + (n & 1);
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int q = 0; q < S::KS; ++q) {
          v0 += red[tt * S::KS + q][0][cc][cl];
          if (GATE_UP) v1 += red[tt * S::KS + q][S::NM - 1][cc][cl];
        }
        if (n0 + n < cnt) {
          const int pr = pl[n0 + n];
          const long long o = (long long)pr * rows + (long long)tile * 16 * S::RT + rr;
          if (GATE_UP)
            dst[o] = to_bf16_bits(v0 / (1.0f + __expf(-v0)) * v1);
          else if (comb_s)  // top-1 combine: pair pr is token pr
            dst[o] = to_bf16_bits(fmaf(comb_gate[pr], v0, __uint_as_float((uint32_t)comb_s[o] << 16)));
          else
            dst[o] = to_bf16_bits(v0);
        }
      }
    }
    // The next copies reuse this unit's stage, the next sums this unit's `red`.
    __syncthreads();
  }
  cp_async_wait<0>();
}

template <bool GATE_UP>
size_t tcd_smem_bytes(int d, int f) {
  using S = TcdShape<GATE_UP>;
  const int K = GATE_UP ? d : f;
  return (size_t)tcd_stages<GATE_UP>() * S::ROWS * (K / 2 + 16 + K / 16 + 16) + sizeof(float) * TCD_WARPS * S::NM * 4 * 32 +
         sizeof(int) * (TCD_WARPS + 1) * kDirectMaxPairs + (GATE_UP ? sizeof(int) * (f / 16) : 0);
}

// Four CTAs per SM at the Nano shapes (the limits admit larger ones at lower occupancy).
constexpr int kTcdMaxSmemGateUp = 110 * 1024, kTcdMaxSmemDown = 54 * 1024;

bool tc_direct_supported(bool gate_up, int d, int f, int block, const void* wq, const void* ws, const void* src) {
  const bool aligned = ((reinterpret_cast<uintptr_t>(wq) | reinterpret_cast<uintptr_t>(ws) |
                         reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
  if (!aligned) return false;
  return gate_up ? (d % 256 == 0 && f % 16 == 0 && block % 16 == 0 && tcd_smem_bytes<true>(d, f) <= (size_t)kTcdMaxSmemGateUp)
                 : (f % 256 == 0 && d % 32 == 0 && tcd_smem_bytes<false>(d, f) <= (size_t)kTcdMaxSmemDown);
}

int decode_grid() {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return 4 * sms;
}

// The tensor-core kernels' shared-memory limits, raised once per device to the largest
// size the support check admits.
cudaError_t tcd_raise_smem_limits() {
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(int4_tc_direct_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTcdMaxSmemGateUp);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(int4_tc_direct_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kTcdMaxSmemDown);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  return cudaSuccess;
}


}  // namespace

cudaError_t launch_int4_gate_up(const int32_t* active, const int32_t* offsets, const uint8_t* wq,
                                const uint16_t* ws, const uint16_t* xp, uint16_t* h, int d, int f,
                                int block, cudaStream_t s, const int32_t* slot) {
  return launch_pdl(int4_gate_up_kernel, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, active,
                    offsets, wq, ws, xp, h, d, f, block, slot);
}

cudaError_t launch_int4_direct(bool gate_up, const int32_t* idx, int pairs, int k, const uint8_t* wq,
                               const uint16_t* ws, const uint16_t* src, uint16_t* dst, int d, int f,
                               int block, cudaStream_t s, const int32_t* slot) {
  if (pairs < 1 || pairs > kDirectMaxPairs) return cudaErrorInvalidValue;
  if (tc_direct_supported(gate_up, d, f, block, wq, ws, src)) {
    // At most `pairs` distinct experts; one resident wave of CTAs walks the units.
    const long long units = (long long)pairs * (gate_up ? f / 16 : d / 32);
    const int grid = (int)std::min<long long>(units, decode_grid());  // four resident CTAs per SM
    const size_t smem = gate_up ? tcd_smem_bytes<true>(d, f) : tcd_smem_bytes<false>(d, f);
    const cudaError_t ea = tcd_raise_smem_limits();
    if (ea != cudaSuccess) return ea;
    const uint16_t* no_s = nullptr;
    const float* no_g = nullptr;
    if (gate_up)
      return launch_pdl(int4_tc_direct_kernel<true>, dim3(grid), dim3(TCD_WARPS * 32), smem, s, idx, pairs, k,
                        wq, ws, src, dst, d, f, block, slot, no_s, no_g);
    return launch_pdl(int4_tc_direct_kernel<false>, dim3(grid), dim3(TCD_WARPS * 32), smem, s, idx, pairs, k,
                      wq, ws, src, dst, d, f, block, slot, no_s, no_g);
  }
  if (gate_up)
    return launch_pdl(int4_direct_kernel<true>, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, idx,
                      pairs, k, wq, ws, src, dst, d, f, block, slot);
  return launch_pdl(int4_direct_kernel<false>, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, idx,
                    pairs, k, wq, ws, src, dst, d, f, block, slot);
}

bool int4_direct_down_combine_supported(int d, int f, int k, const void* wq, const void* ws, const void* h) {
  return k == 1 && tc_direct_supported(false, d, f, 16, wq, ws, h);
}

cudaError_t launch_int4_direct_down_combine(const int32_t* idx, int pairs, const uint8_t* wq, const uint16_t* ws,
                                            const uint16_t* h, const uint16_t* s_in, const float* gate,
                                            uint16_t* out, int d, int f, cudaStream_t s, const int32_t* slot) {
  if (pairs < 1 || pairs > kDirectMaxPairs || !int4_direct_down_combine_supported(d, f, 1, wq, ws, h) || !s_in ||
      !gate)
    return cudaErrorInvalidValue;
  const cudaError_t ea = tcd_raise_smem_limits();
  if (ea != cudaSuccess) return ea;
  const int grid = (int)std::min<long long>((long long)pairs * (d / 32), decode_grid());
  return launch_pdl(int4_tc_direct_kernel<false>, dim3(grid), dim3(TCD_WARPS * 32), tcd_smem_bytes<false>(d, f), s,
                    idx, pairs, 1, wq, ws, h, out, d, f, 0, slot, s_in, gate);
}

cudaError_t launch_int4_down(const int32_t* active, const int32_t* offsets, const uint8_t* wq,
                             const uint16_t* ws, const uint16_t* h, uint16_t* y, int d, int f,
                             cudaStream_t s, const int32_t* slot) {
  return launch_pdl(int4_down_kernel, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, active,
                    offsets, wq, ws, h, y, d, f, slot);
}

}  // namespace moe
