// int4 container support for the top-1 serving path.
//
// Relay article, opening section, second paragraph: experts ship in an int4
// container.  Format (this library's reading): symmetric, groups of 32 consecutive
// input elements, fp16 scale = fp16(fl32(max|w| / 7)), code = clamp(rint(fl32(w /
// scale)), -7, 7) (0 where the scale is 0), two's-complement nibbles with the even
// index in the low nibble.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

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

int decode_grid() {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return 4 * sms;
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
  if (gate_up)
    return launch_pdl(int4_direct_kernel<true>, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, idx,
                      pairs, k, wq, ws, src, dst, d, f, block, slot);
  return launch_pdl(int4_direct_kernel<false>, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, idx,
                    pairs, k, wq, ws, src, dst, d, f, block, slot);
}

cudaError_t launch_int4_down(const int32_t* active, const int32_t* offsets, const uint8_t* wq,
                             const uint16_t* ws, const uint16_t* h, uint16_t* y, int d, int f,
                             cudaStream_t s, const int32_t* slot) {
  return launch_pdl(int4_down_kernel, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, active,
                    offsets, wq, ws, h, y, d, f, slot);
}

}  // namespace moe
