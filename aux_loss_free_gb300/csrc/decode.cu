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
// weight row once, which makes the step bound by weight bytes.  Lane l of a warp
// owns input group g = l, l + 32, ... (32 consecutive inputs, one fp16 scale),
// dequantises w = q * scale and accumulates against the group's token values;
// a warp reduction gives the row's dot product for every token of the expert.
namespace moe {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Dequantise one group: 16 bytes of two's-complement nibbles (even index low) and
// its fp16 scale into 32 floats.
__device__ __forceinline__ void dequant_group(const uint8_t* codes, uint16_t scale_bits, float (&w)[32]) {
  const uint4 u = *reinterpret_cast<const uint4*>(codes);
  const float s = __half2float(__ushort_as_half(scale_bits));
  const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int q = static_cast<int>((words[i] >> (4 * n)) & 0xFu);
      w[8 * i + n] = static_cast<float>(q >= 8 ? q - 16 : q) * s;
    }
}

// 32 bf16 values (64 bytes) as floats.
__device__ __forceinline__ void load_bf16x32(const uint16_t* p, float (&v)[32]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = q[i];
    const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(ws[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ uint16_t to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

constexpr int DEC_WARPS = 8;

// Gate/up of the routed experts: unit (active expert a, hidden unit j) computes
// h[p][j] = silu(Wg_e[j] . xp[p]) * (Wu_e[j] . xp[p]) for the expert's rows p.
__global__ void __launch_bounds__(DEC_WARPS * 32) int4_gate_up_kernel(
    const int32_t* __restrict__ active, const int32_t* __restrict__ offsets,
    const uint8_t* __restrict__ wq, const uint16_t* __restrict__ ws, const uint16_t* __restrict__ xp,
    uint16_t* __restrict__ h, int d, int f, int block) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x % 32;
  const long long units = (long long)active[kMaxE] * f;  // active[kMaxE] holds the count
  const long long stride = (long long)gridDim.x * DEC_WARPS;
  const int ngroups = d / 32;
  for (long long u = (long long)blockIdx.x * DEC_WARPS + threadIdx.x / 32; u < units; u += stride) {
    const int e = active[u / f];
    const int j = (int)(u % f);
    const long long grow = (long long)e * 2 * f + (j / block) * 2 * block + j % block;
    const long long urow = grow + block;
    const int p0 = offsets[e], p1 = offsets[e + 1];
    for (int p = p0; p < p1; ++p) {
      float gs = 0.f, us = 0.f;
      for (int g = lane; g < ngroups; g += 32) {
        float wg[32], wu[32], xv[32];
        dequant_group(wq + grow * (d / 2) + g * 16, ws[grow * ngroups + g], wg);
        dequant_group(wq + urow * (d / 2) + g * 16, ws[urow * ngroups + g], wu);
        load_bf16x32(xp + (long long)p * d + g * 32, xv);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          gs = fmaf(wg[i], xv[i], gs);
          us = fmaf(wu[i], xv[i], us);
        }
      }
      gs = warp_sum(gs);
      us = warp_sum(us);
      if (lane == 0) h[(long long)p * f + j] = to_bf16_bits(gs / (1.0f + __expf(-gs)) * us);
    }
  }
}

// Down projection of the routed experts: unit (active expert a, output row i)
// computes y[p][i] = Wd_e[i] . h[p] for the expert's rows p.
__global__ void __launch_bounds__(DEC_WARPS * 32) int4_down_kernel(
    const int32_t* __restrict__ active, const int32_t* __restrict__ offsets,
    const uint8_t* __restrict__ wq, const uint16_t* __restrict__ ws, const uint16_t* __restrict__ h,
    uint16_t* __restrict__ y, int d, int f) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x % 32;
  const long long units = (long long)active[kMaxE] * d;
  const long long stride = (long long)gridDim.x * DEC_WARPS;
  const int ngroups = f / 32;
  for (long long u = (long long)blockIdx.x * DEC_WARPS + threadIdx.x / 32; u < units; u += stride) {
    const int e = active[u / d];
    const int i = (int)(u % d);
    const long long row = (long long)e * d + i;
    const int p0 = offsets[e], p1 = offsets[e + 1];
    for (int p = p0; p < p1; ++p) {
      float acc = 0.f;
      for (int g = lane; g < ngroups; g += 32) {
        float w[32], hv[32];
        dequant_group(wq + row * (f / 2) + g * 16, ws[row * ngroups + g], w);
        load_bf16x32(h + (long long)p * f + g * 32, hv);
#pragma unroll
        for (int k2 = 0; k2 < 32; ++k2) acc = fmaf(w[k2], hv[k2], acc);
      }
      acc = warp_sum(acc);
      if (lane == 0) y[(long long)p * d + i] = to_bf16_bits(acc);
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
                                int block, cudaStream_t s) {
  return launch_pdl(int4_gate_up_kernel, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, active,
                    offsets, wq, ws, xp, h, d, f, block);
}

cudaError_t launch_int4_down(const int32_t* active, const int32_t* offsets, const uint8_t* wq,
                             const uint16_t* ws, const uint16_t* h, uint16_t* y, int d, int f,
                             cudaStream_t s) {
  return launch_pdl(int4_down_kernel, dim3(decode_grid()), dim3(DEC_WARPS * 32), 0, s, active,
                    offsets, wq, ws, h, y, d, f);
}

}  // namespace moe
