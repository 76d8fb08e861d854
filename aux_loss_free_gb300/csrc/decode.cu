// int4 container support for the top-1 serving path.
//
// Relay article, opening section, second paragraph: experts ship in an int4
// container.  Format (this library's reading): symmetric, groups of 32 consecutive
// input elements, fp16 scale = fp16(fl32(max|w| / 7)), code = clamp(rint(fl32(w /
// scale)), -7, 7) (0 where the scale is 0), two's-complement nibbles with the even
// index in the low nibble.
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
