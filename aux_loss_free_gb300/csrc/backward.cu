// Kernels of the MoE layer backward (besides the grouped GEMMs).
//
// The relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B
// de NanoColibri por $200") states the forward: opening section, architecture
// paragraph (sigmoid-plus-bias router, routed experts, always-resident shared expert)
// and section "Entrenamiento por relevos", top-2 paragraph (gates renormalised over the
// winners).  The backward is the chain rule through it, with the selection held fixed
// (the biased top-k is piecewise constant and the bias gets no gradient):
//   dy = g dout_t, dh = Wd_e^T dy, da = dh b silu'(a), db = dh silu(a),
//   dg = <dout_t, y> = <Wd_e^T dout_t, h>, ds_j = (dg_j - sum_i dg_i g_i) / S
//   (renormalised) or dg_j, dz_j = ds_j s_j (1 - s_j), dx_t += sum_j dz_j W_r[e_j].
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"

namespace moe {
namespace {

// Padded layout of the permuted rows: expert e's n_e rows start at poff[e], the sum
// of the earlier experts' counts rounded up to multiples of 64, so that every expert's
// rows form whole 64-row K atoms of the weight-gradient GEMMs (the padding rows are
// zero in every operand).  Each block derives poff from the offsets in shared memory
// (one warp, E <= 256); block 0 stores it.  Thread i then writes tok_pad[i] (source
// token of padded row i, -1 for padding and for rows past poff[E]) for i < q_max and,
// for pair i < pairs, its padded row inv_pad[i] and gperm[inv_pad[i]] = gate[i].
__global__ void pad_map_kernel(const int32_t* __restrict__ off, const int32_t* __restrict__ perm_tok,
                               const int32_t* __restrict__ idx, const int32_t* __restrict__ inv_pos,
                               const float* __restrict__ gate, int E, long long pairs, long long q_max,
                               int32_t* __restrict__ poff_out, int32_t* __restrict__ tok_pad,
                               int32_t* __restrict__ inv_pad, float* __restrict__ gperm) {
  __shared__ int s_off[kMaxE + 1], s_poff[kMaxE + 1];
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    constexpr int PER = kMaxE / 32;
    int cnt[PER], sum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      cnt[i] = e < E ? (off[e + 1] - off[e] + 63) / 64 * 64 : 0;
      if (e <= E) s_off[e] = off[e];
      sum += cnt[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      if (e <= E) s_poff[e] = run;
      run += cnt[i];
    }
    if (lane == 0 && E == kMaxE) s_off[E] = off[E];
    if (lane == 31 && E == kMaxE) s_poff[E] = incl;
  }
  __syncthreads();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) poff_out[e] = s_poff[e];
  if (i < q_max) {
    int tok = -1;
    if (i < s_poff[E]) {
      int lo = 0, hi = E - 1;  // last expert with s_poff <= i
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_poff[mid] <= i) lo = mid; else hi = mid - 1;
      }
      const long long r = s_off[lo] + (i - s_poff[lo]);
      if (r < s_off[lo + 1]) tok = perm_tok[r];
    }
    tok_pad[i] = tok;
    if (tok < 0) gperm[i] = 0.f;  // padding rows carry a zero gate (never garbage)
  }
  if (i < pairs) {
    const int e = idx[i];
    const int q = s_poff[e] + (inv_pos[i] - s_off[e]);
    inv_pad[i] = q;
    gperm[q] = gate[i];
  }
}

// xp[q] = x[tok_pad[q]], dp[q] = dout[tok_pad[q]] (zero rows for tok_pad < 0) for
// q < *rows_limit (= poff[E]), bf16, 16 bytes per thread.
__global__ void gather_pad_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ dout,
                                  const int32_t* __restrict__ tok_pad, long long q_max,
                                  const int32_t* __restrict__ rows_limit, int d,
                                  uint16_t* __restrict__ xp, uint16_t* __restrict__ dp) {
  const int vpr = d / 8;  // 16-byte vectors per row
  const long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= q_max * vpr) return;
  const long long q = v / vpr;
  if (q >= *rows_limit) return;  // rows past the padded layout's end are never read
  const int c = (int)(v % vpr);
  const int t = tok_pad[q];
  uint4 a = make_uint4(0, 0, 0, 0), b = a;
  if (t >= 0) {
    a = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d) + c);
    b = __ldg(reinterpret_cast<const uint4*>(dout + (size_t)t * d) + c);
  }
  reinterpret_cast<uint4*>(xp + q * d)[c] = a;
  reinterpret_cast<uint4*>(dp + q * d)[c] = b;
}

// Router backward and the input gradient, one warp per token (lane j < k holds pair j):
//   dg_j = sum of the pair's partial <dh, h> (in order), ds_j = (dg_j - sum_i dg_i g_i)
//   / S with S the sum of the winners' scores (renormalised gates) or dg_j (raw),
//   dz_j = ds_j s_j (1 - s_j) -> dzp[padded row of pair j],
//   dx_t = dxs_t + sum_j (dxp[padded row j] + dz_j W_r[e_j]) (+ dout_t),
// summed in fp32 (16-byte loads, 8 columns a lane), rounded once to bf16.  dgate
// (optional) receives dg per pair.
__global__ void router_bwd_dx_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate,
                                     const float* __restrict__ scores, const int32_t* __restrict__ inv_pad,
                                     const float* __restrict__ dgp, int nparts,
                                     const float* __restrict__ w_router, const uint16_t* __restrict__ dxp,
                                     const uint16_t* __restrict__ dxs, const uint16_t* __restrict__ dout,
                                     int T, int d, int E, int k, int renorm, float* __restrict__ dzp,
                                     float* __restrict__ dgate, uint16_t* __restrict__ dx) {
  const int lane = threadIdx.x % 32;
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  float dg = 0.f, g = 0.f, sc = 0.f;
  int e = 0, q = 0;
  if (lane < k) {
    e = idx[(size_t)t * k + lane];
    q = inv_pad[(size_t)t * k + lane];
    for (int p = 0; p < nparts; ++p) dg += dgp[(size_t)q * nparts + p];
    g = gate[(size_t)t * k + lane];
    sc = scores[(size_t)t * E + e];
    if (dgate) dgate[(size_t)t * k + lane] = dg;
  }
  float S = sc, dgg = dg * g;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
    dgg += __shfl_xor_sync(0xFFFFFFFFu, dgg, o);
  }
  const float dz = (renorm ? (dg - dgg) / S : dg) * sc * (1.0f - sc);
  if (lane < k) dzp[q] = dz;
  for (int c = 8 * lane; c < d; c += 256) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
    auto add8 = [&](const uint16_t* src) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] += __uint_as_float(w4[i] << 16);
        v[2 * i + 1] += __uint_as_float(w4[i] & 0xFFFF0000u);
      }
    };
    if (dxs) add8(dxs + (size_t)t * d + c);
    for (int j = 0; j < k; ++j) {
      const int qj = __shfl_sync(0xFFFFFFFFu, q, j);
      const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
      const float zj = __shfl_sync(0xFFFFFFFFu, dz, j);
      add8(dxp + (size_t)qj * d + c);
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w_router + (size_t)ej * d + c));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w_router + (size_t)ej * d + c + 4));
      v[0] = fmaf(zj, w0.x, v[0]);
      v[1] = fmaf(zj, w0.y, v[1]);
      v[2] = fmaf(zj, w0.z, v[2]);
      v[3] = fmaf(zj, w0.w, v[3]);
      v[4] = fmaf(zj, w1.x, v[4]);
      v[5] = fmaf(zj, w1.y, v[5]);
      v[6] = fmaf(zj, w1.z, v[6]);
      v[7] = fmaf(zj, w1.w, v[7]);
    }
    if (dout) add8(dout + (size_t)t * d + c);
    uint4 o;
    o.x = __bfloat16_as_ushort(__float2bfloat16_rn(v[0])) | ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[1])) << 16);
    o.y = __bfloat16_as_ushort(__float2bfloat16_rn(v[2])) | ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[3])) << 16);
    o.z = __bfloat16_as_ushort(__float2bfloat16_rn(v[4])) | ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[5])) << 16);
    o.w = __bfloat16_as_ushort(__float2bfloat16_rn(v[6])) | ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[7])) << 16);
    *reinterpret_cast<uint4*>(dx + (size_t)t * d + c) = o;
  }
}

// dW_r[e][c] = sum over expert e's rows q of dzp[q] * xp[q][c] (padded layout).
// Block (256 columns, expert e), 8 warps: warp w takes rows w, w + 8, ... with 8
// columns a lane (16-byte loads, four rows in flight); the warps' partial sums are
// added in warp order through shared memory, so the result is deterministic.
__global__ void router_wgrad_kernel(const float* __restrict__ dzp, const int32_t* __restrict__ off,
                                    const int32_t* __restrict__ poff, const uint16_t* __restrict__ xp,
                                    int d, float* __restrict__ dwr) {
  __shared__ float part[8][256];
  const int e = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = blockIdx.x * 256 + 8 * lane;
  const int q0 = poff[e], n = off[e + 1] - off[e];
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (c < d) {
    int r = warp;
    for (; r + 24 < n; r += 32) {
      uint4 u[4];
      float z[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        u[j] = __ldg(reinterpret_cast<const uint4*>(xp + (size_t)(q0 + r + 8 * j) * d + c));
        z[j] = dzp[q0 + r + 8 * j];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w4[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(z[j], __uint_as_float(w4[i] << 16), acc[2 * i]);
          acc[2 * i + 1] = fmaf(z[j], __uint_as_float(w4[i] & 0xFFFF0000u), acc[2 * i + 1]);
        }
      }
    }
    for (; r < n; r += 8) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(xp + (size_t)(q0 + r) * d + c));
      const float z = dzp[q0 + r];
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(z, __uint_as_float(w4[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(z, __uint_as_float(w4[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[warp][8 * lane + i] = acc[i];
  __syncthreads();
  const int col = blockIdx.x * 256 + threadIdx.x;
  if (col < d) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += part[w][threadIdx.x];
    dwr[(size_t)e * d + col] = sum;
  }
}

}  // namespace

cudaError_t launch_pad_map(const int32_t* off, const int32_t* perm_tok, const int32_t* idx,
                           const int32_t* inv_pos, const float* gate, int E, long long pairs,
                           long long q_max, int32_t* poff, int32_t* tok_pad, int32_t* inv_pad,
                           float* gperm, cudaStream_t s) {
  const long long n = std::max(q_max, pairs);
  pad_map_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(off, perm_tok, idx, inv_pos, gate, E, pairs,
                                                             q_max, poff, tok_pad, inv_pad, gperm);
  return cudaGetLastError();
}

cudaError_t launch_gather_pad(const uint16_t* x, const uint16_t* dout, const int32_t* tok_pad,
                              long long q_max, const int32_t* rows_limit, int d, uint16_t* xp,
                              uint16_t* dp, cudaStream_t s) {
  const long long n = q_max * (d / 8);
  gather_pad_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, dout, tok_pad, q_max, rows_limit, d, xp, dp);
  return cudaGetLastError();
}

cudaError_t launch_router_bwd_dx(const int32_t* idx, const float* gate, const float* scores,
                                 const int32_t* inv_pad, const float* dgp, int nparts, const float* w_router,
                                 const uint16_t* dxp, const uint16_t* dxs, const uint16_t* dout, int T,
                                 int d, int E, int k, int renorm, float* dzp, float* dgate, uint16_t* dx,
                                 cudaStream_t s) {
  router_bwd_dx_kernel<<<(unsigned)((T + 7) / 8), 256, 0, s>>>(idx, gate, scores, inv_pad, dgp, nparts,
                                                               w_router, dxp, dxs, dout, T, d, E, k, renorm,
                                                               dzp, dgate, dx);
  return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const float* dzp, const int32_t* off, const int32_t* poff,
                                const uint16_t* xp, int d, int E, float* dwr, cudaStream_t s) {
  router_wgrad_kernel<<<dim3((unsigned)((d + 255) / 256), (unsigned)E), 256, 0, s>>>(dzp, off, poff, xp, d,
                                                                                   dwr);
  return cudaGetLastError();
}

}  // namespace moe
