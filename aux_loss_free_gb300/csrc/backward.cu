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
// zero in every operand).  One launch builds it and gathers the rows:
//   - every block derives poff from the offsets in shared memory (one warp, E <= 256);
//     block 0 stores it;
//   - thread i < pairs writes pair i's padded row inv_pad[i] and gperm[inv_pad[i]] =
//     gate[i];
//   - block b's warps copy padded rows [64 b, 64 b + 64) below poff[E]: xp[q] = x[tok],
//     dp[q] = dout[tok] for the row's token, zero rows (and a zero gate) for padding;
//     a lane keeps all of its 16-byte loads of both rows in flight before storing.
constexpr int PAD_ROWS = 64;

__global__ void __launch_bounds__(256) pad_gather_kernel(
    const int32_t* __restrict__ off, const int32_t* __restrict__ perm_tok, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ inv_pos, const float* __restrict__ gate, int E, long long pairs,
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ dout, int d, int32_t* __restrict__ poff_out,
    int32_t* __restrict__ inv_pad, float* __restrict__ gperm, uint16_t* __restrict__ xp,
    uint16_t* __restrict__ dp) {
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
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) poff_out[e] = s_poff[e];
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < pairs) {
    const int e = idx[i];
    const int q = s_poff[e] + (inv_pos[i] - s_off[e]);
    inv_pad[i] = q;
    gperm[q] = gate[i];
  }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int vpr = d / 8;  // 16-byte vectors per row (d <= 8192: at most 32 per lane)
  for (int rr = warp; rr < PAD_ROWS; rr += 8) {
    const long long q = (long long)blockIdx.x * PAD_ROWS + rr;
    if (q >= s_poff[E]) break;
    int lo = 0, hi = E - 1;  // last expert with s_poff <= q
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_poff[mid] <= q) lo = mid; else hi = mid - 1;
    }
    const long long r = s_off[lo] + (q - s_poff[lo]);
    const int tok = r < s_off[lo + 1] ? perm_tok[r] : -1;
    uint4* xo = reinterpret_cast<uint4*>(xp + q * d);
    uint4* dq = reinterpret_cast<uint4*>(dp + q * d);
    if (tok < 0) {
      if (lane == 0) gperm[q] = 0.f;  // padding rows carry a zero gate (never garbage)
      for (int v = lane; v < vpr; v += 32) xo[v] = dq[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* xi = reinterpret_cast<const uint4*>(x + (size_t)tok * d);
    const uint4* di = reinterpret_cast<const uint4*>(dout + (size_t)tok * d);
    for (int v0 = 0; v0 < vpr; v0 += 128) {  // 4 vectors of each row per lane in flight
      uint4 a[4], g[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = v0 + lane + 32 * j;
        if (v < vpr) {
          a[j] = __ldg(xi + v);
          g[j] = __ldg(di + v);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = v0 + lane + 32 * j;
        if (v < vpr) {
          xo[v] = a[j];
          dq[v] = g[j];
        }
      }
    }
  }
}

// Router backward and the input gradient, one warp per token (lane j < k holds pair j):
//   dg_j = sum of the pair's partial <dh, h> (in order), ds_j = (dg_j - sum_i dg_i g_i)
//   / S with S the sum of the winners' scores (renormalised gates) or dg_j (raw),
//   dz_j = ds_j s_j (1 - s_j) -> dzp[padded row of pair j],
//   dx_t = dxs_t (+ dxs2_t) + sum_j (dxp[padded row j] + dz_j W_r[e_j]) (+ dout_t),
// summed in fp32 (16-byte loads, 8 columns a lane), rounded once to bf16.  dgate
// (optional) receives dg per pair.
// KT: pairs held in registers (k <= KT).
template <int KT>
__global__ void router_bwd_dx_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate,
                                     const float* __restrict__ scores, const int32_t* __restrict__ inv_pad,
                                     const float* __restrict__ dgp, int nparts,
                                     const float* __restrict__ w_router, const uint16_t* __restrict__ dxp,
                                     const uint16_t* __restrict__ dxs, const uint16_t* __restrict__ dxs2,
                                     const uint16_t* __restrict__ dout,
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
  // Every lane's copy of the pairs' rows, experts and dz (shuffles while all lanes are
  // converged: the column loop below runs a lane-dependent number of steps).
  int qa[KT], ea[KT];
  float za[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    qa[j] = __shfl_sync(0xFFFFFFFFu, q, j);
    ea[j] = __shfl_sync(0xFFFFFFFFu, e, j);
    za[j] = __shfl_sync(0xFFFFFFFFu, dz, j);
  }
  // Two blocks of 8 columns per lane per step, every load of both issued before use.
  for (int c0 = 8 * lane; c0 < d; c0 += 512) {
    const bool two = c0 + 256 < d;  // lane-dependent when d is not a multiple of 512
    float v[2][8];
    uint4 u_s[2], u_s2[2], u_d[2], u_p[2][KT];
    float4 w_r[2][KT][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + 256 * h;
      if (h == 1 && !two) break;
      if (dxs) u_s[h] = __ldg(reinterpret_cast<const uint4*>(dxs + (size_t)t * d + c));
      if (dxs2) u_s2[h] = __ldg(reinterpret_cast<const uint4*>(dxs2 + (size_t)t * d + c));
      if (dout) u_d[h] = __ldg(reinterpret_cast<const uint4*>(dout + (size_t)t * d + c));
#pragma unroll
      for (int j = 0; j < KT; ++j) {
        if (j >= k) break;
        const int qj = qa[j], ej = ea[j];
        u_p[h][j] = __ldg(reinterpret_cast<const uint4*>(dxp + (size_t)qj * d + c));
        w_r[h][j][0] = __ldg(reinterpret_cast<const float4*>(w_router + (size_t)ej * d + c));
        w_r[h][j][1] = __ldg(reinterpret_cast<const float4*>(w_router + (size_t)ej * d + c + 4));
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + 256 * h;
      if (h == 1 && !two) break;
#pragma unroll
      for (int i = 0; i < 8; ++i) v[h][i] = 0.f;
      auto add8 = [&](const uint4& u) {
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[h][2 * i] += __uint_as_float(w4[i] << 16);
          v[h][2 * i + 1] += __uint_as_float(w4[i] & 0xFFFF0000u);
        }
      };
      if (dxs) add8(u_s[h]);
      if (dxs2) add8(u_s2[h]);
#pragma unroll
      for (int j = 0; j < KT; ++j) {
        if (j >= k) break;
        const float zj = za[j];
        add8(u_p[h][j]);
        const float4 w0 = w_r[h][j][0], w1 = w_r[h][j][1];
        v[h][0] = fmaf(zj, w0.x, v[h][0]);
        v[h][1] = fmaf(zj, w0.y, v[h][1]);
        v[h][2] = fmaf(zj, w0.z, v[h][2]);
        v[h][3] = fmaf(zj, w0.w, v[h][3]);
        v[h][4] = fmaf(zj, w1.x, v[h][4]);
        v[h][5] = fmaf(zj, w1.y, v[h][5]);
        v[h][6] = fmaf(zj, w1.z, v[h][6]);
        v[h][7] = fmaf(zj, w1.w, v[h][7]);
      }
      if (dout) add8(u_d[h]);
      uint4 o;
      o.x = __bfloat16_as_ushort(__float2bfloat16_rn(v[h][0])) |
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[h][1])) << 16);
      o.y = __bfloat16_as_ushort(__float2bfloat16_rn(v[h][2])) |
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[h][3])) << 16);
      o.z = __bfloat16_as_ushort(__float2bfloat16_rn(v[h][4])) |
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[h][5])) << 16);
      o.w = __bfloat16_as_ushort(__float2bfloat16_rn(v[h][6])) |
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[h][7])) << 16);
      *reinterpret_cast<uint4*>(dx + (size_t)t * d + c) = o;
    }
  }
}

// dW_r[e][c] = sum over expert e's rows q of dzp[q] * xp[q][c] (padded layout).
// Block (256 columns, expert e), 8 warps: warp w takes rows w, w + 8, ... with 8
// columns a lane (16-byte loads, eight rows in flight); the warps' partial sums are
// added in warp order through shared memory, so the result is deterministic.
__global__ void __launch_bounds__(256, 2) router_wgrad_kernel(const float* __restrict__ dzp, const int32_t* __restrict__ off,
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
    // Sixteen rows of a warp in flight per step, then eight, then one at a time: each
    // warp still adds its rows warp, warp + 8, ... in ascending order.
    for (; r + 120 < n; r += 128) {
      uint4 u[16];
      float z[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        u[j] = __ldg(reinterpret_cast<const uint4*>(xp + (size_t)(q0 + r + 8 * j) * d + c));
        z[j] = dzp[q0 + r + 8 * j];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t w4[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(z[j], __uint_as_float(w4[i] << 16), acc[2 * i]);
          acc[2 * i + 1] = fmaf(z[j], __uint_as_float(w4[i] & 0xFFFF0000u), acc[2 * i + 1]);
        }
      }
    }
    for (; r + 56 < n; r += 64) {
      uint4 u[8];
      float z[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        u[j] = __ldg(reinterpret_cast<const uint4*>(xp + (size_t)(q0 + r + 8 * j) * d + c));
        z[j] = dzp[q0 + r + 8 * j];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
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

cudaError_t launch_pad_gather(const int32_t* off, const int32_t* perm_tok, const int32_t* idx,
                              const int32_t* inv_pos, const float* gate, int E, long long pairs,
                              long long q_max, const uint16_t* x, const uint16_t* dout, int d,
                              int32_t* poff, int32_t* inv_pad, float* gperm, uint16_t* xp, uint16_t* dp,
                              cudaStream_t s) {
  const long long blocks = std::max((q_max + PAD_ROWS - 1) / PAD_ROWS, (pairs + 255) / 256);
  pad_gather_kernel<<<(unsigned)blocks, 256, 0, s>>>(off, perm_tok, idx, inv_pos, gate, E, pairs, x, dout, d,
                                                     poff, inv_pad, gperm, xp, dp);
  return cudaGetLastError();
}

cudaError_t launch_router_bwd_dx(const int32_t* idx, const float* gate, const float* scores,
                                 const int32_t* inv_pad, const float* dgp, int nparts, const float* w_router,
                                 const uint16_t* dxp, const uint16_t* dxs, const uint16_t* dxs2,
                                 const uint16_t* dout, int T,
                                 int d, int E, int k, int renorm, float* dzp, float* dgate, uint16_t* dx,
                                 cudaStream_t s) {
  const unsigned blocks = (unsigned)((T + 7) / 8);
  if (k <= 2)
    router_bwd_dx_kernel<2><<<blocks, 256, 0, s>>>(idx, gate, scores, inv_pad, dgp, nparts, w_router, dxp, dxs,
                                                   dxs2, dout, T, d, E, k, renorm, dzp, dgate, dx);
  else
    router_bwd_dx_kernel<kMaxK><<<blocks, 256, 0, s>>>(idx, gate, scores, inv_pad, dgp, nparts, w_router, dxp,
                                                       dxs, dxs2, dout, T, d, E, k, renorm, dzp, dgate, dx);
  return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const float* dzp, const int32_t* off, const int32_t* poff,
                                const uint16_t* xp, int d, int E, float* dwr, cudaStream_t s) {
  router_wgrad_kernel<<<dim3((unsigned)((d + 255) / 256), (unsigned)E), 256, 0, s>>>(dzp, off, poff, xp, d,
                                                                                   dwr);
  return cudaGetLastError();
}

}  // namespace moe
