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

// SwiGLU backward, one warp per row, in place.  ab: [rows][2w] pre-activations, gate
// and up columns interleaved in blocks of `block` (as the packed weights' rows);
// dh: [rows][w] = dout Wd (the gate not yet applied).  With g = gperm[row] (1 when
// gperm is null), h = silu(a) * b, dh' = g * dh:
//   ab <- (dh' * b * silu'(a), dh' * silu(a))   (same interleave),
//   dh <- g * h   (the down projection's weight-gradient operand),
//   dg[row] = <dh, h>   (when dg is set: the gate's gradient <dout, y>).
// Rows at or past *rows_limit (when set) are left alone.
__global__ void swiglu_bwd_kernel(uint16_t* __restrict__ ab, uint16_t* __restrict__ dh,
                                  const float* __restrict__ gperm, long long rows,
                                  const int32_t* __restrict__ rows_limit, int w, int block,
                                  float* __restrict__ dg) {
  const long long r = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (r >= rows || (rows_limit && r >= *rows_limit)) return;
  const float g = gperm ? gperm[r] : 1.0f;
  uint16_t* abr = ab + r * 2 * w;
  uint16_t* dhr = dh + r * w;
  float dot = 0.f;
  for (int j0 = 2 * lane; j0 < w; j0 += 64) {  // pairs of columns (block is even)
    const int blk = j0 / block, within = j0 % block;
    const long long cg = (long long)blk * 2 * block + within, cu = cg + block;
    const __nv_bfloat162 a2 = *reinterpret_cast<const __nv_bfloat162*>(abr + cg);
    const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(abr + cu);
    const __nv_bfloat162 d2 = *reinterpret_cast<const __nv_bfloat162*>(dhr + j0);
    const float a[2] = {__low2float(a2), __high2float(a2)};
    const float b[2] = {__low2float(b2), __high2float(b2)};
    const float dd[2] = {__low2float(d2), __high2float(d2)};
    float da[2], db[2], hg[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float sig = 1.0f / (1.0f + __expf(-a[i]));
      const float sa = a[i] * sig;
      const float h = sa * b[i];
      dot = fmaf(dd[i], h, dot);
      const float dhg = g * dd[i];
      da[i] = dhg * b[i] * (sig * (1.0f + a[i] * (1.0f - sig)));
      db[i] = dhg * sa;
      hg[i] = g * h;
    }
    *reinterpret_cast<__nv_bfloat162*>(abr + cg) = __floats2bfloat162_rn(da[0], da[1]);
    *reinterpret_cast<__nv_bfloat162*>(abr + cu) = __floats2bfloat162_rn(db[0], db[1]);
    *reinterpret_cast<__nv_bfloat162*>(dhr + j0) = __floats2bfloat162_rn(hg[0], hg[1]);
  }
  if (dg) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
    if (lane == 0) dg[r] = dot;
  }
}

// Router backward and the input gradient, one block per token:
//   ds_j = (dg_j - sum_i dg_i g_i) / S (renormalised gates, S = sum of the winners'
//   scores) or dg_j (raw), dz_j = ds_j s_j (1 - s_j)  -> dzp[padded row of pair j],
//   dx_t = sum_j dxp[padded row j] + dxs_t + sum_j dz_j W_r[e_j] (+ dout_t),
// summed in fp32, rounded once to bf16.  dgate (optional) receives dg per pair.
__global__ void router_bwd_dx_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate,
                                     const float* __restrict__ scores, const int32_t* __restrict__ inv_pad,
                                     const float* __restrict__ dgp, const float* __restrict__ w_router,
                                     const uint16_t* __restrict__ dxp, const uint16_t* __restrict__ dxs,
                                     const uint16_t* __restrict__ dout, int d, int E, int k, int renorm,
                                     float* __restrict__ dzp, float* __restrict__ dgate,
                                     uint16_t* __restrict__ dx) {
  const int t = blockIdx.x;
  __shared__ float s_dz[kMaxK];
  __shared__ int s_e[kMaxK];
  __shared__ int s_q[kMaxK];
  if (threadIdx.x == 0) {
    float dg[kMaxK], g[kMaxK], sc[kMaxK], S = 0.f, dgg = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      const int q = inv_pad[(size_t)t * k + j];
      s_e[j] = e;
      s_q[j] = q;
      dg[j] = dgp[q];
      g[j] = gate[(size_t)t * k + j];
      sc[j] = scores[(size_t)t * E + e];
      S += sc[j];
      dgg = fmaf(dg[j], g[j], dgg);
      if (dgate) dgate[(size_t)t * k + j] = dg[j];
    }
    for (int j = 0; j < k; ++j) {
      const float ds = renorm ? (dg[j] - dgg) / S : dg[j];
      s_dz[j] = ds * sc[j] * (1.0f - sc[j]);
      dzp[s_q[j]] = s_dz[j];
    }
  }
  __syncthreads();
  for (int c = 2 * threadIdx.x; c < d; c += 2 * blockDim.x) {
    float v0 = 0.f, v1 = 0.f;
    if (dxs) {
      const __nv_bfloat162 u = *reinterpret_cast<const __nv_bfloat162*>(dxs + (size_t)t * d + c);
      v0 = __low2float(u);
      v1 = __high2float(u);
    }
    for (int j = 0; j < k; ++j) {
      const __nv_bfloat162 u = *reinterpret_cast<const __nv_bfloat162*>(dxp + (size_t)s_q[j] * d + c);
      const float2 wr = *reinterpret_cast<const float2*>(w_router + (size_t)s_e[j] * d + c);
      v0 += __low2float(u);
      v1 += __high2float(u);
      v0 = fmaf(s_dz[j], wr.x, v0);
      v1 = fmaf(s_dz[j], wr.y, v1);
    }
    if (dout) {
      const __nv_bfloat162 u = *reinterpret_cast<const __nv_bfloat162*>(dout + (size_t)t * d + c);
      v0 += __low2float(u);
      v1 += __high2float(u);
    }
    *reinterpret_cast<__nv_bfloat162*>(dx + (size_t)t * d + c) = __floats2bfloat162_rn(v0, v1);
  }
}

// dW_r[e][c] = sum over expert e's rows q of dzp[q] * xp[q][c] (padded layout; rows
// in order, so the sum is deterministic).  Block (e, 512 columns), 2 columns a thread.
__global__ void router_wgrad_kernel(const float* __restrict__ dzp, const int32_t* __restrict__ off,
                                    const int32_t* __restrict__ poff, const uint16_t* __restrict__ xp,
                                    int d, float* __restrict__ dwr) {
  const int e = blockIdx.y;
  const int c = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (c >= d) return;
  const int q0 = poff[e], n = off[e + 1] - off[e];
  float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
  for (int i = 0; i < n; ++i) {
    const float z = dzp[q0 + i];
    const __nv_bfloat162 u = *reinterpret_cast<const __nv_bfloat162*>(xp + (size_t)(q0 + i) * d + c);
    a0 = fmaf(z, __low2float(u), a0);
    a1 = fmaf(z, __high2float(u), a1);
  }
  *reinterpret_cast<float2*>(dwr + (size_t)e * d + c) = make_float2(a0, a1);
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

cudaError_t launch_swiglu_bwd(uint16_t* ab, uint16_t* dh, const float* gperm, long long rows,
                              const int32_t* rows_limit, int w, int block, float* dg, cudaStream_t s) {
  swiglu_bwd_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(ab, dh, gperm, rows, rows_limit, w, block, dg);
  return cudaGetLastError();
}

cudaError_t launch_router_bwd_dx(const int32_t* idx, const float* gate, const float* scores,
                                 const int32_t* inv_pad, const float* dgp, const float* w_router,
                                 const uint16_t* dxp, const uint16_t* dxs, const uint16_t* dout, int T,
                                 int d, int E, int k, int renorm, float* dzp, float* dgate, uint16_t* dx,
                                 cudaStream_t s) {
  router_bwd_dx_kernel<<<T, 128, 0, s>>>(idx, gate, scores, inv_pad, dgp, w_router, dxp, dxs, dout, d, E, k,
                                         renorm, dzp, dgate, dx);
  return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const float* dzp, const int32_t* off, const int32_t* poff,
                                const uint16_t* xp, int d, int E, float* dwr, cudaStream_t s) {
  router_wgrad_kernel<<<dim3((unsigned)((d / 2 + 255) / 256), (unsigned)E), 256, 0, s>>>(dzp, off, poff, xp,
                                                                                       d, dwr);
  return cudaGetLastError();
}

}  // namespace moe
