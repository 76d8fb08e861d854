// Token permutation (stable counting sort by expert), row gather, combine, bias
// update and weight packing.
//
// Counting sort in two launches: per-chunk expert counts (the router produces them
// on the fused path) and one scatter launch in which every block derives its
// chunk's bases from the count table and ranks its pairs (see scatter_kernel).  The
// scatter also gathers the token rows into the permuted activation buffer the
// grouped GEMM reads.
#include <cuda_bf16.h>

#include "internal.h"
#include "select.cuh"

namespace moe {
namespace {

constexpr unsigned FULL = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Copy one token row (d elements) to a bf16 destination row with one warp.  For bf16
// rows every lane issues all of its 16-byte loads before its stores (up to 8 in
// flight per lane), which the copy needs to reach HBM bandwidth.
__device__ __forceinline__ void copy_row_bf16(const void* x, int x_is_f32, long long src_row, int d,
                                              uint16_t* dst, int lane) {
  const int nvec = d / 8;  // 8 bf16 = 16 bytes per vector
  uint4* out = reinterpret_cast<uint4*>(dst);
  if (!x_is_f32 && nvec <= 256) {
    const uint4* in = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + src_row * d);
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane + 32 * j < nvec) v[j] = __ldg(in + lane + 32 * j);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane + 32 * j < nvec) out[lane + 32 * j] = v[j];
    return;
  }
  if (x_is_f32) {
    const float4* in = reinterpret_cast<const float4*>(static_cast<const float*>(x) + src_row * d);
    for (int v = lane; v < nvec; v += 32) {
      const float4 a = in[2 * v], b = in[2 * v + 1];
      out[v] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                          pack_bf16x2(b.z, b.w));
    }
  } else {
    const uint4* in = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + src_row * d);
    for (int v = lane; v < nvec; v += 32) out[v] = in[v];
  }
}

__global__ void count_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int chunk_tokens,
                             int32_t* __restrict__ counts, int* status) {
  const long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= (long long)T * k) return;
  const int t = (int)(p / k);
  const int e = idx[p];
  if (e < 0 || e >= E) {  // not counted: a bad id must not write past the count table
    atomicOr(status, kDevCheck);
    return;
  }
  atomicAdd(&counts[(long long)(t / chunk_tokens) * E + e], 1);
}

constexpr int SC_THREADS = 256;
constexpr int SC_ROUND = 256;  // pairs ranked per round (8 warp batches)

// One launch does the whole permutation from the per-chunk count table:
//  1. every block reads the table (a few KB, one batched L2 round trip) and forms,
//     for each expert, the pairs of earlier chunks and the expert totals; the
//     totals' exclusive scan gives the expert offsets (block 0 also writes them,
//     the loads and, if asked, the bias update);
//  2. a block of 32 tokens adds the pairs of the earlier blocks of its chunk;
//  3. the block ranks its own pairs in (token, slot) order with a warp match, which
//     keeps tokens ascending inside every expert's rows, writes perm_tok / inv_pos
//     and gathers the token rows (16-byte vectors) into the permuted activations.
__global__ void __launch_bounds__(SC_THREADS) scatter_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ counts, int chunks, int T, int k,
    int E, int chunk_tokens, int32_t* __restrict__ offsets, int32_t* __restrict__ load_out,
    float* bias, float gamma, long long tokens_times_k, int32_t* __restrict__ perm_tok,
    int32_t* __restrict__ inv_pos, const void* __restrict__ x, int x_is_f32, int d,
    uint16_t* __restrict__ xp, uint16_t* __restrict__ xb, int32_t* __restrict__ active,
    moe_balance_t* __restrict__ balance, int* status) {
  __shared__ int32_t run[kMaxE];
  __shared__ int32_t tot_e[kMaxE];
  __shared__ int32_t off[kMaxE + 1];
  __shared__ int32_t part_pre[SC_THREADS];
  __shared__ int32_t part_tot[SC_THREADS];
  __shared__ int32_t s_pos[SC_ROUND];
  __shared__ int32_t s_tok[SC_ROUND];
  asm volatile("griddepcontrol.wait;" ::: "memory");  // counts / idx come from the router
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int block_tokens = chunk_tokens <= 128 ? 32 : chunk_tokens;
  const long long t_begin = (long long)blockIdx.x * block_tokens;
  const long long chunk = t_begin / chunk_tokens;
  const long long p_begin = t_begin * k;
  const long long p_end = min((long long)T * k, p_begin + (long long)block_tokens * k);

  // ---- 1. chunk prefix and totals per expert
  const int parts = SC_THREADS / E;
  const int e = tid % E, part = tid / E;
  if (part < parts) {
    const int L = (chunks + parts - 1) / parts;
    const int lo = part * L, hi = min(chunks, lo + L);
    int pre = 0, tot = 0;
    for (int c0 = lo; c0 < hi; c0 += 16) {
      int v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = (c0 + j < hi) ? __ldcg(&counts[(long long)(c0 + j) * E + e]) : 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        tot += v[j];
        if (c0 + j < chunk) pre += v[j];
      }
    }
    part_pre[part * E + e] = pre;
    part_tot[part * E + e] = tot;
  }
  __syncthreads();
  if (tid < E) {
    int pre = 0, tot = 0;
    for (int q = 0; q < parts; ++q) {
      pre += part_pre[q * E + tid];
      tot += part_tot[q * E + tid];
    }
    run[tid] = pre;
    tot_e[tid] = tot;
  }
  __syncthreads();
  if (tid < 32) {  // exclusive scan of the totals over experts, 32 at a time
    int carry = 0;
    for (int b = 0; b < E; b += 32) {
      const int v = (b + tid < E) ? tot_e[b + tid] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(FULL, incl, o);
        if (tid >= o) incl += n;
      }
      if (b + tid < E) off[b + tid] = carry + incl - v;
      carry += __shfl_sync(FULL, incl, 31);
    }
    if (tid == 0) off[E] = carry;
  }
  __syncthreads();
  if (tid < E) run[tid] += off[tid];
  if (blockIdx.x == 0) {
    if (active && tid < 32) {  // compact list of the experts with pairs, ascending
      int n = 0;
      for (int b = 0; b < E; b += 32) {
        const bool has = b + tid < E && tot_e[b + tid] > 0;
        const unsigned m = __ballot_sync(FULL, has);
        if (has) active[n + __popc(m & ((1u << tid) - 1u))] = b + tid;
        n += __popc(m);
      }
      if (tid == 0) active[kMaxE] = n;
    }
    for (int i = tid; i <= E; i += SC_THREADS) offsets[i] = off[i];
    if (balance && warp == 1) warp_balance(tot_e, E, balance, lane);
    if (tid < E) {
      if (load_out) load_out[tid] = tot_e[tid];
      // Aux-loss-free update: sign(T*k - E*load) is sign(target - load), sign(0) = 0.
      if (bias) bias[tid] = biased_step(bias[tid], tokens_times_k, E, tot_e[tid], gamma);
    }
  }
  __syncthreads();

  // ---- 2. pairs of the earlier blocks of the same chunk come first
  for (long long q = chunk * chunk_tokens * k + tid; q < p_begin; q += SC_THREADS) {
    const int ex = idx[q];
    if (ex >= 0 && ex < E) atomicAdd(&run[ex], 1);
  }
  __syncthreads();

  // ---- 3. rank, scatter, gather
  for (long long r0 = p_begin; r0 < p_end; r0 += SC_ROUND) {
    const int n = (int)min((long long)SC_ROUND, p_end - r0);
    if (warp == 0) {
      for (int b = 0; b < n; b += 32) {
        const int q = b + lane;
        int ex = q < n ? idx[r0 + q] : -1;
        if (q < n && (ex < 0 || ex >= E)) {  // a bad id is not ranked (the count skipped it)
          atomicOr(status, kDevCheck);
          ex = -1;
        }
        const bool valid = ex >= 0;
        const unsigned peers = __match_any_sync(FULL, ex);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (q < n && !valid) s_pos[q] = -1;  // the row gather skips it
        if (valid) {
          const int pos = run[ex] + rank;
          const long long pr = r0 + q;
          const int t = (int)(pr / k);
          perm_tok[pos] = t;
          inv_pos[pr] = pos;
          s_pos[q] = pos;
          s_tok[q] = (pr % k == 0) ? t : -1 - t;  // slot 0 marks the token's first pair
        }
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) run[ex] += __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
    if (xp) {
#pragma unroll 2
      for (int q = warp; q < n; q += SC_THREADS / 32) {
        if (s_pos[q] < 0) continue;
        const int st = s_tok[q];
        const int t = st >= 0 ? st : -1 - st;
        copy_row_bf16(x, x_is_f32, t, d, xp + (long long)s_pos[q] * d, lane);
        if (xb && st >= 0) copy_row_bf16(x, x_is_f32, t, d, xb + (long long)t * d, lane);
      }
    }
    __syncthreads();
  }
}

__global__ void gather_kernel(const void* __restrict__ x, int x_is_f32,
                              const int32_t* __restrict__ perm_tok, long long rows, int d,
                              uint16_t* __restrict__ xp) {
  const long long r = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= rows) return;
  copy_row_bf16(x, x_is_f32, perm_tok[r], d, xp + r * d, threadIdx.x % 32);
}

__global__ void to_bf16_kernel(const float* __restrict__ x, long long n8, uint16_t* __restrict__ xb) {
  const long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(x)[2 * v];
  const float4 b = reinterpret_cast<const float4*>(x)[2 * v + 1];
  reinterpret_cast<uint4*>(xb)[v] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                               pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
}

// One block of 256 threads (E <= 256).  tokens_times_k < 0: the global T*k is the sum
// of the loads (each token contributes k pairs), taken here so that no host round trip
// is needed after the loads were summed over replicas.
__global__ void bias_update_kernel(int E, long long tokens_times_k, const int32_t* __restrict__ load,
                                   float gamma, float* bias, moe_balance_t* balance) {
  __shared__ long long s_part[8];
  const int e = threadIdx.x, warp = e / 32, lane = e % 32;
  const int v = e < E ? load[e] : 0;
  if (balance && warp == 0) warp_balance(load, E, balance, lane);
  if (tokens_times_k < 0) {
    long long s = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
    if (lane == 0) s_part[warp] = s;
    __syncthreads();
    tokens_times_k = 0;
    for (int w = 0; w < (int)(blockDim.x / 32); ++w) tokens_times_k += s_part[w];
  }
  if (e >= E || !bias) return;
  bias[e] = biased_step(bias[e], tokens_times_k, E, v, gamma);
}

// out[t] = residual[t] + shared[t] + sum_j gate[t][j] * y[inv_pos[t][j]]; one thread per
// 16 output columns (32-byte loads and stores when every row starts on a 32-byte
// boundary, else two 16-byte halves), fp32 sum, one rounding to bf16.
__device__ __forceinline__ void load16_bf16(const uint16_t* row, int v8, uint32_t (&w)[8]) {
  if (v8) {
    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                   "=r"(w[7])
                 : "l"(row));
  } else {
    const uint4 a = reinterpret_cast<const uint4*>(row)[0], b = reinterpret_cast<const uint4*>(row)[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
}

// out[t] = residual[t] + shared[t] + sum_j gate[t][j] * y[inv_pos[t][j]] (y[t * k + j]
// without inv_pos), 16 columns per thread.  With KC = k (1 or 2) every row load of a thread is issued before the
// first use, so only the inv_pos -> y dependency is exposed; KC = 0 loops over k.
template <int KC>
__global__ void combine_kernel(const uint16_t* __restrict__ y, const uint16_t* __restrict__ shared,
                               const int32_t* __restrict__ inv_pos, const float* __restrict__ gate,
                               const uint16_t* __restrict__ residual, uint16_t* __restrict__ out,
                               int T, int k, int d, int v8) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // y / shared come from the GEMM
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int vpr = d / 16;
  const long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= (long long)T * vpr) return;
  const long long t = v / vpr;
  const int c = (int)(v % vpr) * 16;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  auto add = [&](const uint32_t (&ws)[8], float w) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      acc[2 * i] = fmaf(w, bf16_lo(ws[i]), acc[2 * i]);
      acc[2 * i + 1] = fmaf(w, bf16_hi(ws[i]), acc[2 * i + 1]);
    }
  };
  if (KC > 0) {
    int pos[KC > 0 ? KC : 1];
    float g[KC > 0 ? KC : 1];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      pos[j] = inv_pos ? inv_pos[t * KC + j] : (int)(t * KC + j);
      g[j] = gate[t * KC + j];
    }
    uint32_t wr[8], wsh[8], wy[KC > 0 ? KC : 1][8];
    if (residual) load16_bf16(residual + t * d + c, v8, wr);
    if (shared) load16_bf16(shared + t * d + c, v8, wsh);
#pragma unroll
    for (int j = 0; j < KC; ++j) load16_bf16(y + (long long)pos[j] * d + c, v8, wy[j]);
    if (residual) add(wr, 1.f);
    if (shared) add(wsh, 1.f);
#pragma unroll
    for (int j = 0; j < KC; ++j) add(wy[j], g[j]);
  } else {
    uint32_t ws[8];
    if (residual) {
      load16_bf16(residual + t * d + c, v8, ws);
      add(ws, 1.f);
    }
    if (shared) {
      load16_bf16(shared + t * d + c, v8, ws);
      add(ws, 1.f);
    }
    for (int j = 0; j < k; ++j) {
      load16_bf16(y + (long long)(inv_pos ? inv_pos[t * k + j] : t * k + j) * d + c, v8, ws);
      add(ws, gate[t * k + j]);
    }
  }
  uint32_t p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
  uint16_t* dst = out + t * d + c;
  if (v8) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(p[0]),
                 "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7])
                 : "memory");
  } else {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(p[0], p[1], p[2], p[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(p[4], p[5], p[6], p[7]);
  }
}

__global__ void pack_gate_up_kernel(int width, int d, int block, const uint16_t* __restrict__ wg,
                                    const uint16_t* __restrict__ wu, uint16_t* __restrict__ wgu,
                                    long long total_rows) {
  const long long r = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= total_rows) return;
  const long long g = r / (2 * width);
  const int rr = (int)(r % (2 * width));
  const int blk = rr / (2 * block), within = rr % (2 * block);
  const bool is_up = within >= block;
  const long long src_row = g * width + (long long)blk * block + (is_up ? within - block : within);
  const uint4* src = reinterpret_cast<const uint4*>((is_up ? wu : wg) + src_row * d);
  uint4* dst = reinterpret_cast<uint4*>(wgu + r * d);
  for (int v = threadIdx.x % 32; v < d / 8; v += 32) dst[v] = src[v];
}

}  // namespace

cudaError_t launch_count(const int32_t* idx, int T, int k, int E, int chunk_tokens,
                         int32_t* counts, cudaStream_t s) {
  const long long n = (long long)T * k;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevicePointer;
  count_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(idx, T, k, E, chunk_tokens, counts, status);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const int32_t* idx, const int32_t* counts, int T, int k, int E,
                           int chunk_tokens, int32_t* offsets, int32_t* load_out, float* bias,
                           float gamma, long long tokens_times_k, int32_t* perm_tok,
                           int32_t* inv_pos, const void* x, int x_is_f32, int d, uint16_t* xp,
                           uint16_t* xb, cudaStream_t s, int32_t* active, moe_balance_t* balance) {
  const int chunks = (T + chunk_tokens - 1) / chunk_tokens;
  const int block_tokens = chunk_tokens <= 128 ? 32 : chunk_tokens;
  const int blocks = (T + block_tokens - 1) / block_tokens;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevicePointer;
  return launch_pdl(scatter_kernel, dim3(blocks), dim3(SC_THREADS), 0, s, idx, counts, chunks, T, k,
                    E, chunk_tokens, offsets, load_out, bias, gamma, tokens_times_k, perm_tok,
                    inv_pos, x, x_is_f32, d, xp, xb, active, balance, status);
}

cudaError_t launch_gather(const void* x, int x_is_f32, const int32_t* perm_tok, long long rows,
                          int d, uint16_t* xp, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  gather_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(x, x_is_f32, perm_tok, rows, d, xp);
  return cudaGetLastError();
}

cudaError_t launch_to_bf16(const float* x, long long n, uint16_t* xb, cudaStream_t s) {
  const long long n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  to_bf16_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(x, n8, xb);
  return cudaGetLastError();
}

cudaError_t launch_bias_update(int E, long long tokens_times_k, const int32_t* load, float gamma,
                               float* bias, cudaStream_t s, moe_balance_t* balance) {
  if (E < 1 || E > 256) return cudaErrorInvalidValue;
  bias_update_kernel<<<1, 256, 0, s>>>(E, tokens_times_k, load, gamma, bias, balance);
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* y_perm, const uint16_t* shared_out,
                           const int32_t* inv_pos, const float* gate, const uint16_t* residual,
                           uint16_t* out, int T, int k, int d, cudaStream_t s) {
  const long long n = (long long)T * (d / 16);
  auto a32 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 32 == 0; };
  // d % 64 == 0, so every row starts on a 32-byte boundary when its base does.
  const int v8 = a32(y_perm) && a32(out) && (!shared_out || a32(shared_out)) &&
                 (!residual || a32(residual));
  const dim3 grid((unsigned)((n + 255) / 256));
  if (k == 1)
    return launch_pdl(combine_kernel<1>, grid, dim3(256), 0, s, y_perm, shared_out, inv_pos, gate,
                      residual, out, T, k, d, v8);
  if (k == 2)
    return launch_pdl(combine_kernel<2>, grid, dim3(256), 0, s, y_perm, shared_out, inv_pos, gate,
                      residual, out, T, k, d, v8);
  return launch_pdl(combine_kernel<0>, grid, dim3(256), 0, s, y_perm, shared_out, inv_pos, gate,
                    residual, out, T, k, d, v8);
}

cudaError_t launch_pack_gate_up(int G, int width, int d, int block, const uint16_t* wg,
                                const uint16_t* wu, uint16_t* wgu, cudaStream_t s) {
  const long long rows = (long long)G * 2 * width;
  pack_gate_up_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(width, d, block, wg, wu, wgu,
                                                                    rows);
  return cudaGetLastError();
}

}  // namespace moe
