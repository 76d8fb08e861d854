// Expert-parallel bookkeeping: the experts are split into `world` contiguous ranges,
// each rank sends the rows its routing gave to another rank's experts there, and the
// owner groups the rows it receives by its local expert before the grouped GEMM.
// Relay article, top-2 paragraph: the leftover imbalance is what expert parallelism
// meets; the aux-loss-free bias keeps the per-expert (and so per-rank) loads close to
// even.  The rows arrive source by source, each source's rows by local expert (the
// sender's permuted order); grouped, expert e's rows are the sources' runs for e in
// source order, so with consecutive token shards per rank each expert's rows come in
// global token order, as one GPU's permutation would have them.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

// One block per (source s, local expert e) run: its first received row and its first
// grouped row are prefix sums over the count table, then the run is filled.
// perm[grouped row] = received row; inv[received row] = grouped row.
__global__ void ep_regroup_kernel(int world, int el, const int32_t* __restrict__ counts,
                                  int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                  int32_t* __restrict__ offsets) {
  const int s = blockIdx.x / el, e = blockIdx.x % el;
  __shared__ long long part[3][32];
  long long src = 0, dst = 0, off_e = 0;
  // src: runs before (s, e) in source-major order; dst: rows of experts < e plus the
  // rows of expert e from sources < s.
  for (int i = threadIdx.x; i < world * el; i += blockDim.x) {
    const int si = i / el, ei = i % el;
    const long long c = counts[i];
    if (si < s || (si == s && ei < e)) src += c;
    if (ei < e) off_e += c;
    if (ei == e && si < s) dst += c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    src += __shfl_xor_sync(0xFFFFFFFFu, src, o);
    dst += __shfl_xor_sync(0xFFFFFFFFu, dst, o);
    off_e += __shfl_xor_sync(0xFFFFFFFFu, off_e, o);
  }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0) {
    part[0][warp] = src;
    part[1][warp] = dst;
    part[2][warp] = off_e;
  }
  __syncthreads();
  src = dst = off_e = 0;
  for (int w = 0; w < (int)(blockDim.x / 32); ++w) {
    src += part[0][w];
    dst += part[1][w];
    off_e += part[2][w];
  }
  dst += off_e;
  if (s == 0 && threadIdx.x == 0) offsets[e] = (int32_t)off_e;
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    long long total = 0;
    for (int i = 0; i < world * el; ++i) total += counts[i];
    offsets[el] = (int32_t)total;
  }
  const int n = counts[s * el + e];
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    perm[dst + j] = (int32_t)(src + j);
    inv[src + j] = (int32_t)(dst + j);
  }
}

}  // namespace

cudaError_t launch_ep_regroup(int world, int el, const int32_t* counts, int32_t* perm, int32_t* inv,
                              int32_t* offsets, cudaStream_t s) {
  ep_regroup_kernel<<<world * el, 256, 0, s>>>(world, el, counts, perm, inv, offsets);
  return cudaGetLastError();
}

}  // namespace moe
