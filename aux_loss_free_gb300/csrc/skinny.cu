// Shared-expert projections for a few tokens (T <= 64): "skinny" GEMMs on tcgen05.
//
// Relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B de
// NanoColibri por $200"), opening section, architecture paragraph: one shared expert
// of width 2048 is always resident and runs on every token; section "Entrenamiento por
// relevos", top-2 paragraph: the serving engine runs one routed expert per token.  At
// serving batch sizes the step is bound by reading the weights, so the shared expert's
// 12.6 MB must stream across the whole GPU.
//
// D[w][t] = W[w][K] . X[t][K]^T with the weight rows in the MMA's M (128 per CTA) and
// the tokens in N (T rounded up to 16): tcgen05.mma.cta_group::1.kind::f16, both
// operands K-major with the 128-byte swizzle, the accumulator in TMEM.  K is split over
// an 8-CTA cluster; each CTA loads its whole K slice with TMA in one go (weights before
// the programmatic-dependency wait, since no earlier kernel writes them), multiplies,
// moves its partial sums to shared memory, and after a cluster barrier CTA r reduces
// rows [16r, 16r + 16) of the 128 over the cluster's shared memory and finishes them:
//   mode 0 (gate/up): weights [2F][K] with gate and up rows interleaved in blocks of
//           128, one CTA covers one block pair (two accumulators) and writes
//           h[t][j] = silu(g) * u in bf16;
//   mode 1 (down):   weights [d][F], writes out[t][n] = acc (+ residual[t][n]
//           + sum_j gate[t][j] * y_perm[inv_pos[t][j]][n] when combining; without
//           inv_pos the routed rows are indexed by pair, t * k + j), bf16.
// Every wait is bounded; on a timeout the CTA records it in the status word and still
// reaches both cluster barriers and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int SK_SPLIT = 8;       // CTAs per cluster = K split
constexpr int SK_THREADS = 128;   // 4 warps = the 128 TMEM lanes
constexpr int SK_ROWS = 128;      // weight rows per accumulator
constexpr int SK_ATOM_K = 64;     // K per 128-byte swizzle atom (bf16)
constexpr int SK_W_ATOM = SK_ROWS * SK_ATOM_K * 2;  // 16 KB
constexpr int SK_MAX_ATOMS = 8;   // K slice <= 512
constexpr int SK_RED_ROWS = SK_ROWS / SK_SPLIT;      // rows each CTA finishes

struct SkinnyParams {
  CUtensorMap w;    // [rows][K], box 128 x 64
  CUtensorMap x;    // [T][K], box N x 64
  int mode;         // 0 gate/up SwiGLU, 1 down (+ combine)
  int T, N, atoms;  // N = T rounded up to 16; atoms = K slice / 64
  uint16_t* out;
  int ldo;
  const uint16_t* residual;  // mode 1, nullable
  const uint16_t* y_perm;    // mode 1, nullable: routed rows to add
  const int32_t* inv_pos;
  const float* gate;
  int k;
  int* status;
};

__device__ __forceinline__ uint32_t sk_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void sk_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ float sk_ld_cluster(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ float sk_bf16(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__global__ void __cluster_dims__(SK_SPLIT, 1, 1) __launch_bounds__(SK_THREADS, 1)
    skinny_gemm_kernel(const __grid_constant__ SkinnyParams p) {
  extern __shared__ uint8_t sk_smem_raw[];
  __shared__ __align__(8) uint64_t full_bar;
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_holder;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = sk_cluster_rank();
  const int unit = blockIdx.x / SK_SPLIT;
  const int nmat = p.mode == 0 ? 2 : 1;
  const int N = p.N;
  const uint32_t base = (smem_u32(sk_smem_raw) + 1023u) & ~1023u;
  uint8_t* base_ptr = sk_smem_raw + (base - smem_u32(sk_smem_raw));
  const uint32_t w_smem = base;                                        // [nmat][atoms][16 KB]
  const uint32_t x_smem = base + (uint32_t)(nmat * p.atoms * SK_W_ATOM);  // [atoms][N x 128 B]
  float* part = reinterpret_cast<float*>(base_ptr);                    // [nmat][N][128] afterwards
  const uint32_t ncols = nmat * N <= 32 ? 32u : (nmat * N <= 64 ? 64u : 128u);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&full_bar), 1);
    mbar_init(smem_u32(&done_bar), 1);
    fence_mbar_init();
    tma_prefetch_desc(&p.w);
    tma_prefetch_desc(&p.x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const int k0 = (int)rank * p.atoms * SK_ATOM_K;

  bool ok = true;
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)(nmat * p.atoms * SK_W_ATOM + p.atoms * N * 128);
    mbar_arrive_expect_tx(smem_u32(&full_bar), bytes);
    // The weights are not written by any earlier kernel: request them before waiting.
    for (int m = 0; m < nmat; ++m) {
      const int row0 = p.mode == 0 ? unit * 2 * SK_ROWS + m * SK_ROWS : unit * SK_ROWS;
      for (int a = 0; a < p.atoms; ++a)
        tma_load_2d(w_smem + (uint32_t)((m * p.atoms + a) * SK_W_ATOM), &p.w, smem_u32(&full_bar),
                    k0 + a * SK_ATOM_K, row0);
    }
  }
  pdl_wait();  // the tokens (and the combine's inputs) come from earlier kernels
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int a = 0; a < p.atoms; ++a)
      tma_load_2d(x_smem + (uint32_t)(a * N * 128), &p.x, smem_u32(&full_bar), k0 + a * SK_ATOM_K, 0);
    ok = mbar_wait(smem_u32(&full_bar), 0, p.status);
    if (!ok) mbar_wait(smem_u32(&full_bar), 0, p.status);  // let late copies land first
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(SK_ROWS, N);
      for (int a = 0; a < p.atoms; ++a) {
        const uint64_t xd = sw128_kmajor_desc(x_smem + (uint32_t)(a * N * 128));
        for (int m = 0; m < nmat; ++m) {
          const uint64_t wd = sw128_kmajor_desc(w_smem + (uint32_t)((m * p.atoms + a) * SK_W_ATOM));
#pragma unroll
          for (int kk = 0; kk < SK_ATOM_K / 16; ++kk)
            tc_mma_bf16(tmem + (uint32_t)(m * N), wd + 2 * kk, xd + 2 * kk, idesc, (a | kk) != 0);
        }
      }
    }
    tc_commit(smem_u32(&done_bar));  // also when nothing was issued: arrives at once
  }
  // Partial sums: TMEM lane = weight row, column = token.  They overwrite the operand
  // tiles, which the finished MMAs no longer read.
  const bool got = mbar_wait(smem_u32(&done_bar), 0, p.status);
  tc_fence_after();
  const int row = warp * 32 + lane;
  for (int m = 0; m < nmat; ++m)
    for (int c = 0; c < N; c += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(m * N + c), v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        part[((size_t)m * N + c + i) * SK_ROWS + row] = got ? __uint_as_float(v[i]) : 0.f;
    }
  tc_fence_before();
  sk_cluster_sync();

  // Reduce rows [16r, 16r + 16) over the cluster and finish them.
  const uint32_t part_addr = smem_u32(part);
  const int r0 = (int)rank * SK_RED_ROWS;
  for (int i = threadIdx.x; i < SK_RED_ROWS * p.T; i += SK_THREADS) {
    const int rr = r0 + i % SK_RED_ROWS, t = i / SK_RED_ROWS;
    float acc[2] = {0.f, 0.f};
    for (int m = 0; m < nmat; ++m)
      for (uint32_t q = 0; q < SK_SPLIT; ++q)
        acc[m] += sk_ld_cluster(part_addr + 4u * (uint32_t)(((size_t)m * N + t) * SK_ROWS + rr), q);
    if (p.mode == 0) {
      const float g = acc[0], u = acc[1];
      const float h = __fdividef(g, 1.0f + __expf(-g)) * u;
      p.out[(size_t)t * p.ldo + unit * SK_ROWS + rr] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
    } else {
      const int col = unit * SK_ROWS + rr;
      float o = acc[0];
      if (p.residual) o += sk_bf16(p.residual[(size_t)t * p.ldo + col]);
      if (p.y_perm)
        for (int j = 0; j < p.k; ++j)
          o = fmaf(p.gate[(size_t)t * p.k + j],
                   sk_bf16(p.y_perm[(p.inv_pos ? (size_t)p.inv_pos[(size_t)t * p.k + j]
                                               : (size_t)t * p.k + j) * p.ldo + col]), o);
      p.out[(size_t)t * p.ldo + col] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
    }
  }
  sk_cluster_sync();  // no CTA leaves while another may still read its partial sums
  if (warp == 1) tmem_dealloc(tmem, ncols);
  (void)ok;
}

}  // namespace

bool skinny_supported(int mode, int T, int rows, int K, int gate_block) {
  if (T < 1 || T > kSkinnyMaxT) return false;
  if (K % (SK_ATOM_K * SK_SPLIT) != 0 || K / (SK_ATOM_K * SK_SPLIT) > SK_MAX_ATOMS) return false;
  if (mode == 0) return gate_block == SK_ROWS && rows % (2 * SK_ROWS) == 0;
  return rows % SK_ROWS == 0;
}

cudaError_t launch_skinny(int mode, const uint16_t* w, int rows, int K, const uint16_t* x, int T,
                          uint16_t* out, int ldo, const CombineInputs* comb, cudaStream_t s) {
  SkinnyParams p;
  std::memset(&p, 0, sizeof(p));
  p.mode = mode;
  p.T = T;
  p.N = (T + 15) / 16 * 16;
  p.atoms = K / (SK_ATOM_K * SK_SPLIT);
  p.out = out;
  p.ldo = ldo;
  if (comb) {
    p.residual = comb->residual;
    p.y_perm = comb->y_perm;
    p.inv_pos = comb->inv_pos;
    p.gate = comb->gate;
    p.k = comb->k;
  }
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;
  if (!make_tma_map_bf16(&p.w, w, (uint64_t)K, (uint64_t)rows, SK_ROWS) ||
      !make_tma_map_bf16(&p.x, x, (uint64_t)K, (uint64_t)T, (uint32_t)p.N))
    return cudaErrorInvalidValue;
  const int nmat = mode == 0 ? 2 : 1;
  const size_t operands = (size_t)nmat * p.atoms * SK_W_ATOM + (size_t)p.atoms * p.N * 128;
  const size_t partials = (size_t)nmat * p.N * SK_ROWS * 4;
  const size_t dyn = (operands > partials ? operands : partials) + 1024;
  cudaError_t e = cudaFuncSetAttribute(skinny_gemm_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  const int units = mode == 0 ? rows / (2 * SK_ROWS) : rows / SK_ROWS;
  return launch_pdl(skinny_gemm_kernel, dim3(units * SK_SPLIT), dim3(SK_THREADS), dyn, s, p);
}

}  // namespace moe
