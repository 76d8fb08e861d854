// Grouped expert GEMM on tcgen05 tensor cores (sm_103a).
//
// One persistent launch runs up to two operand sets: the routed experts (E groups,
// row ranges read from the device offsets of the counting sort, so there is no
// host round trip) and the shared expert (one group over all tokens).  Relay
// article, opening section, architecture paragraph: 64 routed experts plus one
// always-resident shared expert; SwiGLU is this library's reading of the expert FFN.
//
// CTA layout (192 threads, one CTA per SM):
//   warp 0      TMA producer: A tile 128 x 64 and B tile BN x 64 (bf16, 128-byte
//               swizzle) per stage into a 4-stage shared-memory ring;
//   warp 1      owns the TMEM allocation; one thread issues tcgen05.mma
//               (M = 128, N = BN, K = 16) into one of two 128 x 256 fp32
//               accumulators, committing stage releases and accumulator-ready
//               barriers;
//   warps 2..5  epilogue: tcgen05.ld of their 32 TMEM lanes (rows), then
//               SWIGLU  h = silu(gate) * up -> bf16   (gate / up rows interleaved
//                       in the weights so one tile holds matching columns),
//               STORE   y -> bf16,
//               COMBINE out = acc + residual + sum_j gate_j * y_perm[inv_pos_j]
//                       (the shared expert's down projection adds the routed
//                       outputs of the same token: the layer's combine step).
// Every barrier wait is bounded (ptx.cuh); on a timeout the CTA records it in the
// status word, drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN_MAX = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN_MAX * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN_MAX;
constexpr int DYN_SMEM = STAGES * STAGE_BYTES + 1024;
constexpr unsigned FULL = 0xFFFFFFFFu;

struct OperandSet {
  CUtensorMap a;
  CUtensorMap b;
  void* out;
  int ldo, n_total, k_total, bn, mode, enabled, rows, pad;
};

struct Params {
  OperandSet shared;
  OperandSet routed;
  const int32_t* offsets;
  const uint16_t* y_perm;
  const int32_t* inv_pos;
  const float* gate;
  const uint16_t* residual;
  int* status;
  int E, k;
};

struct Tile {
  int set;    // 0 shared, 1 routed
  int row0;   // first A row (and output row)
  int rows;   // valid rows in this tile
  int brow;   // first B row
  int n0;     // first output column of the accumulator tile
};

__device__ __forceinline__ Tile decode_tile(const Params& p, int tile, int shared_tiles,
                                            const int* s_off, const int* s_cum) {
  Tile t;
  if (tile < shared_tiles) {
    const int nt = p.shared.n_total / p.shared.bn;
    const int m = tile / nt, n = tile % nt;
    t.set = 0;
    t.row0 = m * BM;
    t.rows = min(BM, p.shared.rows - t.row0);
    t.n0 = n * p.shared.bn;
    t.brow = t.n0;
  } else {
    const int r = tile - shared_tiles;
    int lo = 0, hi = p.E;  // largest g with s_cum[g] <= r (that group is non-empty)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_cum[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    const int nt = p.routed.n_total / p.routed.bn;
    const int local = r - s_cum[g];
    const int m = local / nt, n = local % nt;
    t.set = 1;
    t.row0 = s_off[g] + m * BM;
    t.rows = min(BM, s_off[g + 1] - t.row0);
    t.n0 = n * p.routed.bn;
    t.brow = g * p.routed.n_total + t.n0;
  }
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float a) { return a / (1.0f + __expf(-a)); }

__device__ __forceinline__ void add_bf16_row32(float (&o)[32], const uint16_t* src, float w) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 u = s[v];
    const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[v * 8 + 2 * i] = fmaf(w, __uint_as_float(ws[i] << 16), o[v * 8 + 2 * i]);
      o[v * 8 + 2 * i + 1] = fmaf(w, __uint_as_float(ws[i] & 0xFFFF0000u), o[v * 8 + 2 * i + 1]);
    }
  }
}

__device__ __forceinline__ void store_bf16_row32(uint16_t* dst, const float (&o)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v)
    d[v] = make_uint4(pack_bf16x2(o[8 * v + 0], o[8 * v + 1]), pack_bf16x2(o[8 * v + 2], o[8 * v + 3]),
                      pack_bf16x2(o[8 * v + 4], o[8 * v + 5]), pack_bf16x2(o[8 * v + 6], o[8 * v + 7]));
}

__global__ void __launch_bounds__(NUM_THREADS, 1) grouped_gemm_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_cum[kMaxE + 1];
  __shared__ int s_total;

  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int shared_tiles =
      p.shared.enabled ? ((p.shared.rows + BM - 1) / BM) * (p.shared.n_total / p.shared.bn) : 0;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull_bar[a]), 1);
      mbar_init(smem_u32(&tempty_bar[a]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_mbar_init();
    if (p.shared.enabled) {
      tma_prefetch_desc(&p.shared.a);
      tma_prefetch_desc(&p.shared.b);
    }
    if (p.routed.enabled) {
      tma_prefetch_desc(&p.routed.a);
      tma_prefetch_desc(&p.routed.b);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    // Tile table of the routed groups: s_cum[g] = tiles of groups < g.
    int carry = 0;
    if (p.routed.enabled) {
      const int nt = p.routed.n_total / p.routed.bn;
      for (int b = 0; b < p.E; b += 32) {
        const int g = b + lane;
        int v = 0;
        if (g < p.E) {
          const int o0 = p.offsets[g], o1 = p.offsets[g + 1];
          s_off[g] = o0;
          if (g == p.E - 1) s_off[p.E] = o1;
          v = ((o1 - o0 + BM - 1) / BM) * nt;
        }
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += n;
        }
        if (g < p.E) s_cum[g] = carry + incl - v;
        carry += __shfl_sync(FULL, incl, 31);
      }
      if (lane == 0) s_cum[p.E] = carry;
    }
    if (lane == 0) s_total = shared_tiles + carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;
  const int total = s_total;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode_tile(p, tile, shared_tiles, s_off, s_cum);
        const OperandSet& S = t.set ? p.routed : p.shared;
        const int nkb = (S.k_total + BK - 1) / BK;
        const uint32_t bytes = A_BYTES + S.bn * BK * 2;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = ring + stage * STAGE_BYTES;
          const uint32_t fb = smem_u32(&full_bar[stage]);
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_2d(sa, &S.a, fb, kb * BK, t.row0);
          tma_load_2d(sa + A_BYTES, &S.b, fb, kb * BK, t.brow);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy this CTA started must land before the CTA may exit.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(smem_u32(&full_bar[s]), (last_par >> s) & 1u, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode_tile(p, tile, shared_tiles, s_off, s_cum);
        const OperandSet& S = t.set ? p.routed : p.shared;
        const int nkb = (S.k_total + BK - 1) / BK;
        const uint32_t idesc = idesc_bf16_f32(BM, S.bn);
        if (!mbar_wait(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN_MAX;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&full_bar[stage]), phase, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = ring + stage * STAGE_BYTES;
          const uint64_t adesc = sw128_kmajor_desc(sa);
          const uint64_t bdesc = sw128_kmajor_desc(sa + A_BYTES);
          const int kleft = S.k_total - kb * BK;
          const int nkk = kleft >= BK ? BK / 16 : (kleft + 15) / 16;
          for (int kk = 0; kk < nkk; ++kk)
            tc_mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
          tc_commit(smem_u32(&empty_bar[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull_bar[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA this thread issued must finish before TMEM is released.
      tc_commit(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, p.status);
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lanes [32q, 32q + 32) are this warp's rows
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode_tile(p, tile, shared_tiles, s_off, s_cum);
      const OperandSet& S = t.set ? p.routed : p.shared;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, p.status) ? 1 : 0;
      ok = __shfl_sync(FULL, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int r = q * 32 + lane;
      const bool valid = r < t.rows;
      const long long orow = (long long)t.row0 + r;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN_MAX;
      uint16_t* out = static_cast<uint16_t*>(S.out);
      if (S.mode == EPI_SWIGLU) {
        const int half = S.bn / 2;
        for (int c = 0; c < half; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c, g);
          tmem_ld32(tbase + half + c, u);
          tmem_wait_ld();
          float h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) h[i] = silu(__uint_as_float(g[i])) * __uint_as_float(u[i]);
          if (valid) store_bf16_row32(out + orow * S.ldo + t.n0 / 2 + c, h);
        }
      } else if (S.mode == EPI_STORE) {
        for (int c = 0; c < S.bn; c += 32) {
          uint32_t v[32];
          tmem_ld32(tbase + c, v);
          tmem_wait_ld();
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]);
          if (valid) store_bf16_row32(out + orow * S.ldo + t.n0 + c, o);
        }
      } else {
        float gj[kMaxK];
        long long pj[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
          gj[j] = 0.f;
          pj[j] = 0;
          if (valid && j < p.k) {
            gj[j] = p.gate[orow * p.k + j];
            pj[j] = p.inv_pos[orow * p.k + j];
          }
        }
        for (int c = 0; c < S.bn; c += 32) {
          uint32_t v[32];
          tmem_ld32(tbase + c, v);
          tmem_wait_ld();
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]);
          if (valid) {
            const long long col = t.n0 + c;
            if (p.residual) add_bf16_row32(o, p.residual + orow * S.ldo + col, 1.f);
#pragma unroll
            for (int j = 0; j < kMaxK; ++j)
              if (j < p.k) add_bf16_row32(o, p.y_perm + pj[j] * S.ldo + col, gj[j]);
            store_bf16_row32(out + orow * S.ldo + col, o);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// bf16 matrix [outer][inner] row-major, box [box_outer][64] with the 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int gate_up_block(int width) { return width % 128 == 0 ? 128 : (width % 64 == 0 ? 64 : 32); }

int choose_bn(int mode, int N) {
  if (mode == EPI_SWIGLU) return 2 * gate_up_block(N / 2);
  return N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : 64);
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

bool fill_set(OperandSet& t, const GemmOperandSet& o) {
  std::memset(&t, 0, sizeof(t));
  if (!o.a) return true;
  t.enabled = 1;
  t.bn = choose_bn(o.mode, o.N);
  t.n_total = o.N;
  t.k_total = o.K;
  t.ldo = o.ldo;
  t.mode = o.mode;
  t.rows = o.rows;
  t.out = o.out;
  if (o.N % t.bn != 0) return false;
  if (!make_map(&t.a, o.a, o.K, o.a_rows, BM)) return false;
  if (!make_map(&t.b, o.b, o.K, (uint64_t)o.groups * o.N, t.bn)) return false;
  return true;
}

}  // namespace

cudaError_t launch_grouped_gemm(const GemmOperandSet& routed, const int32_t* offsets, int E,
                                const GemmOperandSet& shared, const CombineInputs& comb,
                                long long max_routed_rows, cudaStream_t s, int* bad_arg) {
  Params p;
  std::memset(&p, 0, sizeof(p));
  *bad_arg = 0;
  if (!fill_set(p.shared, shared) || !fill_set(p.routed, routed)) {
    *bad_arg = 1;
    return cudaErrorInvalidValue;
  }
  if (!p.shared.enabled && !p.routed.enabled) return cudaSuccess;
  p.offsets = offsets;
  p.E = E;
  p.y_perm = comb.y_perm;
  p.inv_pos = comb.inv_pos;
  p.gate = comb.gate;
  p.residual = comb.residual;
  p.k = comb.k;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;

  long long tiles = 0;
  if (p.shared.enabled)
    tiles += (long long)((p.shared.rows + BM - 1) / BM) * (p.shared.n_total / p.shared.bn);
  if (p.routed.enabled)
    tiles += ((max_routed_rows + BM - 1) / BM + E) * (long long)(p.routed.n_total / p.routed.bn);
  const int grid = (int)std::min<long long>(num_sms(), std::max<long long>(tiles, 1));
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, DYN_SMEM);
  if (e != cudaSuccess) return e;
  grouped_gemm_kernel<<<grid, NUM_THREADS, DYN_SMEM, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
