// Causal grouped-query attention with per-head QK-norm on tcgen05 tensor cores (sm_103a).
//
// Relay article ("Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B de
// NanoColibri por $200"), opening section, architecture paragraph: grouped-query
// attention with four query heads per key/value head and a per-head QK-norm.  This
// library's readings: head width 128; the norm is an RMS normalisation of each head's
// 128 values without a learned scale; scores q.k / sqrt(128), causal within each
// sequence, no positional encoding.
//
// qk_norm_kernel normalises the query and key heads of the projected [T][C] rows in
// place (C = (n_head + 2 n_kv_head) * 128: query heads, key heads, value heads), one
// warp per row.
// gqa_attention_kernel computes one 128-query tile of one head per CTA:
//   - warp 0 (one thread): TMA copies of the query tile (once) and of the key tiles of
//     the head's group into a 2-stage ring, each stage freed as soon as its S MMA is
//     done, so the key tile two ahead streams in during the softmax; warp 6 (one
//     thread): the value tiles into their own 2-stage ring, freed by the P V MMA;
//   - warp 1 (one thread): tcgen05.mma, S_j = Q K_j^T into one of two TMEM score
//     buffers, and O += P_j V_j into the TMEM output (V read MN-major through the
//     instruction descriptor, no transposed copy) with P_j read from one of two TMEM
//     buffers as the MMA's A operand; S_{j+1} is issued before P_j V_j, and the softmax
//     of tile j + 1 writes the other P buffer while P_j V_j runs, so the tensor core and
//     the softmax warps overlap;
//   - warps 2-5 (one query row per thread, its TMEM lane): the online softmax in the
//     log2 domain on the row's 128 scores held in registers (causal mask on the
//     diagonal tile only), writing P_j as bf16 pairs into the row's TMEM lane, and
//     rescaling the O row in TMEM only when the row's
//     maximum grew by more than 8 (2^8), which keeps every exponential below 256; at
//     the end O / l rounded to bf16.
// Every barrier wait is bounded; on a timeout the status word is set and the CTA exits.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int HD = kAttnHeadDim;              // head width
constexpr int BQ = 128;                       // query rows per CTA (TMEM lanes)
constexpr int BKV = 128;                      // keys per tile
constexpr int AT = 64;                        // columns per 128-byte swizzle atom (bf16)
constexpr int ATOM_BYTES = 128 * AT * 2;      // 16 KB: 128 rows x 64
constexpr int TILE_BYTES = 2 * ATOM_BYTES;    // 32 KB: 128 rows x 128
constexpr int KV_STAGES = 2;
constexpr int Q_OFF = 0;
constexpr int K_OFF = TILE_BYTES;                       // key stage s at K_OFF + s TILE
constexpr int V_OFF = K_OFF + KV_STAGES * TILE_BYTES;   // value stage s at V_OFF + s TILE
constexpr int ATT_SMEM = V_OFF + KV_STAGES * TILE_BYTES + 1024;
constexpr int P_BUFS = 2;
constexpr int ATT_THREADS = 224;
constexpr uint32_t S_COL = 0;                 // score buffers: columns [0, 128) and [128, 256)
constexpr uint32_t O_COL = 256;               // output accumulator: columns [256, 384)
constexpr uint32_t P_COL = 384;               // P buffers, bf16 pairs: columns [384, 448) and [448, 512)
constexpr uint32_t ATT_TMEM_COLS = 512;
constexpr unsigned FULL = 0xFFFFFFFFu;

struct AttnParams {
  CUtensorMap qkv;   // [T][C] bf16 viewed as (64, T, C / 64), box (64, 128, 2)
  uint16_t* out;     // [T][n_head * HD] bf16
  int* status;
  int batch, seq, n_head, n_kv_head, qtiles;
  float scale_log2;  // log2(e) / sqrt(HD)
};

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem], one 128 x N x 16 step with A read from tensor memory:
// row m of A in lane m, two bf16 values per 32-bit column (the even k in the low half).
__device__ __forceinline__ void tc_mma_bf16_a_tmem(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2^x by the hardware's approximate base-2 exponential (relative error near 2^-22;
// 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One warp per token row: every query and key head of the row (u / sqrt(mean(u^2) +
// eps) over the head's 128 values, rounded to bf16 in place); all of the row's loads are
// issued before the first reduction.
constexpr int QKN_MAX_HEADS = 16;
__global__ void qk_norm_kernel(uint16_t* __restrict__ qkv, long long rows, int C, int heads, float eps) {
  pdl_wait();
  pdl_trigger();
  const long long t = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (t >= rows) return;
  uint2* row = reinterpret_cast<uint2*>(qkv + t * C) + lane;  // 4 values per lane and head
  for (int h0 = 0; h0 < heads; h0 += QKN_MAX_HEADS) {
    const int nh = min(QKN_MAX_HEADS, heads - h0);
    uint2 v[QKN_MAX_HEADS];
#pragma unroll
    for (int i = 0; i < QKN_MAX_HEADS; ++i)
      if (i < nh) v[i] = row[(h0 + i) * (HD / 4)];
#pragma unroll
    for (int i = 0; i < QKN_MAX_HEADS; ++i) {
      if (i < nh) {
        const float a = __uint_as_float(v[i].x << 16), b = __uint_as_float(v[i].x & 0xFFFF0000u);
        const float c = __uint_as_float(v[i].y << 16), d = __uint_as_float(v[i].y & 0xFFFF0000u);
        float ss = a * a + b * b + c * c + d * d;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
        const float f = rsqrtf(ss * (1.0f / HD) + eps);
        row[(h0 + i) * (HD / 4)] = make_uint2(pack_bf16x2(a * f, b * f), pack_bf16x2(c * f, d * f));
      }
    }
  }
}

__global__ void __launch_bounds__(ATT_THREADS, 1) gqa_attention_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full;
  __shared__ __align__(8) uint64_t k_full[KV_STAGES];
  __shared__ __align__(8) uint64_t k_empty[KV_STAGES];
  __shared__ __align__(8) uint64_t v_full[KV_STAGES];
  __shared__ __align__(8) uint64_t v_empty[KV_STAGES];
  __shared__ __align__(8) uint64_t s_full[2];
  __shared__ __align__(8) uint64_t s_free[2];
  __shared__ __align__(8) uint64_t p_full[P_BUFS];
  __shared__ __align__(8) uint64_t pv_done[P_BUFS];
  __shared__ uint32_t tmem_holder;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // The longest query tiles (most key tiles under the causal mask) go first.
  const int per_tile = p.n_head * p.batch;
  const int qi = p.qtiles - 1 - (int)blockIdx.x / per_tile;
  const int rem = (int)blockIdx.x % per_tile;
  const int h = rem % p.n_head, b = rem / p.n_head;
  const int g = h / (p.n_head / p.n_kv_head);
  const int row0 = b * p.seq + qi * BQ;  // first token row of the query tile
  const int ntiles = qi + 1;              // key tiles 0..qi
  const int q_atom = h * (HD / AT), k_atom = (p.n_head + g) * (HD / AT),
            v_atom = (p.n_head + p.n_kv_head + g) * (HD / AT);

  if (warp == 0 && lane == 0) {
    mbar_init(smem_u32(&q_full), 1);
    for (int s = 0; s < KV_STAGES; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_free[s]), 4);
    }
    for (int s = 0; s < P_BUFS; ++s) {
      mbar_init(smem_u32(&p_full[s]), 4);
      mbar_init(smem_u32(&pv_done[s]), 1);
    }
    fence_mbar_init();
    tma_prefetch_desc(&p.qkv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), ATT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  pdl_wait();  // the projected, normalised rows come from earlier kernels
  pdl_trigger();

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producers: keys (warp 0,
      // which also copies the query tile) and values (warp 6)
      const bool keys = warp == 0;
      uint64_t* const full = keys ? k_full : v_full;
      uint64_t* const empty = keys ? k_empty : v_empty;
      const uint32_t ring = base + (keys ? K_OFF : V_OFF);
      const int atom = keys ? k_atom : v_atom;
      if (keys) {
        mbar_arrive_expect_tx(smem_u32(&q_full), TILE_BYTES);
        tma_load_3d(base + Q_OFF, &p.qkv, smem_u32(&q_full), 0, row0, q_atom);
      }
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % KV_STAGES;
        const uint32_t ph = (uint32_t)(j / KV_STAGES) & 1u;
        if (!mbar_wait_spin(smem_u32(&empty[st]), ph ^ 1u, p.status)) break;
        const uint32_t fb = smem_u32(&full[st]);
        mbar_arrive_expect_tx(fb, TILE_BYTES);
        tma_load_3d(ring + st * TILE_BYTES, &p.qkv, fb, 0, b * p.seq + j * BKV, atom);
        issued = j + 1;
      }
      // No copy may still be landing when the CTA exits.
      if (keys) mbar_wait_spin(smem_u32(&q_full), 0, p.status);
      for (int j = issued > KV_STAGES ? issued - KV_STAGES : 0; j < issued; ++j)
        mbar_wait_spin(smem_u32(&full[j % KV_STAGES]), (uint32_t)(j / KV_STAGES) & 1u, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t id_s = idesc_bf16_f32(BQ, BKV, 0, 0);
      constexpr uint32_t id_pv = idesc_bf16_f32(BQ, HD, 0, 1);
      bool ok = mbar_wait_spin(smem_u32(&q_full), 0, p.status);
      tc_fence_after();
      const uint64_t qdesc = sw128_kmajor_desc(base + Q_OFF);
      for (int j = 0; j <= ntiles && ok; ++j) {
        if (j < ntiles) {
          const int st = j % KV_STAGES;
          const int sb = j & 1;
          if (!mbar_wait_spin(smem_u32(&k_full[st]), (uint32_t)(j / KV_STAGES) & 1u, p.status) ||
              !mbar_wait_spin(smem_u32(&s_free[sb]), ((uint32_t)(j >> 1) & 1u) ^ 1u, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kdesc = sw128_kmajor_desc(base + K_OFF + st * TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)  // atom kk / 4, 32 bytes per K step inside it
            tc_mma_bf16(tmem + S_COL + sb * BKV, qdesc + (kk >> 2) * (ATOM_BYTES >> 4) + 2 * (kk & 3),
                        kdesc + (kk >> 2) * (ATOM_BYTES >> 4) + 2 * (kk & 3), id_s, kk != 0);
          tc_commit(smem_u32(&k_empty[st]));
          tc_commit(smem_u32(&s_full[sb]));
        }
        if (j >= 1) {
          const int jp = j - 1, st = jp % KV_STAGES, pb = jp & 1;
          if (!mbar_wait_spin(smem_u32(&p_full[pb]), (uint32_t)(jp >> 1) & 1u, p.status) ||
              !mbar_wait_spin(smem_u32(&v_full[st]), (uint32_t)(jp / KV_STAGES) & 1u, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // V [keys][HD] is the MN-major B of O += P V: 64-column atoms 16 KB apart, a
          // 16-key step two 1024-byte atoms further.
          const uint64_t vdesc = sw128_mnmajor_desc(base + V_OFF + st * TILE_BYTES, ATOM_BYTES);
          const uint32_t pcol = tmem + P_COL + pb * (BKV / 2);  // 16 keys = 8 columns per step
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            tc_mma_bf16_a_tmem(tmem + O_COL, pcol + kk * 8, vdesc + kk * 128u, id_pv, (jp | kk) != 0);
          tc_commit(smem_u32(&v_empty[st]));
          tc_commit(smem_u32(&pv_done[pb]));
        }
      }
    }
  } else if (warp <= 5) {
    // -------------------------------------------------- softmax warps 2..5
    const int q4 = warp & 3;             // TMEM lanes [32 q4, 32 q4 + 32)
    const int r = q4 * 32 + lane;        // query row of the tile
    const int qpos = qi * BQ + r;        // position in the sequence
    const bool valid = qpos < p.seq;
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1;
      int w = 1;
      if (lane == 0) w = mbar_wait(smem_u32(&s_full[sb]), (uint32_t)(j >> 1) & 1u, p.status) ? 1 : 0;
      if (!__shfl_sync(FULL, w, 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t scol = tl + S_COL + sb * BKV;
      const int k0 = j * BKV;
      // The row's 128 scores in registers (one read of the buffer), scaled to the log2
      // domain.  Only the diagonal tile (j == qi) has keys later than some of its
      // queries or past the sequence's end: mask there alone.
      uint32_t v[BKV];
      tmem_ld32(scol, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[64]));
      tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[96]));
      tmem_wait_ld();
      // The scores are in registers: the buffer can take S_{j+2}.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_free[sb]));
      if (j == qi) {
#pragma unroll
        for (int i = 0; i < BKV; ++i) {
          const int kp = k0 + i;
          if (kp > qpos || kp >= p.seq) v[i] = __float_as_uint(-INFINITY);
        }
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(v[i]);
#pragma unroll
      for (int i = 8; i < BKV; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(v[i]));
      float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      tmax *= p.scale_log2;  // the scale is positive: the maximum commutes with it
      float factor = 1.0f;
      bool grow = false;
      if (j == 0) {
        m = tmax;
      } else if (tmax > m + 8.0f) {
        factor = ex2(m - tmax);
        m = tmax;
        grow = true;
      }
      const bool any_grow = __any_sync(FULL, grow);
      // Before P_j is written, the product that last read its buffer (P_{j-2} V_{j-2})
      // must be done; before O is rescaled, every earlier product (P_{j-1} V_{j-1}).
      // Every phase of each buffer's barrier is awaited in order, so no parity wait can
      // be taken for an older phase.
      if (j >= 2) {
        if (lane == 0) w = mbar_wait(smem_u32(&pv_done[j & 1]), (uint32_t)((j - 2) >> 1) & 1u, p.status) ? 1 : 0;
        if (!__shfl_sync(FULL, w, 0)) {
          ok = false;
          break;
        }
      }
      if (any_grow && j >= 1) {
        if (lane == 0)
          w = mbar_wait(smem_u32(&pv_done[(j - 1) & 1]), (uint32_t)((j - 1) >> 1) & 1u, p.status) ? 1 : 0;
        if (!__shfl_sync(FULL, w, 0)) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
      if (any_grow) {
        // Rescale the O row (lanes whose maximum did not grow use factor 1).
        l *= factor;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + O_COL + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
          tmem_st32(tl + O_COL + 32 * c, o);
        }
        tmem_wait_st();
      }
      // Exponentials (one FFMA and one ex2 each; masked keys give 2^-inf = 0), the row
      // sum and P (bf16 pairs, keys 2c and 2c + 1 in column c of the row's P buffer).
      const float2 nm2 = make_float2(-m, -m), sc2 = make_float2(p.scale_log2, p.scale_log2);
      const uint32_t pcol = tl + P_COL + (j & 1) * (BKV / 2);
      float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < BKV / 64; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          // Two scores per packed fp32x2 FMA; the exponentials one by one.
          const float2 a = __ffma2_rn(make_float2(__uint_as_float(v[64 * c + i]), __uint_as_float(v[64 * c + i + 1])),
                                      sc2, nm2);
          const float2 e = make_float2(ex2(a.x), ex2(a.y));
          ls[(i >> 1) & 1] = __fadd2_rn(ls[(i >> 1) & 1], e);
          pk[i / 2] = pack_bf16x2(e.x, e.y);
        }
        tmem_st32(pcol + 32 * c, pk);
      }
      l += (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
      tmem_wait_st();  // P is in TMEM before the MMA may read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[j & 1]));
    }
    if (ok) {
      int w = 1;
      const int last = ntiles - 1;
      if (lane == 0) w = mbar_wait(smem_u32(&pv_done[last & 1]), (uint32_t)(last >> 1) & 1u, p.status) ? 1 : 0;
      if (__shfl_sync(FULL, w, 0)) {
        tc_fence_after();
        const float inv = 1.0f / l;
        uint16_t* dst = p.out + (long long)(b * p.seq + qpos) * (p.n_head * HD) + h * HD;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tl + O_COL + 32 * c, v);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
            for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ATT_TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

cudaError_t launch_qk_norm(uint16_t* qkv, long long rows, int C, int heads, float eps, cudaStream_t s) {
  if (rows == 0 || heads == 0) return cudaSuccess;
  return launch_pdl(qk_norm_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, s, qkv, rows, C, heads, eps);
}

cudaError_t launch_attention(const uint16_t* qkv, int batch, int seq, int n_head, int n_kv_head, uint16_t* out,
                             cudaStream_t s) {
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  auto fn = encode_fn();
  if (!fn) return cudaErrorInvalidValue;
  const long long T = (long long)batch * seq;
  const int C = (n_head + 2 * n_kv_head) * HD;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(AT), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(C / AT)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2, static_cast<cuuint64_t>(AT) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(AT), static_cast<cuuint32_t>(BQ), 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(&p.qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(qkv), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  p.out = out;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;
  p.batch = batch;
  p.seq = seq;
  p.n_head = n_head;
  p.n_kv_head = n_kv_head;
  p.qtiles = (seq + BQ - 1) / BQ;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  cudaError_t e = cudaFuncSetAttribute(gqa_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ATT_SMEM);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.qtiles * n_head * batch;
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(gqa_attention_kernel, dim3((unsigned)blocks), dim3(ATT_THREADS), ATT_SMEM, s, p);
}

}  // namespace moe
