// Grouped expert GEMM on tcgen05 tensor cores, CTA-pair (2-SM) version for sm_103a.
//
// One persistent launch runs up to two operand sets: the routed experts (E groups,
// row ranges read from the device offsets of the counting sort, so there is no
// host round trip) and the shared expert (one group over all tokens).  Relay
// article, opening section, architecture paragraph: 64 routed experts plus one
// always-resident shared expert; SwiGLU is this library's reading of the expert FFN.
//
// Clusters of two CTAs on two SMs compute 256 x BN output tiles with
// tcgen05.mma.cta_group::2 (M = 256, N = BN <= 256, K = 16):
//   - each CTA stages its own 128 rows of A and one half (BN/2 rows) of B per
//     128-wide k-block (two 64-wide 128-byte-swizzle atoms each; 3-stage ring of
//     64 KB); both CTAs' TMA copies complete on the leader CTA's "full" barrier;
//     eight MMAs per barrier round keep the issuing thread ahead of the tensor
//     core (one wait per four MMAs measurably starved it);
//   - one thread of the leader CTA issues the MMAs; the pair's tensor cores read
//     the peer's half of B over the cluster, so each SM stages half the B bytes a
//     single-SM 128 x 256 tile would need;
//   - commits are multicast to both CTAs (stage release, accumulator ready);
//   - each CTA's accumulator holds its 128 rows x BN fp32 columns in TMEM, double
//     buffered (2 x 256 columns); 4 epilogue warps per CTA (one per TMEM lane quadrant) drain it:
//       SWIGLU  h = silu(gate) * up -> bf16 (gate / up rows interleaved in the
//               weights so one tile holds matching columns),
//       STORE   y -> bf16,
//       COMBINE out = acc + residual + sum_j gate_j * y_perm[inv_pos_j] (the shared
//               expert's down projection adds the same token's routed outputs:
//               the layer's combine step),
//       STORE_F32  fp32 out (weight gradients),
//       SWIGLU_BWD the SwiGLU backward from the recomputed pre-activations, dh staged
//               through shared memory by TMA.
// For the backward, either operand may be MN-major (the instruction descriptor's
// transpose bits read stored activations and weights where they are), the routed set
// may be grouped along K (weight gradients over each expert's rows), and the shared
// set may be split along K (separate bf16 parts, or fp32 parts added in order).
// A third, chained operand set may follow the other two in the same launch: routed
// groups whose A operand is the routed set's output (the down projection reading the
// h rows the gate/up tiles write).  Its tiles come after all others; each waits until
// every gate/up tile of its 256-row block has published its rows (a per-block counter:
// each epilogue warp fences its stores and adds one), so the down projection starts
// on pairs that are done with their gate/up work instead of after the launch ends.
// Every barrier wait is bounded (ptx.cuh); on a timeout the CTA records it in the
// status word, the pair drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 256;        // rows per CTA-pair tile
constexpr int HM = 128;        // rows per CTA
constexpr int AK = 64;         // K width of one 128-byte swizzle atom (bf16)
constexpr int ATOMS = 2;       // swizzle atoms per pipeline stage
constexpr int BK = ATOMS * AK; // K per pipeline stage: 8 MMAs per barrier round
constexpr int BN_MAX = 256;
constexpr int STAGES = 3;
constexpr int A_ATOM = HM * AK * 2;               // 16 KB: 128 rows x 64
constexpr int B_ATOM = (BN_MAX / 2) * AK * 2;     // 16 KB: up to 128 rows (half of B) x 64
constexpr int A_BYTES = ATOMS * A_ATOM;
constexpr int STAGE_BYTES = A_BYTES + ATOMS * B_ATOM; // 64 KB
constexpr int EPI_WARPS = 4;
constexpr int EPI_GROUPS = EPI_WARPS / 4;  // warps per TMEM lane quadrant
constexpr int CS = 32 * EPI_GROUPS;        // column stride between one warp's chunks
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int KS_BLOCK = 32;  // output tiles per block of a K-split shared set
constexpr uint32_t TMEM_COLS = 2 * BN_MAX;
// EPI_SWIGLU_BWD stages dh through shared memory: per epilogue warp two buffers of its
// 32 rows x 32 columns (bf16), filled by TMA.
constexpr int DH_COLS = 32;
constexpr int DH_BUF = 32 * DH_COLS * 2;                 // 2 KB
constexpr int DH_BYTES = EPI_WARPS * 2 * DH_BUF;         // 16 KB
constexpr int DYN_SMEM = STAGES * STAGE_BYTES + DH_BYTES + 1024;
constexpr unsigned FULL = 0xFFFFFFFFu;

struct OperandSet {
  // With kblock set (K a multiple of 64), both maps view a [rows][K] matrix as (64
  // columns, rows, K / 64 atoms) so that one copy brings a k-block's two 64-column
  // atoms: 128 rows x 64 x 2 for A, BN/2 rows for B (TMA's cost per copy makes two
  // 32 KB copies much faster than four of 16 KB).  Otherwise plain 2-D maps, box
  // (64, rows), one copy per atom.
  CUtensorMap a;
  CUtensorMap b;
  int kblock;
  void* out;
  int ldo, n_total, k_total, bn, mode, enabled, rows;
  int v8;   // output rows start on 32-byte boundaries: 256-bit stores allowed
  int v8h;  // the same for EPI_SWIGLU_BWD's dh rows
  int b_stream;  // B is streamed once (expert weights): its lines are the first L2 evicts
  // MN-major operands: the map views [K rows][M or N] as (64 elements, K rows, atoms
  // of 64 along M/N), box (64, BK, atoms per CTA), one copy per operand per k-block.
  int a_mn, b_mn;
  // Shared set split along K into ksplit >= 1 parts: EPI_STORE parts write out + part *
  // part_stride; EPI_STORE_F32 parts add into out in part order (see Params::kdep).
  int ksplit;
  long long part_stride;
  // EPI_SWIGLU_BWD operands (see GemmOperandSet); dhm views dh as [rows][n_total / 2]
  // with a 32 x 32 box.
  CUtensorMap dhm;
  uint16_t* dh;
  const float* gperm;
  float* dgpart;
};

struct Params {
  OperandSet shared;
  OperandSet routed;
  // Chained set (enabled or not): routed groups over the same offsets, A = the routed
  // set's output.  dep[m] counts the epilogue warps that have published routed 256-row
  // block m; a chained tile of block m waits for dep_target of them.
  OperandSet chain;
  int* dep;
  int dep_target;
  // fp32 K parts of the shared set: kdep[tile] counts the epilogue warps that have
  // written (part 0) or added (later parts) that output tile; part p adds once it
  // reaches 8 p, so the parts are summed in order and the result does not depend on
  // timing.  Zeroed by the caller.
  int* kdep;
  const int32_t* offsets;
  const uint16_t* y_perm;
  const int32_t* inv_pos;
  const float* gate;
  const uint16_t* residual;
  int* status;
  // Non-zero: the routed set is grouped along K instead of along the rows: group g
  // multiplies A[:, koff[g]..koff[g+1]) by B[:, same] (offsets holds koff, each a
  // multiple of 64) into its own output, out + g * group_stride; groups with an empty
  // range are skipped.  Used for the weight gradients, K running over tokens.
  int kgroup;
  long long group_stride;
  // Non-zero: the offsets and both sets' B operands were complete before the previous
  // kernel in the stream started, so the tile table and the first tile's B copies
  // may be issued before the dependency wait (the A copies and every output wait).
  int early;
  int E, k;
};

struct Tile {
  int set;    // 0 shared, 1 routed
  int row0;   // first A row of the pair's 256-row tile
  int rend;   // end (exclusive) of the group's rows
  int brow;   // first B row of the BN-row weight tile
  int n0;     // first accumulator column in the output
  int k0;     // first K column (K-grouped sets; else 0)
  int klen;   // K columns
  int group;  // K group (K-grouped sets; else 0)
  int bk;     // first K row of the group's B (MN-major B of an M-grouped set)
  int mblk;   // routed 256-row block index (routed and chained tiles)
};

// ---------------------------------------------------------------- cluster PTX

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Arrive without release semantics: for the accumulator hand-back, which orders only
// the epilogue's TMEM reads (complete once tcgen05.wait::ld returned) before the next
// MMAs.  A release here would hold every epilogue thread until its global stores of
// the tile were acknowledged.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA tile load whose completion is counted on a barrier of the CTA pair (here the
// leader's), given as a shared::cluster address.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}

// One k-block (two 64-column atoms) of a 3-D operand map, completion counted on the
// pair's (leader's) barrier.
__device__ __forceinline__ void tma_load_kblock_pair(uint32_t dst, const CUtensorMap* map,
                                                     uint32_t bar_cluster, int32_t row, int32_t atom) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(atom), "r"(bar_cluster)
      : "memory");
}

// The same with an L2 cache policy (createpolicy) for the copied lines.
__device__ __forceinline__ void tma_load_kblock_pair_hint(uint32_t dst, const CUtensorMap* map,
                                                          uint32_t bar_cluster, int32_t row, int32_t atom,
                                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(atom), "r"(bar_cluster), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void mma_pair_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at the same offset in both CTAs once this thread's MMAs finish.
__device__ __forceinline__ void commit_pair_multicast(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(0x3))
      : "memory");
}

__device__ __forceinline__ void commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// ---------------------------------------------------------------- helpers

// Tile order: with both operand sets present, shared-expert tiles (compute bound)
// and routed tiles (which stream expert weights from DRAM) are interleaved evenly,
// so every stretch of the launch mixes the two; each set keeps its own order.
// Largest group g with s_cum[g] <= r (that group is non-empty).
__device__ __forceinline__ int find_group(const int* s_cum, int E, int r) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_cum[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// `total` here is the end of the shared and routed tiles; chained tiles follow it.
__device__ __forceinline__ Tile decode_tile(const Params& p, int tile, int shared_tiles,
                                            const int* s_off, const int* s_cum, int total) {
  if (tile >= total) {
    // Chained tile: routed 256-row block m (the same blocks as the routed set's, whose
    // tile table counts nt1 tiles per block), column tile n.
    const int nt1 = p.routed.n_total / p.routed.bn, nt2 = p.chain.n_total / p.chain.bn;
    const int r = tile - total;
    const int m = r / nt2, n = r % nt2;
    const int g = find_group(s_cum, p.E, m * nt1);
    Tile t;
    t.set = 2;
    t.row0 = s_off[g] + (m - s_cum[g] / nt1) * BM;
    t.rend = s_off[g + 1];
    t.n0 = n * p.chain.bn;
    t.brow = g * p.chain.n_total + t.n0;
    t.k0 = 0;
    t.klen = p.chain.k_total;
    t.group = 0;
    t.bk = g * p.chain.k_total;
    t.mblk = m;
    return t;
  }
  const int routed_tiles = total - shared_tiles;
  if (shared_tiles > 0 && routed_tiles > 0) {
    // 32-bit arithmetic (tile counts stay far below 2^15).
    const unsigned r_before = (unsigned)tile * (unsigned)routed_tiles / (unsigned)total;
    const unsigned r_after = (unsigned)(tile + 1) * (unsigned)routed_tiles / (unsigned)total;
    tile = (r_after > r_before) ? shared_tiles + (int)r_before : tile - (int)r_before;
  }
  Tile t;
  t.k0 = 0;
  t.group = 0;
  t.bk = 0;
  t.mblk = 0;
  if (tile < shared_tiles) {
    // K parts in blocks of KS_BLOCK output tiles: the block's part 0 tiles, then its
    // part 1 tiles, ...: a tile's next part comes about two waves later, when the
    // previous one is done and its output still in L2.
    const int nt = p.shared.n_total / p.shared.bn, ks = p.shared.ksplit;
    const int mn_count = ((p.shared.rows + BM - 1) / BM) * nt;
    const int blk = tile / (KS_BLOCK * ks), within = tile % (KS_BLOCK * ks);
    const int nb = min(KS_BLOCK, mn_count - blk * KS_BLOCK);
    const int part = within / nb, mn = blk * KS_BLOCK + within % nb;
    const int m = mn / nt, n = mn % nt;
    t.set = 0;
    t.row0 = m * BM;
    t.rend = p.shared.rows;
    t.n0 = n * p.shared.bn;
    t.brow = t.n0;
    t.klen = p.shared.k_total / ks;
    t.k0 = part * t.klen;
    t.group = part;
    t.mblk = mn;
  } else if (p.kgroup) {
    const int r = tile - shared_tiles;
    const int nt = p.routed.n_total / p.routed.bn;
    const int tpg = ((p.routed.rows + BM - 1) / BM) * nt;
    const int g = r / tpg, local = r % tpg;
    t.set = 1;
    t.row0 = (local / nt) * BM;
    t.rend = p.routed.rows;
    t.n0 = (local % nt) * p.routed.bn;
    t.brow = t.n0;
    t.group = g;
    t.k0 = s_off[g];
    t.klen = s_off[g + 1] - s_off[g];
  } else {
    const int r = tile - shared_tiles;
    const int g = find_group(s_cum, p.E, r);
    const int nt = p.routed.n_total / p.routed.bn;
    const int local = r - s_cum[g];
    const int m = local / nt, n = local % nt;
    t.set = 1;
    t.row0 = s_off[g] + m * BM;
    t.rend = s_off[g + 1];
    t.n0 = n * p.routed.bn;
    t.brow = g * p.routed.n_total + t.n0;
    t.bk = g * p.routed.k_total;
    t.klen = p.routed.k_total;
    t.mblk = r / nt;  // s_cum[g] is a multiple of nt
  }
  return t;
}

// Which operand set a tile belongs to (1 = routed), by the same interleave as
// decode_tile: all the MMA issuer needs, without the search over the groups.
__device__ __forceinline__ int tile_set(int tile, int shared_tiles, int total) {
  if (tile >= total) return 2;
  const int routed_tiles = total - shared_tiles;
  if (shared_tiles > 0 && routed_tiles > 0) {
    const unsigned r_before = (unsigned)tile * (unsigned)routed_tiles / (unsigned)total;
    const unsigned r_after = (unsigned)(tile + 1) * (unsigned)routed_tiles / (unsigned)total;
    return r_after > r_before ? 1 : 0;
  }
  return shared_tiles > 0 && tile < shared_tiles ? 0 : 1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// silu(a) = a / (1 + e^-a).  The fast division has no special-value slow path; for
// very negative a the denominator overflows and the quotient is the correct 0.
__device__ __forceinline__ float silu(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// 32 bf16 values (64 bytes), cached in L2 only (gathered rows, used once).
__device__ __forceinline__ void load_row32(const uint16_t* src, uint4 (&u)[4]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int v = 0; v < 4; ++v) u[v] = __ldcg(s + v);
}

// o += w * (32 bf16 values in u).
__device__ __forceinline__ void accumulate_row32(float (&o)[32], const uint4 (&u)[4], float w) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint32_t ws[4] = {u[v].x, u[v].y, u[v].z, u[v].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[v * 8 + 2 * i] = fmaf(w, __uint_as_float(ws[i] << 16), o[v * 8 + 2 * i]);
      o[v * 8 + 2 * i + 1] = fmaf(w, __uint_as_float(ws[i] & 0xFFFF0000u), o[v * 8 + 2 * i + 1]);
    }
  }
}

__device__ __forceinline__ void add_bf16_row32(float (&o)[32], const uint16_t* src, float w) {
  uint4 u[4];
  load_row32(src, u);
  accumulate_row32(o, u, w);
}

// 32 fp32 values (raw bits) -> dst: four 256-bit stores with v8, else eight 128-bit.
__device__ __forceinline__ void store_f32_row32(float* dst, const uint32_t (&v)[32], int v8) {
  if (v8) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 8 * i),
                   "r"(v[8 * i]), "r"(v[8 * i + 1]), "r"(v[8 * i + 2]), "r"(v[8 * i + 3]),
                   "r"(v[8 * i + 4]), "r"(v[8 * i + 5]), "r"(v[8 * i + 6]), "r"(v[8 * i + 7])
                   : "memory");
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

// dst[0..32) += 32 fp32 values (raw bits), as eight 128-bit reductions performed in L2.
__device__ __forceinline__ void red_add_f32_row32(float* dst, const uint32_t (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * i), "f"(__uint_as_float(v[4 * i])),
                 "f"(__uint_as_float(v[4 * i + 1])), "f"(__uint_as_float(v[4 * i + 2])),
                 "f"(__uint_as_float(v[4 * i + 3]))
                 : "memory");
}

// 8 packed bf16 pairs (32 bytes) -> dst: one 256-bit store with v8, else two 128-bit.
__device__ __forceinline__ void store_packed16(uint16_t* dst, const uint32_t (&p)[8], int v8) {
  if (v8) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(p[0]),
                 "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7])
                 : "memory");
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(p[0], p[1], p[2], p[3]);
    d[1] = make_uint4(p[4], p[5], p[6], p[7]);
  }
}

// 32 values -> 64 bytes of bf16.  With v8, two 256-bit stores: half the store
// instructions of 128-bit ones and whole 32-byte sectors (the epilogue's rows are
// one per thread, so each warp store touches 32 lines).
__device__ __forceinline__ void store_bf16_row32(uint16_t* dst, const float (&o)[32], int v8) {
  uint32_t p[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);
  if (v8) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * h),
                   "r"(p[8 * h]), "r"(p[8 * h + 1]), "r"(p[8 * h + 2]), "r"(p[8 * h + 3]),
                   "r"(p[8 * h + 4]), "r"(p[8 * h + 5]), "r"(p[8 * h + 6]), "r"(p[8 * h + 7])
                   : "memory");
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < 4; ++v) d[v] = make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
  }
}

// Waits (acquire, at GPU scope) until *ctr >= target, then orders this thread's later
// TMA reads (async proxy) after the generic-proxy stores the counter published.
// Bounded like the barrier waits.
__device__ __forceinline__ bool dep_wait(const int* ctr, int target, int* status) {
  if (!wait_counter_geq(ctr, target, status, kWaitLimitNs)) return false;
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];   // used in the leader
  __shared__ __align__(8) uint64_t empty_bar[STAGES];  // both CTAs
  __shared__ __align__(8) uint64_t tfull_bar[2];       // both CTAs
  __shared__ __align__(8) uint64_t tempty_bar[2];      // used in the leader
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t dh_bar[EPI_WARPS][2];  // dh staging buffers
  __shared__ uint32_t tmem_holder;
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_cum[kMaxE + 1];
  __shared__ int s_total;
  __shared__ int s_t1;  // end of the shared and routed tiles (chained tiles follow)

  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int shared_tiles =
      p.shared.enabled ? ((p.shared.rows + BM - 1) / BM) * (p.shared.n_total / p.shared.bn) * p.shared.ksplit
                       : 0;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull_bar[a]), 1);
      mbar_init(smem_u32(&tempty_bar[a]), 2 * EPI_WARPS);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    for (int w = 0; w < EPI_WARPS; ++w) {
      mbar_init(smem_u32(&dh_bar[w][0]), 1);
      mbar_init(smem_u32(&dh_bar[w][1]), 1);
    }
    fence_mbar_init();
    if (p.shared.enabled) {
      tma_prefetch_desc(&p.shared.a);
      tma_prefetch_desc(&p.shared.b);
    }
    if (p.routed.enabled) {
      tma_prefetch_desc(&p.routed.a);
      tma_prefetch_desc(&p.routed.b);
    }
    if (p.chain.enabled) {
      tma_prefetch_desc(&p.chain.a);
      tma_prefetch_desc(&p.chain.b);
    }
    if (p.shared.mode == EPI_SWIGLU_BWD && p.shared.enabled) tma_prefetch_desc(&p.shared.dhm);
    if (p.routed.mode == EPI_SWIGLU_BWD && p.routed.enabled) tma_prefetch_desc(&p.routed.dhm);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_holder), TMEM_COLS);
    tmem_relinquish_pair();
  }
  // Set-up above is CTA-local; the offsets and operands come from earlier kernels.
  // With `early`, everything up to the first tile's B copies runs before the wait.
  if (!p.early) {
    pdl_wait();
    pdl_trigger();
  }
  if (warp == 2) {
    // Tile table of the routed groups: s_cum[g] = tiles of groups < g.
    int carry = 0;
    if (p.routed.enabled && p.kgroup) {
      // K-grouped: a fixed number of tiles per group; s_off holds the K offsets.
      for (int g = lane; g <= p.E; g += 32) s_off[g] = p.offsets[g];
      carry = p.E * ((p.routed.rows + BM - 1) / BM) * (p.routed.n_total / p.routed.bn);
    } else if (p.routed.enabled) {
      const int nt = p.routed.n_total / p.routed.bn;
      // All offsets in one round trip, then the counts from shared memory.
      int ov[(kMaxE + 1 + 31) / 32];
#pragma unroll
      for (int i = 0; i < (kMaxE + 1 + 31) / 32; ++i)
        if (lane + 32 * i <= p.E) ov[i] = p.offsets[lane + 32 * i];
#pragma unroll
      for (int i = 0; i < (kMaxE + 1 + 31) / 32; ++i)
        if (lane + 32 * i <= p.E) s_off[lane + 32 * i] = ov[i];
      __syncwarp();
      for (int b = 0; b < p.E; b += 32) {
        const int g = b + lane;
        int v = 0;
        if (g < p.E) v = ((s_off[g + 1] - s_off[g] + BM - 1) / BM) * nt;
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
    if (lane == 0) {
      // Chained tiles: one row of nt2 column tiles per routed 256-row block.
      const int chained = (p.chain.enabled && p.routed.enabled && !p.kgroup)
                              ? carry / (p.routed.n_total / p.routed.bn) * (p.chain.n_total / p.chain.bn)
                              : 0;
      s_t1 = shared_tiles + carry;
      s_total = shared_tiles + carry + chained;
    }
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;
  const int total = s_total, t1 = s_t1;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      const uint64_t evict_first = l2_evict_first_policy();
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      // Early start: the first tile's B copies (and the stage's expected bytes) go out
      // now, into the empty ring; after the wait its first `pre` k-blocks load A only.
      int pre = 0;
      if (p.early) {
        if (cluster < t1) {
          const Tile t = decode_tile(p, cluster, shared_tiles, s_off, s_cum, t1);
          const OperandSet& S = t.set == 2 ? p.chain : (t.set ? p.routed : p.shared);
          const int nkb = (t.klen + BK - 1) / BK;
          const int half = S.bn / 2;
          if (S.kblock) {
            pre = min(nkb, STAGES);
            for (int kb = 0; kb < pre; ++kb) {
              const uint32_t sa = ring + kb * STAGE_BYTES;
              const uint32_t fb = map_to_rank(smem_u32(&full_bar[kb]), 0);
              if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[kb]), 2u * ATOMS * (A_ATOM + half * AK * 2));
              if (S.b_mn)
                tma_load_kblock_pair(sa + A_BYTES, &S.b, fb, t.bk + t.k0 + kb * BK, (t.n0 + half * (int)rank) / AK);
              else
                tma_load_kblock_pair(sa + A_BYTES, &S.b, fb, t.brow + half * (int)rank, t.k0 / AK + kb * ATOMS);
            }
          }
        }
        pdl_wait();
        pdl_trigger();
      }
      for (int tile = cluster; tile < total && ok; tile += nclusters) {
        const Tile t = decode_tile(p, tile, shared_tiles, s_off, s_cum, t1);
        const OperandSet& S = t.set == 2 ? p.chain : (t.set ? p.routed : p.shared);
        // A chained tile's A rows are written by this launch's gate/up tiles.
        if (t.set == 2 && !dep_wait(p.dep + t.mblk, p.dep_target, p.status)) {
          ok = false;
          break;
        }
        const int nkb = (t.klen + BK - 1) / BK;  // 0 for an empty K group: nothing loaded
        const int half = S.bn / 2;
        const int katom0 = t.k0 / AK;
        for (int kb = 0; kb < nkb; ++kb) {
          const bool b_done = tile == cluster && kb < pre;  // B (and the byte count) already out
          if (!b_done && !mbar_wait_spin(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          // Both atoms of the k-block in one copy per operand (an atom past K arrives
          // zero-filled and is not multiplied); with 2-D maps, atoms past K are not
          // loaded at all.  MN-major operands: one copy of BK rows (k) by the CTA's
          // 64-element atoms along M / N; rows past K arrive as zeros or belong to the
          // next group and meet zero (or unmultiplied) columns of the other operand.
          const int natoms = S.kblock ? ATOMS : min(ATOMS, (t.klen - kb * BK + AK - 1) / AK);
          const uint32_t pair_bytes = 2u * natoms * (A_ATOM + half * AK * 2);
          const uint32_t sa = ring + stage * STAGE_BYTES;
          const uint32_t fb = map_to_rank(smem_u32(&full_bar[stage]), 0);
          const uint32_t b_atom = (uint32_t)half * AK * 2;
          if (leader && !b_done) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), pair_bytes);
          if (S.a_mn | S.b_mn) {
            const int kk0 = t.k0 + kb * BK;
            if (S.a_mn)
              tma_load_kblock_pair(sa, &S.a, fb, kk0, (t.row0 + HM * (int)rank) / AK);
            else
              tma_load_kblock_pair(sa, &S.a, fb, t.row0 + HM * (int)rank, katom0 + kb * ATOMS);
            if (b_done) {
            } else if (S.b_mn) {
              tma_load_kblock_pair(sa + A_BYTES, &S.b, fb, t.bk + kk0, (t.n0 + half * (int)rank) / AK);
            } else {
              tma_load_kblock_pair(sa + A_BYTES, &S.b, fb, t.brow + half * (int)rank, katom0 + kb * ATOMS);
            }
          } else if (S.kblock) {
            tma_load_kblock_pair(sa, &S.a, fb, t.row0 + HM * (int)rank, katom0 + kb * ATOMS);
            if (b_done) {
            } else if (S.b_stream) {
              tma_load_kblock_pair_hint(sa + A_BYTES, &S.b, fb, t.brow + half * (int)rank, katom0 + kb * ATOMS,
                                        evict_first);
            } else {
              tma_load_kblock_pair(sa + A_BYTES, &S.b, fb, t.brow + half * (int)rank, katom0 + kb * ATOMS);
            }
          } else {
            for (int at = 0; at < natoms; ++at) {
              tma_load_2d_pair(sa + at * A_ATOM, &S.a, fb, t.k0 + kb * BK + at * AK,
                               t.row0 + HM * (int)rank);
              tma_load_2d_pair(sa + A_BYTES + at * b_atom, &S.b, fb, t.k0 + kb * BK + at * AK,
                               t.brow + half * (int)rank);
            }
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // The leader's full barriers count both CTAs' copies: wait for all of them.
      if (leader)
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1u) mbar_wait_spin(smem_u32(&full_bar[s]), (last_par >> s) & 1u, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer (leader only)
      // The loop body is kept to the barrier waits and the MMAs: the operand set's
      // fields are read (as plain kernel-parameter loads) once per tile, not through a
      // reference into parameter space on every k-block.
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += nclusters) {
        const int set = tile_set(tile, shared_tiles, t1);
        int k_total = set == 2 ? p.chain.k_total : (set ? p.routed.k_total : p.shared.k_total / p.shared.ksplit);
        if (set == 1 && p.kgroup) {  // this tile's K group
          k_total = decode_tile(p, tile, shared_tiles, s_off, s_cum, t1).klen;
          if (k_total == 0) continue;  // empty group: no MMA, no accumulator hand-off
        }
        const int bn = set == 2 ? p.chain.bn : (set ? p.routed.bn : p.shared.bn);
        const int a_mn = set == 2 ? p.chain.a_mn : (set ? p.routed.a_mn : p.shared.a_mn);
        const int b_mn = set == 2 ? p.chain.b_mn : (set ? p.routed.b_mn : p.shared.b_mn);
        const int nkb = (k_total + BK - 1) / BK;
        const int nkk_last = (k_total - (nkb - 1) * BK + 15) / 16;
        const uint32_t b_atom = (uint32_t)bn / 2 * AK * 2;
        const uint32_t idesc = idesc_bf16_f32(BM, bn, a_mn, b_mn);
        // Descriptor advance (16-byte units) of K step kk = 4 * x + y: K-major, x picks
        // the 64-column atom and y moves 32 B inside its rows; MN-major, every step is
        // two 1024-byte atoms further along K.
        const uint32_t ax = a_mn ? 512u : (uint32_t)(A_ATOM >> 4), ay = a_mn ? 128u : 2u;
        const uint32_t bx = b_mn ? 512u : (b_atom >> 4), by = b_mn ? 128u : 2u;
        if (!mbar_wait_spin(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN_MAX;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_spin(smem_u32(&full_bar[stage]), phase, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = ring + stage * STAGE_BYTES;
          // MN-major: atom columns (64 elements x BK rows) are BK * 128 B apart.
          const uint64_t adesc = a_mn ? sw128_mnmajor_desc(sa, BK * 128) : sw128_kmajor_desc(sa);
          const uint64_t bdesc = b_mn ? sw128_mnmajor_desc(sa + A_BYTES, BK * 128)
                                      : sw128_kmajor_desc(sa + A_BYTES);
          if (kb + 1 < nkb) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_pair_bf16(d_tmem, adesc + (kk >> 2) * ax + (kk & 3) * ay,
                            bdesc + (kk >> 2) * bx + (kk & 3) * by, idesc, (kb | kk) != 0);
          } else {
            for (int kk = 0; kk < nkk_last; ++kk)
              mma_pair_bf16(d_tmem, adesc + (kk >> 2) * ax + (kk & 3) * ay,
                            bdesc + (kk >> 2) * bx + (kk & 3) * by, idesc, (kb | kk) != 0);
          }
          commit_pair_multicast(smem_u32(&empty_bar[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        commit_pair_multicast(smem_u32(&tfull_bar[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA must finish before TMEM is released.
      commit_pair_local(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, p.status);
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;                 // TMEM lanes [32q, 32q + 32) are this warp's rows
    const int colh = (warp - 2) / 4;        // which interleaved share of the column chunks
    const uint32_t tempty_leader0 = map_to_rank(smem_u32(&tempty_bar[0]), 0);
    const uint32_t tempty_leader1 = map_to_rank(smem_u32(&tempty_bar[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t dh_par = 0;  // parity of this warp's two dh buffers
    const uint32_t dh_stage = ring + STAGES * STAGE_BYTES + (uint32_t)(warp - 2) * 2 * DH_BUF;
    if (p.early) pdl_wait();  // outputs and epilogue inputs belong to earlier kernels
    for (int tile = cluster; tile < total; tile += nclusters) {
      const Tile t = decode_tile(p, tile, shared_tiles, s_off, s_cum, t1);
      const OperandSet& S = t.set == 2 ? p.chain : (t.set ? p.routed : p.shared);
      if (t.klen == 0) {
        // Empty K group (an expert without tokens): the issuer skipped it; its fp32
        // output is zero.
        const long long orow = (long long)t.row0 + HM * (int)rank + q * 32 + lane;
        if (S.mode == EPI_STORE_F32 && orow < t.rend) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(S.out) +
                                                  (long long)t.group * p.group_stride + orow * S.ldo + t.n0);
          for (int c = 4 * colh; c < S.bn / 4; c += 4 * EPI_GROUPS)
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[c + i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        continue;
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, p.status) ? 1 : 0;
      ok = __shfl_sync(FULL, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int r = q * 32 + lane;
      const long long orow = (long long)t.row0 + HM * (int)rank + r;
      const bool valid = orow < t.rend;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN_MAX;
      uint16_t* out = static_cast<uint16_t*>(S.out) + (t.set == 0 ? t.group * S.part_stride : 0);
      if (S.mode == EPI_SWIGLU) {
        const int half = S.bn / 2;
        for (int c = 32 * colh; c < half; c += CS) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c, g);
          tmem_ld32(tbase + half + c, u);
          tmem_wait_ld();
          float h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) h[i] = silu(__uint_as_float(g[i])) * __uint_as_float(u[i]);
          if (valid) store_bf16_row32(out + orow * S.ldo + t.n0 / 2 + c, h, S.v8);
        }
      } else if (S.mode == EPI_SWIGLU_BWD) {
        // SwiGLU backward with the pre-activations in TMEM (gate columns [0, half),
        // up columns [half, bn) of the tile, as for EPI_SWIGLU): with dh read from
        // memory and g the row's gate, da = g dh b silu'(a) and db = g dh silu(a) go to
        // out (the accumulator's column order), g h replaces dh, and the partial
        // <dh, h> of the tile's columns goes to dgpart.
        const int half = S.bn / 2, w = S.n_total / 2;
        const float g = (valid && S.gperm) ? S.gperm[orow] : 1.0f;
        uint16_t* dhr = S.dh + orow * w + t.n0 / 2;
        uint16_t* o = out + orow * S.ldo + t.n0;
        // The element math runs on column pairs with the packed fp32x2 instructions
        // (the exponential and the reciprocal per element).
        const float2 one2 = make_float2(1.0f, 1.0f), g2 = make_float2(g, g);
        float2 dot2 = make_float2(0.f, 0.f);
        auto chunk = [&](int c, const uint4 (&u)[2]) {
          uint32_t va[16], vb[16];
          tmem_ld16(tbase + c, va);
          tmem_ld16(tbase + half + c, vb);
          tmem_wait_ld();
          if (!valid) return;
          uint32_t pa[8], pb[8], ph[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t dw = reinterpret_cast<const uint32_t*>(u)[i];
            const float2 a = make_float2(__uint_as_float(va[2 * i]), __uint_as_float(va[2 * i + 1]));
            const float2 b = make_float2(__uint_as_float(vb[2 * i]), __uint_as_float(vb[2 * i + 1]));
            const float2 dh = make_float2(__uint_as_float(dw << 16), __uint_as_float(dw & 0xFFFF0000u));
            const float2 den = __fadd2_rn(one2, make_float2(__expf(-a.x), __expf(-a.y)));
            const float2 sig = make_float2(__fdividef(1.0f, den.x), __fdividef(1.0f, den.y));
            const float2 sa = __fmul2_rn(a, sig);                       // silu(a)
            const float2 h = __fmul2_rn(sa, b);
            dot2 = __ffma2_rn(dh, h, dot2);
            const float2 dhg = __fmul2_rn(g2, dh);
            // silu'(a) = sig (1 + a (1 - sig))
            const float2 oms = __ffma2_rn(sig, make_float2(-1.0f, -1.0f), one2);
            const float2 ds = __fmul2_rn(sig, __ffma2_rn(a, oms, one2));
            const float2 da = __fmul2_rn(__fmul2_rn(dhg, b), ds);
            const float2 db = __fmul2_rn(dhg, sa);
            const float2 gh = __fmul2_rn(g2, h);
            pa[i] = pack_bf16x2(da.x, da.y);
            pb[i] = pack_bf16x2(db.x, db.y);
            ph[i] = pack_bf16x2(gh.x, gh.y);
          }
          store_packed16(o + c, pa, S.v8);
          store_packed16(o + half + c, pb, S.v8);
          store_packed16(dhr + c, ph, S.v8h);
        };
        // dh arrives by TMA, 32 rows x 32 columns per piece into this warp's two shared
        // buffers, one piece ahead: read row by row from global memory, each thread's
        // loads (32 rows per warp instruction) beside its stores cost the epilogue more
        // than its math.
        static_assert(EPI_GROUPS == 1, "one epilogue warp per TMEM lane quadrant");
        const int pieces = half / DH_COLS;  // half is 32, 64 or 128
        const int wrow = t.row0 + HM * (int)rank + q * 32;
        auto issue = [&](int pc) {
          const uint32_t bar = smem_u32(&dh_bar[warp - 2][pc & 1]);
          mbar_arrive_expect_tx(bar, DH_BUF);
          tma_load_2d(dh_stage + (pc & 1) * DH_BUF, &S.dhm, bar, t.n0 / 2 + pc * DH_COLS, wrow);
        };
        if (lane == 0) {
          issue(0);
          if (pieces > 1) issue(1);
        }
        bool dh_ok = true;
        for (int pc = 0; pc < pieces && dh_ok; ++pc) {
          const int b = pc & 1;
          dh_ok = mbar_wait(smem_u32(&dh_bar[warp - 2][b]), (dh_par >> b) & 1u, p.status);
          dh_par ^= 1u << b;
          if (!dh_ok) break;
          const uint32_t row = dh_stage + b * DH_BUF + lane * (DH_COLS * 2);
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {
            uint4 u[2];
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(u[0].x), "=r"(u[0].y), "=r"(u[0].z), "=r"(u[0].w) : "r"(row + sub * 32));
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(u[1].x), "=r"(u[1].y), "=r"(u[1].z), "=r"(u[1].w) : "r"(row + sub * 32 + 16));
            chunk(pc * DH_COLS + sub * 16, u);
          }
          // Every lane has read buffer b: the next piece may overwrite it.
          __syncwarp();
          if (lane == 0 && pc + 2 < pieces) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(pc + 2);
          }
        }
        if (!dh_ok) break;
        if (valid && S.dgpart) S.dgpart[orow * (S.n_total / S.bn) + t.n0 / S.bn] = dot2.x + dot2.y;
      } else if (S.mode == EPI_STORE_F32) {
        // fp32 output (weight gradients); K groups write their own matrices.  Two
        // 32-column chunks per TMEM round trip; 256-bit stores (whole 32-byte sectors,
        // one row per thread) when aligned.
        // A later K part of the shared set waits for the earlier ones, then adds.
        const int part = (t.set == 0 && S.ksplit > 1) ? t.group : 0;
        if (part > 0) {
          int ok2 = 1;
          if (lane == 0) ok2 = dep_wait(p.kdep + t.mblk, 2 * EPI_WARPS * part, p.status) ? 1 : 0;
          ok2 = __shfl_sync(FULL, ok2, 0);
          __syncwarp();
          if (!ok2) break;
        }
        float* o32 = static_cast<float*>(S.out) + (t.set == 1 ? (long long)t.group * p.group_stride : 0) +
                     orow * S.ldo + t.n0;
        for (int c = 32 * colh; c < S.bn; c += 2 * CS) {
          const bool two = c + CS < S.bn;  // warp-uniform
          uint32_t v[32], w[32];
          tmem_ld32(tbase + c, v);
          if (two) tmem_ld32(tbase + c + CS, w);
          tmem_wait_ld();
          if (valid && part > 0) {
            red_add_f32_row32(o32 + c, v);
            if (two) red_add_f32_row32(o32 + c + CS, w);
          } else if (valid) {
            store_f32_row32(o32 + c, v, S.v8);
            if (two) store_f32_row32(o32 + c + CS, w, S.v8);
          }
        }
        if (t.set == 0 && S.ksplit > 1) {
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            atomicAdd(p.kdep + t.mblk, 1);
          }
        }
      } else if (S.mode == EPI_STORE) {
        // Two 32-column chunks per TMEM round trip.
        for (int c = 32 * colh; c < S.bn; c += 2 * CS) {
          const bool two = c + CS < S.bn;  // warp-uniform
          uint32_t v[32], w[32];
          tmem_ld32(tbase + c, v);
          if (two) tmem_ld32(tbase + c + CS, w);
          tmem_wait_ld();
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]);
          if (valid) store_bf16_row32(out + orow * S.ldo + t.n0 + c, o, S.v8);
          if (two) {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(w[i]);
            if (valid) store_bf16_row32(out + orow * S.ldo + t.n0 + c + CS, o, S.v8);
          }
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
        for (int c = 32 * colh; c < S.bn; c += CS) {
          uint32_t v[32];
          tmem_ld32(tbase + c, v);
          // The residual and the first two routed rows are requested together, and
          // while the accumulator chunk is read, so their latencies overlap.
          const long long col = t.n0 + c;
          uint4 ur[4], u0[4], u1[4];
          if (valid) {
            if (p.residual) load_row32(p.residual + orow * S.ldo + col, ur);
            if (p.k > 0) load_row32(p.y_perm + pj[0] * S.ldo + col, u0);
            if (p.k > 1) load_row32(p.y_perm + pj[1] * S.ldo + col, u1);
          }
          tmem_wait_ld();
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]);
          if (valid) {
            if (p.residual) accumulate_row32(o, ur, 1.f);
            if (p.k > 0) accumulate_row32(o, u0, gj[0]);
            if (p.k > 1) accumulate_row32(o, u1, gj[1]);
#pragma unroll
            for (int j = 2; j < kMaxK; ++j)
              if (j < p.k) add_bf16_row32(o, p.y_perm + pj[j] * S.ldo + col, gj[j]);
            store_bf16_row32(out + orow * S.ldo + col, o, S.v8);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster_relaxed(acc ? tempty_leader1 : tempty_leader0);
        // Publish the warp's rows of a routed tile to the chained tiles: the stores
        // above (ordered before this lane by the warp barrier), then the count.
        if (t.set == 1 && p.dep) {
          __threadfence();
          atomicAdd(p.dep + t.mblk, 1);
        }
      }

      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the pair still has copies or MMAs in flight
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
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

// bf16 matrix [outer][inner] row-major, box [box_outer][64] (one swizzle atom) with the
// 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(AK), box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same matrix as (64 columns, outer rows, inner / 64 atoms), box (64, box_outer,
// box_atoms): one copy = box_atoms consecutive 64-column atoms, each [box_outer][64]
// with the 128-byte swizzle, box_outer * 128 bytes apart.  K-major operands: inner = K,
// two atoms = one k-block.  MN-major operands: inner = M or N, outer = K rows,
// box_outer = BK.
bool make_map_kblock(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                     uint32_t box_outer, uint32_t box_atoms = ATOMS) {
  auto fn = encode_fn();
  if (!fn || inner % AK != 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(AK), outer, inner / AK};
  const cuuint64_t strides[2] = {inner * 2, static_cast<cuuint64_t>(AK) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(AK), box_outer, box_atoms};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int gate_up_block(int width) { return width % 128 == 0 ? 128 : (width % 64 == 0 ? 64 : 32); }

int choose_bn(int mode, int N) {
  if (mode == EPI_SWIGLU) return 2 * gate_up_block(N / 2);
  if (mode == EPI_STORE_F32) return N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : (N % 64 == 0 ? 64 : 32));
  if (mode == EPI_SWIGLU_BWD) return 2 * gate_up_block(N / 2);
  return N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : 64);
}

// Largest number of co-resident 2-CTA clusters for this kernel on the current device.
int max_active_pairs() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int sms = 1;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int pairs = sms / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = DYN_SMEM;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel, &cfg) == cudaSuccess && n > 0)
    pairs = std::min(pairs, n);
  if (dev >= 0 && dev < 64) cached[dev] = pairs;
  return pairs;
}

bool fill_set(OperandSet& t, const GemmOperandSet& o) {
  std::memset(&t, 0, sizeof(t));
  t.ksplit = 1;
  if (!o.a) return true;
  t.enabled = 1;
  t.bn = choose_bn(o.mode, o.N);
  t.n_total = o.N;
  t.k_total = o.K;
  t.ldo = o.ldo;
  t.mode = o.mode;
  t.rows = o.rows;
  t.out = o.out;
  t.ksplit = o.ksplit > 1 ? o.ksplit : 1;
  t.part_stride = o.part_stride;
  // Every part a whole number of 64-wide K atoms; separate bf16 parts or fp32 sums.
  if (t.ksplit > 1 && (o.K % (AK * t.ksplit) != 0 || (o.mode != EPI_STORE && o.mode != EPI_STORE_F32)))
    return false;
  t.dh = o.dh;
  t.gperm = o.gperm;
  t.dgpart = o.dgpart;
  // 256-bit stores of the h-width rows (EPI_SWIGLU_BWD's dh) need 32-byte alignment too.
  t.v8h = (reinterpret_cast<uintptr_t>(o.dh) % 32 == 0) && ((long long)o.N / 2 * 2) % 32 == 0;
  if (o.mode == EPI_SWIGLU_BWD) {
    // dh [a_rows][N / 2], 32 x 32 boxes at 32-column offsets (64-byte aligned).
    if (!o.dh || (o.N / 2) % DH_COLS != 0) return false;
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(o.N / 2), static_cast<cuuint64_t>(o.a_rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(o.N / 2) * 2};
    const cuuint32_t box[2] = {DH_COLS, 32};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&t.dhm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.dh, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  const int esize = o.mode == EPI_STORE_F32 ? 4 : 2;
  t.v8 = (reinterpret_cast<uintptr_t>(o.out) % 32 == 0) && ((long long)o.ldo * esize) % 32 == 0;
  if (o.N % t.bn != 0) return false;
  t.a_mn = o.a_mn ? 1 : 0;
  t.b_mn = o.b_mn ? 1 : 0;
  t.b_stream = o.b_stream ? 1 : 0;
  if (t.a_mn || t.b_mn) {
    // Whole k-blocks of both operands per copy (the expected byte count assumes it).
    if ((!t.a_mn || !t.b_mn) && o.K % AK != 0) return false;
    if (t.b_mn && t.bn % 128 != 0) return false;
    t.kblock = 1;
    const bool ma = t.a_mn ? make_map_kblock(&t.a, o.a, o.rows, o.K, BK, HM / AK)
                           : make_map_kblock(&t.a, o.a, o.K, o.a_rows, HM);
    const bool mb = t.b_mn ? make_map_kblock(&t.b, o.b, o.N, (uint64_t)o.groups * o.K, BK, t.bn / 2 / AK)
                           : make_map_kblock(&t.b, o.b, o.K, (uint64_t)o.groups * o.N, t.bn / 2);
    return ma && mb;
  }
  t.kblock = o.K % AK == 0;
  if (t.kblock) {
    if (!make_map_kblock(&t.a, o.a, o.K, o.a_rows, HM)) return false;
    if (!make_map_kblock(&t.b, o.b, o.K, (uint64_t)o.groups * o.N, t.bn / 2)) return false;
  } else {
    if (!make_map(&t.a, o.a, o.K, o.a_rows, HM)) return false;
    if (!make_map(&t.b, o.b, o.K, (uint64_t)o.groups * o.N, t.bn / 2)) return false;
  }
  return true;
}

}  // namespace

int gemm_tile_n(int mode, int N) { return choose_bn(mode, N); }

bool make_tma_map_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                       uint32_t box_outer) {
  return make_map(m, ptr, inner, outer, box_outer);
}

int gemm_max_pairs() {
  if (cudaFuncSetAttribute(grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DYN_SMEM) != cudaSuccess)
    return 1;
  return max_active_pairs();
}

cudaError_t launch_grouped_gemm(const GemmOperandSet& routed, const int32_t* offsets, int E,
                                const GemmOperandSet& shared, const CombineInputs& comb,
                                long long max_routed_rows, cudaStream_t s, int* bad_arg,
                                int max_pairs, long long kgroup_stride, int early,
                                const GemmOperandSet* chain, int32_t* dep, int32_t* kdep) {
  Params p;
  std::memset(&p, 0, sizeof(p));
  *bad_arg = 0;
  if (!fill_set(p.shared, shared) || !fill_set(p.routed, routed) ||
      (chain && !fill_set(p.chain, *chain))) {
    *bad_arg = 1;
    return cudaErrorInvalidValue;
  }
  if (p.chain.enabled) {
    // The chained set reads the routed set's output rows block by block.
    if (!p.routed.enabled || kgroup_stride > 0 || !dep || chain->groups != E ||
        chain->a != routed.out || chain->K != routed.ldo || routed.mode != EPI_SWIGLU) {
      *bad_arg = 1;
      return cudaErrorInvalidValue;
    }
    p.dep = dep;
    p.dep_target = (p.routed.n_total / p.routed.bn) * 2 * EPI_WARPS;
  }
  if (p.shared.ksplit > 1 && p.shared.mode == EPI_STORE_F32) {
    if (!kdep) {
      *bad_arg = 1;
      return cudaErrorInvalidValue;
    }
    p.kdep = kdep;
  }
  if (!p.shared.enabled && !p.routed.enabled) return cudaSuccess;
  p.offsets = offsets;
  p.E = E;
  p.y_perm = comb.y_perm;
  p.inv_pos = comb.inv_pos;
  p.gate = comb.gate;
  p.residual = comb.residual;
  p.k = comb.k;
  p.early = early ? 1 : 0;
  p.kgroup = kgroup_stride > 0 ? 1 : 0;
  p.group_stride = kgroup_stride;
  if (p.kgroup && kgroup_stride % 8 != 0) p.routed.v8 = 0;  // groups' fp32 outputs off 32 B
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;

  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, DYN_SMEM);
  if (e != cudaSuccess) return e;
  long long tiles = 0;
  if (p.shared.enabled)
    tiles += (long long)((p.shared.rows + BM - 1) / BM) * (p.shared.n_total / p.shared.bn) * p.shared.ksplit;
  if (p.routed.enabled && p.kgroup)
    tiles += (long long)E * ((p.routed.rows + BM - 1) / BM) * (p.routed.n_total / p.routed.bn);
  else if (p.routed.enabled)
    tiles += ((max_routed_rows + BM - 1) / BM + E) * (long long)(p.routed.n_total / p.routed.bn);
  if (p.chain.enabled)
    tiles += ((max_routed_rows + BM - 1) / BM + E) * (long long)(p.chain.n_total / p.chain.bn);
  int cap = max_active_pairs();
  if (max_pairs > 0 && max_pairs < cap) cap = max_pairs;
  const int pairs = (int)std::min<long long>(cap, std::max<long long>(tiles, 1));
  return launch_pdl(grouped_gemm_kernel, dim3(2 * pairs), dim3(NUM_THREADS), DYN_SMEM, s, p);
}

}  // namespace moe
