// Host-side launcher interface shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include <utility>

#include "moe_gb300.h"

namespace moe {

// Host validation of a layer shape (the envelope of moe_gb300.h); every entry point
// that takes a moe_shape_t returns its status first.
moe_status_t check_shape(const moe_shape_t* s);

// Launch with programmatic dependent launch: the kernel may be scheduled while the
// previous kernel in the stream is still running; it must execute
// griddepcontrol.wait (pdl_wait) before touching memory that earlier work writes
// or reads.  This hides the launch gap between the layer's consecutive kernels.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device status bits (OR-ed into the library's status word).
constexpr int kDevTimeout = 1;
constexpr int kDevCheck = 2;

constexpr int kMaxE = 256;
constexpr int kMaxK = 8;
constexpr int kRouterTokens = 32;   // tokens per router block
constexpr int kRouterClusterMaxT = 256;  // up to this T the SIMT router uses CTA clusters

// Tokens per permutation chunk: a multiple of kRouterTokens chosen so the chunk
// count table (chunks x E int32) stays within kMaxCountEntries.
constexpr int kMaxCountEntries = 32768;
int permute_chunk_tokens(int T, int E);

// Library status word (device), OR-ed by kernels; owned by moe_api.cu.
int* device_status_ptr();

// ---------------------------------------------------------------- router
struct RouterArgs {
  const void* x;
  int x_is_f32;
  const float* w_router;
  const float* logit_offset;
  const float* bias;
  float* scores;        // nullable
  int32_t* idx;
  float* gate;
  int32_t* load;        // nullable (SIMT routers); zeroed by the caller; atomically accumulated
  int32_t* counts;      // nullable: [chunks][E], zeroed by the caller
  int chunk_tokens;
  int T, d, E, k, renorm;
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);
// Router of the permutation-free serving path (bf16 tokens, T <= kDirectMaxPairs, no
// chunk counts): writes the loads outright (no clearing); zeroes its own counter in
// the scratch of router_small_scratch_bytes(T, E).
bool router_small_supported(const RouterArgs& a);
size_t router_small_scratch_bytes(int T, int E);
cudaError_t launch_router_small(const RouterArgs& a, void* scratch, cudaStream_t s);
// Tensor-core router (bf16 tokens, T >= 128, E in {16, 32, 48, 64, 80}); needs
// scratch for the three-way bf16 split of the router weight.
bool router_tc_supported(int T, int E, int x_is_f32);
size_t router_tc_scratch_bytes(int E, int d);
// Also zeroes a.load [E] and, when set, a.counts [(T / chunk_tokens rounded up) * E]
// before the router's atomics (no separate memsets in the launch chain).
cudaError_t launch_router_tc(const RouterArgs& a, void* w3_scratch, cudaStream_t s);

// ---------------------------------------------------------------- permutation
cudaError_t launch_count(const int32_t* idx, int T, int k, int E, int chunk_tokens,
                         int32_t* counts, cudaStream_t s);
// Whole permutation from the per-chunk count table [chunks][E]: expert offsets
// [E+1], perm_tok, inv_pos; block 0 also writes load_out [E] and applies the bias
// update when those pointers are set.  Optionally gathers x rows into xp (bf16) and
// writes a bf16 copy of x into xb (fp32 x).  Blocks of 32 tokens when a chunk holds
// at most 128 tokens (a block recounts the earlier blocks of its chunk), else one
// block per chunk.
// `active` (nullable, [kMaxE + 1]) receives the ids of the experts with pairs and,
// at [kMaxE], their count.
// `balance` (nullable): block 0 writes the loads' balance statistics there.
// Expert ids outside [0, E) are skipped by the counting and the ranking and set the
// kDevCheck bit of the status word.
cudaError_t launch_scatter(const int32_t* idx, const int32_t* counts, int T, int k, int E,
                           int chunk_tokens, int32_t* offsets, int32_t* load_out, float* bias,
                           float gamma, long long tokens_times_k, int32_t* perm_tok,
                           int32_t* inv_pos, const void* x, int x_is_f32, int d, uint16_t* xp,
                           uint16_t* xb, cudaStream_t s, int32_t* active = nullptr,
                           moe_balance_t* balance = nullptr);
cudaError_t run_bounded_wait_selftest(unsigned long long limit_ns, int* gave_up, cudaStream_t s);
cudaError_t launch_ep_regroup(int world, int el, const int32_t* counts, int32_t* perm, int32_t* inv,
                              int32_t* offsets, cudaStream_t s);
cudaError_t launch_gather(const void* x, int x_is_f32, const int32_t* perm_tok, long long rows,
                          int d, uint16_t* xp, cudaStream_t s);
cudaError_t launch_to_bf16(const float* x, long long n, uint16_t* xb, cudaStream_t s);
// tokens_times_k < 0: the kernel takes the sum of `load` as the global T*k.  bias
// (nullable) is updated in place; balance (nullable) receives the loads' statistics.
cudaError_t launch_bias_update(int E, long long tokens_times_k, const int32_t* load,
                               float gamma, float* bias, cudaStream_t s,
                               moe_balance_t* balance = nullptr);
cudaError_t launch_combine(const uint16_t* y_perm, const uint16_t* shared_out,
                           const int32_t* inv_pos, const float* gate, const uint16_t* residual,
                           uint16_t* out, int T, int k, int d, cudaStream_t s);
cudaError_t launch_pack_gate_up(int G, int width, int d, int block, const uint16_t* wg,
                                const uint16_t* wu, uint16_t* wgu, cudaStream_t s);

// ---------------------------------------------------------------- grouped GEMM
enum EpiMode { EPI_SWIGLU = 0, EPI_STORE = 1, EPI_COMBINE = 2, EPI_STORE_F32 = 3, EPI_SWIGLU_BWD = 4 };

struct GemmOperandSet {
  const void* a;        // bf16 [a_rows][K]
  long long a_rows;
  const void* b;        // bf16 [groups * N][K]
  int groups;
  int N, K;
  void* out;            // bf16 output
  int ldo;
  int mode;             // EpiMode
  int rows;             // shared set: rows of the single group
  // MN-major operands (stored [K][M] / [groups * K][N], the M or N index contiguous),
  // read through the tensor cores' transpose bits: no transposed copies.  M, N must
  // be multiples of 128 there (each CTA's half of a 256-wide tile is whole 64-element
  // atoms), and a K-major A beside an MN-major operand needs K % 64 == 0.  An MN-major
  // A takes its M extent from `rows` and its K extent from K.
  int a_mn;
  int b_mn;
  // EPI_SWIGLU_BWD: the accumulator holds the gate/up pre-activations (a, b),
  // interleaved as for EPI_SWIGLU; dh [rows][N / 2] holds dL/dh on entry and receives
  // gate * h; out [rows][N] receives (da, db) in the accumulator's column order;
  // dgpart [rows][N / bn] (nullable) the per-tile partial sums of <dh, h>; gperm
  // [rows] (nullable = 1) is each row's gate.
  uint16_t* dh;
  const float* gperm;
  float* dgpart;
  // Shared set only: split K into ksplit equal parts (multiples of 64).  EPI_STORE: part
  // p writes out + p * part_stride elements and the caller sums the parts.  EPI_STORE_F32:
  // the parts are added into out in part order (launch_grouped_gemm's kdep).
  int ksplit;
  long long part_stride;
  // Non-zero: B is read once per use and not again soon (the routed experts' weights in
  // the forward), so its TMA copies carry an L2 evict-first policy and leave the cache
  // to the activations the launch and the next kernels read again.
  int b_stream;
};
// Column tile width the grouped GEMM uses for an operand set of this mode and N.
int gemm_tile_n(int mode, int N);
struct CombineInputs {
  const uint16_t* y_perm;
  const int32_t* inv_pos;
  const float* gate;
  const uint16_t* residual;
  int k;
};
// Runs up to two operand sets in one persistent launch: `routed` (E groups with
// rows from device `offsets`) and `shared` (one group).  Either may be disabled
// with a null `a`.
// max_pairs > 0 caps the number of 2-SM clusters (leaving SMs to concurrent work).
// kgroup_stride > 0 groups the routed set along K instead: offsets then holds the
// E + 1 K offsets (multiples of 64), `routed.rows` is every group's row count, and
// group g writes out + g * kgroup_stride (EPI_STORE_F32 for fp32 outputs).
// early: the caller guarantees that the offsets and both sets' B operands were
// complete before the previous kernel in the stream started (the launch then reads
// them before its dependency wait).
// chain (nullable): a third set over the same E groups and offsets whose A is the
// routed set's output (an EPI_SWIGLU set: chain->a == routed.out, chain->K ==
// routed.ldo); its tiles run after the others in the same launch, each once the
// routed tiles of its 256-row block have written their rows.  dep: one zeroed int32
// per routed 256-row block (max_routed_rows / 256 + E + 1 suffice), left non-zero.
// kdep: with an fp32 shared set split along K, one zeroed int32 per output tile of it.
cudaError_t launch_grouped_gemm(const GemmOperandSet& routed, const int32_t* offsets, int E,
                                const GemmOperandSet& shared, const CombineInputs& comb,
                                long long max_routed_rows, cudaStream_t s, int* bad_arg,
                                int max_pairs = 0, long long kgroup_stride = 0, int early = 0,
                                const GemmOperandSet* chain = nullptr, int32_t* dep = nullptr,
                                int32_t* kdep = nullptr);
// Number of co-resident 2-SM clusters of the grouped GEMM on the current device.
int gemm_max_pairs();

// ---------------------------------------------------------------- int4 serving
// TMA descriptor for a bf16 matrix [outer][inner] (row-major), box [box_outer][64],
// 128-byte swizzle.
bool make_tma_map_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                       uint32_t box_outer);
// Shared-expert projections for T <= kSkinnyMaxT tokens (weights in the MMA's M, tokens
// in N, K split over an 8-CTA cluster).  mode 0: w = gate/up [rows = 2F][K] interleaved
// in blocks of 128 -> out = h [T][ldo] (SwiGLU); mode 1: w = down [rows = d][K] -> out
// [T][ldo], plus comb's residual and gated routed rows when comb is given.
constexpr int kSkinnyMaxT = 64;
bool skinny_supported(int mode, int T, int rows, int K, int gate_block);
cudaError_t launch_skinny(int mode, const uint16_t* w, int rows, int K, const uint16_t* x, int T,
                          uint16_t* out, int ldo, const CombineInputs* comb, cudaStream_t s);
cudaError_t launch_quantize_int4(long long rows, int K, const uint16_t* w, uint8_t* q,
                                 uint16_t* scale, cudaStream_t s);
// `active` [kMaxE + 1]: ids of the experts with rows (ascending), count at [kMaxE].
// slot (nullable, [E]): expert e's weights sit at position slot[e] of wq / ws (a cache
// slot); else at e.
cudaError_t launch_int4_gate_up(const int32_t* active, const int32_t* offsets, const uint8_t* wq,
                                const uint16_t* ws, const uint16_t* xp, uint16_t* h, int d, int f,
                                int block, cudaStream_t s, const int32_t* slot = nullptr);
// Top-1 serving without the permutation (at most kDirectMaxPairs (token, expert)
// pairs): gate_up: h[p][f] from x[p / k]; down: y[p][d] from h[p]; p = t * k + j.
constexpr int kDirectMaxPairs = 64;

// Top-1 serving with at most kServeMaxPairs (token, expert) pairs in one persistent
// launch (serve.cu): router, selection, bias update, shared and int4 routed experts,
// combine.  bf16 tokens and int4 routed weights; x, W_r and the shared expert's
// weights 16-byte aligned; its shared memory (the CTA's weight slices, x, hs, h, the
// logits) at most kServeMaxSmem bytes.
constexpr int kServeMaxPairs = 8;
constexpr size_t kServeMaxSmem = 200 * 1024;
struct ServeArgs {
  const void* x;
  const float* w_router;
  const float* logit_offset;
  float* bias;
  const moe_weights_t* w;
  const void* residual;
  uint16_t* out;
  float* scores;
  int32_t* idx;
  float* gate;
  int32_t* load;
  moe_balance_t* balance;
  void* scratch;  // serve_fused_scratch_bytes(shape)
  uint16_t* hs;   // [T][F]
  uint16_t* h;    // [T*k][f]
  int update_bias;
  float gamma;
  // Expert cache (or null): the routed weights in w are its slots'; the launch plans
  // the step and copies the missing experts from cache_src first.
  const struct CacheView* cache_view;
  const struct CacheSegments* cache_src;
  int cache_slots;
  long long cache_expert_bytes;
};
bool serve_fused_supported(const moe_shape_t* s, const void* x, const float* w_router, const moe_weights_t* w);
size_t serve_fused_scratch_bytes(const moe_shape_t* s);
cudaError_t launch_serve_fused(const moe_shape_t* s, const ServeArgs& a, cudaStream_t st);
cudaError_t launch_int4_direct(bool gate_up, const int32_t* idx, int pairs, int k, const uint8_t* wq,
                               const uint16_t* ws, const uint16_t* src, uint16_t* dst, int d, int f,
                               int block, cudaStream_t s, const int32_t* slot = nullptr);
// The permutation-free down projection with the combine in its epilogue (one expert
// per token, tensor-core shapes): out[t][n] = bf16(s_in[t][n] + gate[t] * y[t][n]),
// y the routed row in fp32, s_in the shared expert's output (residual included).
bool int4_direct_down_combine_supported(int d, int f, int k, const void* wq, const void* ws, const void* h);
cudaError_t launch_int4_direct_down_combine(const int32_t* idx, int pairs, const uint8_t* wq, const uint16_t* ws,
                                            const uint16_t* h, const uint16_t* s_in, const float* gate,
                                            uint16_t* out, int d, int f, cudaStream_t s, const int32_t* slot);
cudaError_t launch_int4_down(const int32_t* active, const int32_t* offsets, const uint8_t* wq,
                             const uint16_t* ws, const uint16_t* h, uint16_t* y, int d, int f,
                             cudaStream_t s, const int32_t* slot = nullptr);

// ---------------------------------------------------------------- backward
// Padded layout of the permuted rows (each expert's rows start on a multiple of 64):
// poff [E+1], inv_pad [pairs], gperm [q_max] (the gate of each padded row, 0 on
// padding), and the gathered rows xp, dp [q_max][d] (bf16; rows past poff[E] untouched).
cudaError_t launch_pad_gather(const int32_t* off, const int32_t* perm_tok, const int32_t* idx,
                              const int32_t* inv_pos, const float* gate, int E, long long pairs,
                              long long q_max, const uint16_t* x, const uint16_t* dout, int d,
                              int32_t* poff, int32_t* inv_pad, float* gperm, uint16_t* xp, uint16_t* dp,
                              cudaStream_t s);
// dgp: [Q][nparts] partial sums of dL/dgate per padded row (summed in order).
cudaError_t launch_router_bwd_dx(const int32_t* idx, const float* gate, const float* scores,
                                 const int32_t* inv_pad, const float* dgp, int nparts, const float* w_router,
                                 const uint16_t* dxp, const uint16_t* dxs, const uint16_t* dxs2,
                                 const uint16_t* dout, int T,
                                 int d, int E, int k, int renorm, float* dzp, float* dgate, uint16_t* dx,
                                 cudaStream_t s);
cudaError_t launch_router_wgrad(const float* dzp, const int32_t* off, const int32_t* poff,
                                const uint16_t* xp, int d, int E, float* dwr, cudaStream_t s);

// ---------------------------------------------------------------- attention block
// Causal grouped-query attention with per-head QK-norm (attention.cu); head width 128.
constexpr int kAttnHeadDim = 128;
// In place on qkv [rows][C] bf16: the first `heads` heads of 128 values of every row
// (the query and key heads) become u / sqrt(mean(u^2) + eps), rounded to bf16.
cudaError_t launch_qk_norm(uint16_t* qkv, long long rows, int C, int heads, float eps, cudaStream_t s);
// out [batch * seq][n_head * 128] bf16: softmax(q k^T / sqrt(128), causal) v per query
// head, with the key/value head h / (n_head / n_kv_head); qkv [batch * seq][C] holds the
// normalised query heads, the normalised key heads and the value heads, in that order.
cudaError_t launch_attention(const uint16_t* qkv, int batch, int seq, int n_head, int n_kv_head, uint16_t* out,
                             cudaStream_t s);

// ---------------------------------------------------------------- int4 expert cache
constexpr int kMaxCacheSlots = 256;
// Device state of the residency cache (least recently used over `slots` HBM slots).
struct CacheState {
  int step;       // serving steps planned so far (the stamp of the next one)
  int njobs;      // copies the last plan asked for
  int overflow;   // steps that used more experts than slots (not served)
  int pad;
  long long hits, misses, evictions, bytes;
};
// The four per-expert weight segments (gate/up codes and scales, down codes and
// scales): base pointers and bytes per expert.
struct CacheSegments {
  uint8_t* base[4];
  long long bytes[4];
};
struct CacheView {
  CacheState* state;
  int32_t* slot_expert;  // [slots] expert held, -1 empty
  int32_t* stamp;        // [slots] step of last use, -1 never
  int32_t* expert_slot;  // [E] slot, -1 absent
  int2* jobs;            // [max(E, slots)] (expert, slot) copies of the last plan
  CacheSegments slots_w; // the slots' weights, expert-major layout with slots as experts
};
// Plans one serving step from its routing result idx [pairs] and copies the missing
// experts from host_src (device-accessible host memory, expert-major) into the slots.
cudaError_t launch_cache_fetch(const int32_t* idx, int pairs, int E, int slots, const CacheView& v,
                               const CacheSegments& host_src, long long expert_bytes, cudaStream_t s);

}  // namespace moe
