/*
 * moe_gb300.h -- C ABI of the fine-grained MoE layer forward with aux-loss-free
 * bias balancing, for NVIDIA GB300 (sm_103a).
 *
 * Method source: "Una carrera de relevos con GPUs alquiladas entrenó el MoE de 2.7B
 * de NanoColibri por $200" (the same article in Chinese and Arabic), called "the
 * relay article" below.
 *   - opening section, architecture paragraph: hidden width 1024, 64 routed experts
 *     of width 512 with top-2 routing, one always-resident shared expert of width
 *     2048, a sigmoid-plus-bias router, and DeepSeek-V3 load balancing that moves
 *     each layer's expert bias by gamma times sign(target - load);
 *   - section "Entrenamiento por relevos", top-2 paragraph: gates are the scores
 *     renormalised over the winners (at top_k = 1 the weight is the constant 1);
 *     serving runs one expert per token;
 *   - opening section, second paragraph: experts stored in an int4 container.
 * Readings where the article is silent: SwiGLU experts (gate, up, down); ties in
 * the selection key go to the lower expert index; target load = T*k/E with
 * sign(0) = 0; the bias selects experts but never enters the gates; the shared
 * expert is added with weight 1.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates or frees device memory.  Row-major layouts; every pointer
 *     must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work; none synchronises the host except
 *     moe_device_status().
 *   - Host-side validation happens before any launch and returns
 *     MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE with nothing
 *     enqueued.  A failed launch returns MOE_ERR_CUDA.  Device-side conditions
 *     (a bounded wait that ran out) set a device status word read by
 *     moe_device_status(); kernels never trap.
 *   - bf16 tensors are passed as raw 16-bit patterns (void*), fp16 scales as
 *     uint16 patterns.
 */
#ifndef MOE_GB300_H_
#define MOE_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size */
  MOE_ERR_UNSUPPORTED = 2,  /* a size outside the supported envelope */
  MOE_ERR_WORKSPACE = 3,    /* workspace smaller than the *_workspace_size query */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed */
  MOE_ERR_TIMEOUT = 5,      /* device: a bounded wait gave up */
  MOE_ERR_DEVICE = 6        /* device: an in-kernel check failed */
} moe_status_t;

enum { MOE_X_BF16 = 0, MOE_X_F32 = 1 };          /* token activation dtype */
enum { MOE_W_BF16 = 0, MOE_W_INT4_G32 = 1 };     /* routed expert weight format */

/* Sizes of one MoE layer.  T tokens, hidden d, E routed experts of SwiGLU width f,
 * shared SwiGLU expert of width F (0 = none), top-k routing.
 * Supported envelope: 1 <= T <= 2^24, 64 <= d <= 8192 with d % 64 == 0,
 * 1 <= E <= 256, 1 <= k <= min(8, E), f % 32 == 0 (32 <= f <= 8192),
 * F % 32 == 0 (0 <= F <= 16384).  renorm: 1 = gates renormalised over the k
 * winners, 0 = gate is the raw sigmoid score.  MOE_W_INT4_G32 additionally needs
 * k == 1 and T <= 256 (the top-1 serving path). */
typedef struct {
  int32_t T, d, E, f, F, k;
  int32_t renorm;
  int32_t x_dtype;   /* MOE_X_BF16 | MOE_X_F32 */
  int32_t w_format;  /* MOE_W_BF16 | MOE_W_INT4_G32 */
} moe_shape_t;

/* Expert weights (device pointers).
 *   bf16 format:
 *     w_gate_up      [E][2f][d]  bf16, gate and up rows interleaved by
 *                                moe_pack_gate_up (block = moe_gate_up_block(f))
 *     w_down         [E][d][f]   bf16
 *   int4 format (moe_quantize_int4 of the bf16 tensors above):
 *     w_gate_up      [E][2f][d/2]  uint8, two's-complement nibbles, even index low
 *     scale_gate_up  [E][2f][d/32] fp16, groups of 32 along d
 *     w_down         [E][d][f/2]   uint8
 *     scale_down     [E][d][f/32]  fp16, groups of 32 along f
 *   shared expert (bf16 in every format; NULL when F == 0):
 *     shared_gate_up [2F][d] bf16, interleaved by moe_pack_gate_up (block for F)
 *     shared_down    [d][F]  bf16 */
typedef struct {
  const void* w_gate_up;
  const void* w_down;
  const void* scale_gate_up;
  const void* scale_down;
  const void* shared_gate_up;
  const void* shared_down;
} moe_weights_t;

/* Expert-balance statistics of one routing result, computed on the device from the
 * per-expert loads.  Relay article, section "Entrenamiento por relevos": the relay's
 * dashboard tracks expert balance, and the top-2 paragraph reports that the fraction of
 * dead experts stayed low.  This library's definitions (the pages give none): the mean
 * load is pairs / E; an expert is dead when its load is 0.  Each ratio is the fp32
 * value nearest to the exact rational (ties to even); 0 when pairs is 0. */
typedef struct {
  int64_t pairs;        /* sum of the loads: T*k (summed over replicas if the loads were) */
  int32_t max_load;     /* largest load */
  int32_t min_load;     /* smallest load */
  int32_t dead_experts; /* experts with load 0 */
  float max_over_mean;  /* max_load * E / pairs */
  float min_over_mean;  /* min_load * E / pairs */
  float dead_fraction;  /* dead_experts / E */
} moe_balance_t;

/* Optional intermediate outputs of moe_layer_fwd (any field may be NULL). */
typedef struct {
  float* scores;      /* [T][E] fp32 sigmoid scores */
  int32_t* idx;       /* [T][k] */
  float* gate;        /* [T][k] */
  int32_t* load;      /* [E] */
  int32_t* offsets;   /* [E+1] */
  int32_t* perm_tok;  /* [T*k] */
  int32_t* inv_pos;   /* [T][k] */
  moe_balance_t* balance;  /* one struct (device, 8-byte aligned): this forward's balance */
} moe_debug_t;

/* ABI version; bumped on any incompatible change. */
int32_t moe_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t status);

/* Rows per gate/up interleave block for an FFN of width `width` (f or F):
 * 128 if width % 128 == 0, else 64 if width % 64 == 0, else 32. */
int32_t moe_gate_up_block(int32_t width);

/* Router: relay article, architecture paragraph (sigmoid-plus-bias router, top-k)
 * and top-2 paragraph (renormalised gates).
 *   x            [T][d] bf16 or fp32 (shape->x_dtype)
 *   w_router     [E][d] fp32; logits carry fp32 accuracy: with bf16 tokens,
 *                T >= 128 and E in {16, 32, 48, 64, 80} the weight is split exactly
 *                into three bf16 parts and multiplied on the tensor cores with fp32
 *                accumulation (every product exact); otherwise fp32 FMA on CUDA cores
 *   logit_offset [E] fp32 added to every logit, or NULL (used by the skewed workload)
 *   bias         [E] fp32, added to the scores for selection only
 *   scores       [T][E] fp32 sigmoid scores, or NULL to skip writing them
 *   idx          [T][k] int32: the k experts of largest fl32(score + bias), by
 *                descending key, ties to the lower index
 *   gate         [T][k] fp32: score_j / sum of the k winners' scores (renorm),
 *                else score_j
 *   load         [E] int32: pairs routed to each expert (overwritten)
 *   workspace    moe_route_workspace_size(shape) bytes of scratch (may be NULL when
 *                that size is 0). */
size_t moe_route_workspace_size(const moe_shape_t* shape);
moe_status_t moe_route(const moe_shape_t* shape, const void* x, const float* w_router,
                       const float* logit_offset, const float* bias, float* scores,
                       int32_t* idx, float* gate, int32_t* load, void* workspace,
                       size_t ws_bytes, void* stream);

/* Stable counting-sort permutation of the (token, slot) pairs by expert.
 *   idx       [T][k] int32 from moe_route (values in [0, E), distinct per row)
 *   offsets   [E+1] int32: expert e owns rows [offsets[e], offsets[e+1])
 *   perm_tok  [T*k] int32: source token of each row; tokens ascend within a block
 *   inv_pos   [T][k] int32: row holding pair (t, j)
 *   workspace scratch of moe_permute_workspace_size(shape) bytes (no state kept). */
size_t moe_permute_workspace_size(const moe_shape_t* shape);
moe_status_t moe_permute(const moe_shape_t* shape, const int32_t* idx, int32_t* offsets,
                         int32_t* perm_tok, int32_t* inv_pos, void* workspace,
                         size_t ws_bytes, void* stream);

/* moe_permute without a workspace, for callers that cannot give the library device
 * memory: a plugin inside a framework that owns the device memory pool and hands out
 * no scratch, or a serving loop whose device-memory budget was fixed at start-up and
 * may not grow.  The pages have no counterpart to this call; it computes what
 * moe_permute computes and validates the shape as moe_permute does (same status for
 * the same shape).  Arguments as moe_permute (idx, offsets, perm_tok, inv_pos are
 * caller-owned).
 * Scratch: a library-owned static device array of 32768 int32 (128 KiB), held by
 * every GPU that loads the library until the process exits.  Every supported shape
 * fits (the chunking keeps the count table within 32768 entries); a shape that
 * would not fit returns MOE_ERR_UNSUPPORTED before any launch.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, with that
 * device current) and caches it: make that first call before any stream capture.
 * The cached address belongs to the device's context as it was at that call: after
 * cudaDeviceReset the library must not be used again in the process.
 * The call allocates and frees nothing.  All calls share the one array, which
 * keeps the previous call's contents (the call clears what must start at zero), so
 * calls that can overlap on the GPU -- on different streams, or from different
 * host threads -- race: serialise them.  An expert id outside [0, E) in idx is not
 * counted; it sets MOE_ERR_DEVICE in the device status word (moe_device_status) and
 * the outputs are then unspecified. */
moe_status_t moe_permute_noalloc(const moe_shape_t* shape, const int32_t* idx, int32_t* offsets,
                                 int32_t* perm_tok, int32_t* inv_pos, void* stream);

/* Grouped routed-expert FFN and the shared expert (bf16 weights).
 * Relay article, architecture paragraph (routed experts, always-resident shared
 * expert); SwiGLU is this library's reading: h = silu(x Wg^T) * (x Wu^T) stored as
 * bf16, y = h Wd^T; bf16 operands, fp32 accumulation on tcgen05 tensor cores.
 *   x           [T][d] token activations (bf16, or fp32 rounded to bf16 here)
 *   offsets, perm_tok from moe_permute
 *   y_perm      [T*k][d] bf16: routed output of each permuted row
 *   shared_out  [T][d] bf16: shared-expert output, NULL iff F == 0
 *   workspace   moe_expert_ffn_workspace_size(shape) bytes of scratch. */
size_t moe_expert_ffn_workspace_size(const moe_shape_t* shape);
moe_status_t moe_expert_ffn(const moe_shape_t* shape, const void* x, const int32_t* offsets,
                            const int32_t* perm_tok, const moe_weights_t* w, void* y_perm,
                            void* shared_out, void* workspace, size_t ws_bytes,
                            void* stream);

/* Combine: out[t] = residual[t] + shared[t] + sum_j gate[t][j] * y_perm[inv_pos[t][j]],
 * summed in fp32 and rounded once to bf16.  residual and shared_out may be NULL. */
moe_status_t moe_combine(const moe_shape_t* shape, const void* y_perm, const void* shared_out,
                         const int32_t* inv_pos, const float* gate, const void* residual,
                         void* out, void* stream);

/* Row gather: dst[r] = src[index[r]] for r < rows, rows of d bf16 values (d a
 * multiple of 8, both buffers 16-byte aligned, index values valid rows of src).
 * The expert-parallel path sends and receives rows with it (no host round trip). */
moe_status_t moe_gather_rows(int64_t rows, int32_t d, const void* src, const int32_t* index, void* dst,
                             void* stream);

/* Expert-parallel regrouping of received rows.  The experts are split over `world`
 * ranks in contiguous ranges of experts_local; a rank receives, source rank by
 * source rank, each source's rows for its local experts in the source's permuted
 * order (by local expert, then token).  Relay article, top-2 paragraph: expert
 * parallelism is where the leftover per-expert imbalance would show.
 *   counts   [world][experts_local] int32 device: rows source s sent for local expert e
 *   perm     [rows] int32 device: received row of each grouped row (grouped = by local
 *            expert, then source rank, then the source's order); rows = sum of counts
 *   inv      [rows] int32 device: grouped row of each received row
 *   offsets  [experts_local + 1] int32 device: local expert e owns grouped rows
 *            [offsets[e], offsets[e+1])
 * world * experts_local <= 4096; perm and inv must hold sum(counts) entries. */
moe_status_t moe_ep_regroup(int32_t world, int32_t experts_local, const int32_t* counts, int32_t* perm,
                            int32_t* inv, int32_t* offsets, void* stream);

/* Aux-loss-free bias update, relay article, architecture paragraph (DeepSeek-V3
 * recipe): bias[e] = fl32(bias[e] + gamma * sign(tokens_times_k - E * load[e])),
 * i.e. the sign of (target - load) with target = T*k/E and sign(0) = 0.
 * tokens_times_k is the GLOBAL T*k when `load` was summed over data-parallel
 * replicas (the only cross-replica exchange of the method), or MOE_TK_FROM_LOAD: the
 * kernel then sums `load` itself, which is the global T*k exactly (every token adds k
 * pairs), whatever the replicas' shard sizes, with no host round trip.  Other negative
 * values return MOE_ERR_INVALID_ARG.  In place on `bias`. */
#define MOE_TK_FROM_LOAD (-1)
moe_status_t moe_bias_update(int32_t E, int64_t tokens_times_k, const int32_t* load,
                             float gamma, float* bias, void* stream);

/* Expert-balance statistics (moe_balance_t) of `load` [E] int32 (device), written to
 * *balance (device, 8-byte aligned) by one block.  For loads summed over replicas as
 * well as a single forward's. */
moe_status_t moe_load_balance(int32_t E, const int32_t* load, moe_balance_t* balance, void* stream);

/* The whole layer: route, permute, gather, grouped expert FFN, shared expert,
 * combine and (if update_bias) the bias update, enqueued with no host
 * synchronisation.  With bf16 tokens, F > 0 and T >= 1024 the routing runs on a
 * library-owned second stream (one per device, created on first use, joined back
 * with events) while the shared expert's gate/up GEMM runs on `stream`; all work is
 * ordered before anything enqueued on `stream` after the call.  bias is read for selection and then updated in place.
 * residual (NULL or [T][d], same dtype as out) is added to the output.  For
 * MOE_W_INT4_G32 the routed experts run through the int4 dequant-in-GEMM path; with
 * 9 to 64 tokens (top-1, no permutation outputs asked for in dbg) they work straight
 * from the routing result and the shared expert runs on the same library-owned second
 * stream, joined back with an event.
 * Top-1 int4 serving of at most 8 tokens (bf16 tokens, d and f multiples of 256, the
 * weights 16-byte aligned, no permutation outputs asked for in dbg) runs as one
 * persistent launch with one CTA per SM whose CTAs wait on one another (section
 * "Entrenamiento por relevos", top-2 paragraph: one expert per token when serving):
 * it needs every SM free at once, and a wait that does not end within 2 s (other
 * kernels holding SMs that long) sets MOE_ERR_TIMEOUT in the device status word and
 * leaves the outputs unspecified.  The workspace needs no clearing between calls, but
 * two calls must not use the same workspace at the same time.
 *   out        [T][d] bf16
 *   dbg        NULL or intermediate outputs (see moe_debug_t)
 *   workspace  moe_layer_workspace_size(shape) bytes of scratch. */
size_t moe_layer_workspace_size(const moe_shape_t* shape);
moe_status_t moe_layer_fwd(const moe_shape_t* shape, const void* x, const float* w_router,
                           const float* logit_offset, float* bias, float gamma,
                           int32_t update_bias, const moe_weights_t* w, const void* residual,
                           void* out, const moe_debug_t* dbg, void* workspace,
                           size_t ws_bytes, void* stream);

/* Gradients written by moe_layer_bwd (device pointers, caller-owned, overwritten). */
typedef struct {
  void* dx;            /* [T][d] bf16: dL/dx */
  float* dw_router;    /* [E][d] */
  float* dw_gate_up;   /* [E][2f][d], rows interleaved as w_gate_up */
  float* dw_down;      /* [E][d][f] */
  float* ds_gate_up;   /* [2F][d], interleaved as shared_gate_up; NULL iff F == 0 */
  float* ds_down;      /* [d][F]; NULL iff F == 0 */
  float* dgate;        /* [T][k] dL/dgate of each pair, or NULL */
} moe_grads_t;

/* Backward of moe_layer_fwd (bf16 tokens and weights): gradients of a loss L given
 * dout = dL/dout, by the chain rule through the forward the relay article states
 * (architecture paragraph: sigmoid router, routed and shared SwiGLU experts; top-2
 * paragraph: gates renormalised over the winners).  The article says nothing about
 * the backward; this library's readings: the biased top-k selection is held fixed
 * (it is piecewise constant) and the bias gets no gradient (it moves only by the
 * balancing rule); with renormalised gates g_j = s_j / S, ds_j = (dg_j - sum_i dg_i
 * g_i) / S, else ds_j = dg_j; dz_j = ds_j s_j (1 - s_j) for the logit; the
 * gate/up pre-activations are recomputed from x (not stored by the forward).
 *   x, w_router, w  as given to moe_layer_fwd (shape->x_dtype = MOE_X_BF16,
 *                   shape->w_format = MOE_W_BF16)
 *   saved           the forward's scores, idx, gate, offsets, perm_tok and inv_pos
 *                   (moe_debug_t outputs of the same call; all required)
 *   dout            [T][d] bf16
 *   residual        1 if the forward added x to its output (dx then includes dout)
 *   grads           outputs; fp32 weight gradients (zero for an expert without
 *                   tokens), bf16 dx
 *   workspace       moe_layer_bwd_workspace_size(shape) bytes of scratch.
 * Supported: the moe_layer_fwd envelope with d, f and F multiples of 128.  Operands
 * are bf16 with fp32 accumulation; every GEMM runs on the tensor cores, reading the
 * weights and the permuted activations in their stored layouts (no transposed
 * copies); the expert weight gradients are K-grouped GEMMs over each expert's
 * tokens, padded to multiples of 64 rows in the workspace. */
size_t moe_layer_bwd_workspace_size(const moe_shape_t* shape);
moe_status_t moe_layer_bwd(const moe_shape_t* shape, const void* x, const float* w_router,
                           const moe_weights_t* w, const moe_debug_t* saved, const void* dout,
                           int32_t residual, const moe_grads_t* grads, void* workspace,
                           size_t ws_bytes, void* stream);

/* GPU-side residency cache of the int4 routed experts (top-1 serving).
 * Relay article, opening section, second paragraph: the int4 experts are streamed from
 * NVMe through an LRU cache under a memory budget; top-2 paragraph: the skew left after
 * balancing is what such a cache likes.  Here all experts' int4 weights stay in host
 * memory the GPU can read (pinned or managed), HBM holds `slots` of them, and
 * moe_layer_fwd_cached brings each step's experts in on the GPU with no host round
 * trip: after the routing one block plans the step and a grid copies the missing
 * experts over the CPU-GPU link into their slots (with at most 8 tokens, inside the
 * single serving launch of moe_layer_fwd, where a step whose experts are all resident
 * waits for no copy).  Policy (this library's reading of
 * LRU): the experts a step uses are the distinct entries of its routing result,
 * ascending; the resident ones are hits and their slots are stamped with the step
 * number first; then each missing expert, in ascending order, takes the slot with the
 * smallest stamp among the slots not stamped in this step (empty slots have stamp -1),
 * ties to the lowest slot, evicting its previous expert.
 * Shapes: w_format = MOE_W_INT4_G32 (k = 1, T <= 256) and
 * min(E, T*k) <= slots <= 256, so that every step fits.
 *   moe_expert_cache_bytes  device bytes of the cache (state + slots), 0 if unsupported
 *   moe_expert_cache_init   empties the cache (stream-ordered memsets)
 *   moe_expert_cache_read   synchronises `stream`, then copies the counters and (each
 *                           output nullable) slot_expert [slots] (-1 empty),
 *                           expert_slot [E] (-1 absent) and stamp [slots] to the host
 *   moe_layer_fwd_cached    moe_layer_fwd with the routed int4 weights (w_gate_up,
 *                           scale_gate_up, w_down, scale_down of host_w) in host memory,
 *                           layouts as in moe_weights_t; the shared expert's weights are
 *                           device memory as usual.  The output equals moe_layer_fwd's
 *                           with the same weights resident, bit for bit. */
typedef struct {
  int64_t steps, hits, misses, evictions, bytes, overflow;
} moe_cache_stats_t;

size_t moe_expert_cache_bytes(const moe_shape_t* shape, int32_t slots);
moe_status_t moe_expert_cache_init(const moe_shape_t* shape, int32_t slots, void* cache, size_t bytes,
                                   void* stream);
moe_status_t moe_expert_cache_read(const moe_shape_t* shape, int32_t slots, const void* cache,
                                   moe_cache_stats_t* stats, int32_t* slot_expert, int32_t* expert_slot,
                                   int32_t* stamp, void* stream);
moe_status_t moe_layer_fwd_cached(const moe_shape_t* shape, const void* x, const float* w_router,
                                  const float* logit_offset, float* bias, float gamma, int32_t update_bias,
                                  const moe_weights_t* host_w, int32_t slots, void* cache, size_t cache_bytes,
                                  const void* residual, void* out, const moe_debug_t* dbg, void* workspace,
                                  size_t ws_bytes, void* stream);

/* Attention block of the same model: relay article, opening section, architecture
 * paragraph (grouped-query attention with four query heads per key/value head, a
 * per-head QK-norm).  The article states nothing else; this library's readings: head
 * width 128; the QK-norm is an RMS normalisation of each head's 128 values of q and k
 * without a learned scale, u / sqrt(mean(u^2) + eps); scores q.k / sqrt(128), causal
 * within each sequence; no positional encoding; projections without biases.
 * Token rows are batch-major (row b * seq + s).
 *   x       [batch*seq][d] bf16
 *   w_qkv   [(n_head + 2 n_kv_head) * 128][d] bf16: the query, key and value
 *           projections stacked (query heads, then key heads, then value heads)
 *   w_o     [d][n_head * 128] bf16
 *   out     [batch*seq][d] bf16 = x (if residual) + o w_o^T, where o [batch*seq]
 *           [n_head * 128] is the attention output, rounded to bf16
 * The projections run on the tensor cores with fp32 accumulation; q, k, v are stored
 * as bf16 after the projection and again after the norm; the attention kernel keeps the
 * scores and the output accumulator in fp32 (TMEM) and the probabilities in bf16.
 * Supported: head_dim == 128, 1 <= n_kv_head <= n_head, n_head % n_kv_head == 0,
 * n_head * 128 <= 8192, d % 64 == 0 (64 <= d <= 8192), batch >= 1, seq >= 1,
 * batch * seq <= 2^24, eps > 0.
 * moe_attention_core computes only the attention: qkv [batch*seq][C] (C = (n_head +
 * 2 n_kv_head) * 128, the query and key heads already normalised) -> o. */
typedef struct {
  int32_t batch, seq, d, n_head, n_kv_head, head_dim;
  float eps;
} moe_attn_shape_t;

size_t moe_attention_workspace_size(const moe_attn_shape_t* shape);
moe_status_t moe_attention_fwd(const moe_attn_shape_t* shape, const void* x, const void* w_qkv, const void* w_o,
                               int32_t residual, void* out, void* workspace, size_t ws_bytes, void* stream);
moe_status_t moe_attention_core(const moe_attn_shape_t* shape, const void* qkv, void* o, void* stream);

/* Weight preparation, once per weight update and off the hot path: moe_pack_gate_up
 * for every bf16 layer, then moe_quantize_int4 on the packed gate/up and the down
 * weights for int4 serving.
 * moe_pack_gate_up: for each of G matrices, interleave w_gate [G][width][d] and
 * w_up [G][width][d] (bf16) into w_gate_up [G][2*width][d] in blocks of
 * b = moe_gate_up_block(width) rows: block i holds gate rows [i*b, (i+1)*b)
 * followed by up rows [i*b, (i+1)*b).
 * moe_quantize_int4: relay article, opening section (int4 container).  w [rows][K]
 * bf16 -> q [rows][K/2] uint8 (nibbles, even index low) and scale [rows][K/32]
 * fp16 with scale = fp16(fl32(max|w| / 7)) per group of 32 and
 * q = clamp(rint(fl32(w / scale)), -7, 7) (0 where scale is 0).  K % 32 == 0. */
moe_status_t moe_pack_gate_up(int32_t G, int32_t width, int32_t d, const void* w_gate,
                              const void* w_up, void* w_gate_up, void* stream);
moe_status_t moe_quantize_int4(int64_t rows, int32_t K, const void* w, void* q, void* scale,
                               void* stream);

/* Per-stage timing of moe_layer_fwd and moe_layer_bwd (profiling aid).  While
 * enabled, every recorded call places CUDA events on its stream between its stages;
 * after moe_profile_stop, stage slot i (0 <= i < moe_profile_stage_count()) holds the
 * summed milliseconds of the stage named moe_profile_stage_name(i) ("" for an unused
 * slot) over the recorded calls that had it, moe_profile_stage_calls(i) of them.
 * Stages are summed by name, so forward and backward calls can be recorded together.
 * On the large bf16 forward the stages are the shared-expert gate/up GEMM (while the
 * routing runs on a second stream), the remaining wait for the routing, the routed
 * gate/up GEMM, the down GEMM and the combine; the backward's are named after its
 * launches.  moe_profile_start(max_calls, period) records every period-th call, up to
 * max_calls recorded calls (host-side event objects only, no device memory; each
 * event adds about 2 us to the stream, hence the sampling period); moe_profile_stop
 * synchronises, writes ms_per_stage[moe_profile_stage_count()] and the number of
 * recorded calls to *calls, and disables recording. */
int32_t moe_profile_stage_count(void);
const char* moe_profile_stage_name(int32_t stage);
int32_t moe_profile_stage_calls(int32_t stage);
moe_status_t moe_profile_start(int32_t max_calls, int32_t period);
moe_status_t moe_profile_stop(float* ms_per_stage, int32_t* calls);

/* Synchronises `stream`, returns the device status word accumulated by this
 * library's kernels since the last call (MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE) in *device_status, and clears it. */
moe_status_t moe_device_status(void* stream, int32_t* device_status);

/* The same as one call: synchronises `stream`, reads and clears the device status word
 * and returns it (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE), or MOE_ERR_CUDA if the
 * read itself failed. */
moe_status_t moe_last_device_status(void* stream);

/* moe_layer_workspace_size under the short name: bytes of device workspace one
 * moe_layer_fwd call needs for this shape (0 for an unsupported shape). */
size_t moe_workspace_size(const moe_shape_t* shape);

/* Self-test of the failure path (for tests; it faults nothing).  One device thread
 * waits, through the helper the library's dependency waits use, for a counter that
 * nothing raises; after limit_ns nanoseconds of wall-clock time (1 .. 1e9) it gives up,
 * sets the timeout bit of the device status word (read and cleared by
 * moe_device_status, which then reports MOE_ERR_TIMEOUT) and returns.  *gave_up
 * (host) receives 1 when the wait gave up.  Synchronises `stream`. */
moe_status_t moe_selftest_bounded_wait(int64_t limit_ns, int32_t* gave_up, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H_ */
