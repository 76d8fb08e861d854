// C ABI of the MoE layer library: argument validation, workspace layout and the
// launch sequence of each call.  Declarations and their contracts: moe_gb300.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "internal.h"
#include "moe_gb300.h"

namespace moe {

__device__ int g_device_status;

int* device_status_ptr() {
  // One address per device, looked up with that device current.
  static int* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

int permute_chunk_tokens(int T, int E) {
  long long ct = kRouterTokens;
  while (((T + ct - 1) / ct) * (long long)E > kMaxCountEntries) ct *= 2;
  return (int)ct;
}

moe_status_t check_shape(const moe_shape_t* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 1 || s->d < 1 || s->E < 1 || s->k < 1 || s->f < 1 || s->F < 0)
    return MOE_ERR_INVALID_ARG;
  if (s->renorm != 0 && s->renorm != 1) return MOE_ERR_INVALID_ARG;
  if (s->x_dtype != MOE_X_BF16 && s->x_dtype != MOE_X_F32) return MOE_ERR_INVALID_ARG;
  if (s->w_format != MOE_W_BF16 && s->w_format != MOE_W_INT4_G32) return MOE_ERR_INVALID_ARG;
  if (s->T > (1 << 24) || s->d % 64 || s->d < 64 || s->d > 8192) return MOE_ERR_UNSUPPORTED;
  if (s->E > kMaxE || s->k > kMaxK || s->k > s->E) return MOE_ERR_UNSUPPORTED;
  if (s->f % 32 || s->f > 8192 || s->F % 32 || s->F > 16384) return MOE_ERR_UNSUPPORTED;
  if (s->w_format == MOE_W_INT4_G32 && (s->k != 1 || s->T > 256)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kAlign = 1024;

// Bump layout of a workspace: the same code sizes it (base = null) and carves it.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    off = (off + kAlign - 1) / kAlign * kAlign;
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- stage profiler
// A recorded call places up to kMarks named marks; stage i lasts from mark i to mark
// i + 1 and carries mark i's name (names are static strings).  Stages are summed by
// name over the recorded calls, forward and backward calls alike.
constexpr int kMarks = 10;
constexpr int kMaxNames = 16;
struct Profiler {
  std::mutex mu;
  bool on = false;
  int max_calls = 0, calls = 0, period = 1, nmarks = 0;
  long long seen = 0;
  std::vector<cudaEvent_t> ev;           // kMarks per recorded call
  std::vector<const char*> call_names;   // kMarks per recorded call (null = unused)
  const char* names[kMaxNames] = {};     // distinct stage names, first-seen order
  int name_calls[kMaxNames] = {};        // recorded calls that had the stage
} g_prof;

// Whether the call now starting is recorded (every `period`-th call while enabled).
bool prof_begin_call() {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  if (!g_prof.on || g_prof.calls >= g_prof.max_calls) return false;
  g_prof.nmarks = 0;
  return (g_prof.seen++ % g_prof.period) == 0;
}

// Next mark of a recorded call; name == nullptr ends the call.
void prof_mark(const char* name, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  if (!g_prof.on || g_prof.calls >= g_prof.max_calls) return;
  const size_t base = (size_t)g_prof.calls * kMarks;
  if (g_prof.nmarks < kMarks - 1 || (!name && g_prof.nmarks < kMarks)) {
    cudaEventRecord(g_prof.ev[base + g_prof.nmarks], s);
    g_prof.call_names[base + g_prof.nmarks] = name;
    ++g_prof.nmarks;
  }
  if (!name) {
    for (int i = g_prof.nmarks; i < kMarks; ++i) {  // unused slots repeat the end mark
      cudaEventRecord(g_prof.ev[base + i], s);
      g_prof.call_names[base + i] = nullptr;
    }
    ++g_prof.calls;
  }
}

// ---------------------------------------------------------------- fork / join
// moe_layer_fwd runs the routing on a second stream while the shared expert's
// gate/up GEMM (which needs only x) runs on the caller's stream.  One non-blocking
// stream and two events per device, created on first use and kept for the process;
// the mutex serialises enqueues that use them.
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_aux_mu;
AuxStream g_aux[64];

AuxStream* aux_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  AuxStream& a = g_aux[dev];
  if (!a.s) {
    if (cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming) != cudaSuccess) return nullptr;
  }
  return &a;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

size_t route_scratch_bytes(const moe_shape_t* s) {
  return router_tc_supported(s->T, s->E, s->x_dtype == MOE_X_F32) ? router_tc_scratch_bytes(s->E, s->d) : 0;
}

cudaError_t run_router(const RouterArgs& a, void* scratch, cudaStream_t s) {
  if (router_tc_supported(a.T, a.E, a.x_is_f32)) return launch_router_tc(a, scratch, s);
  return launch_router(a, s);
}

int chunks_of(const moe_shape_t* s, int* chunk_tokens) {
  *chunk_tokens = permute_chunk_tokens(s->T, s->E);
  return (s->T + *chunk_tokens - 1) / *chunk_tokens;
}

// Layer path: the tensor-core router counts per CTA of 128 tokens, so its chunks are
// at least 128 tokens (and still keep the count table within kMaxCountEntries).
int layer_chunks_of(const moe_shape_t* s, int* chunk_tokens) {
  int ct = permute_chunk_tokens(s->T, s->E);
  if (router_tc_supported(s->T, s->E, s->x_dtype == MOE_X_F32) && ct < 128) ct = 128;
  *chunk_tokens = ct;
  return (s->T + ct - 1) / ct;
}

struct PermuteWs {
  int32_t* counts;  // [chunks][E] pairs per (token chunk, expert)
};
PermuteWs carve_permute(Carver& c, const moe_shape_t* s) {
  int ct;
  const int chunks = chunks_of(s, &ct);
  PermuteWs w;
  w.counts = static_cast<int32_t*>(c.take(sizeof(int32_t) * chunks * s->E));
  return w;
}

struct FfnWs {
  uint16_t* xp;  // [T*k][d] gathered rows
  uint16_t* h;   // [T*k][f]
  uint16_t* hs;  // [T][F]
  uint16_t* xb;  // [T][d] bf16 copy of fp32 x
  int32_t* dep;  // [T*k / 256 + E + 1] per routed 256-row block: h rows published
};
FfnWs carve_ffn(Carver& c, const moe_shape_t* s) {
  const size_t Tk = (size_t)s->T * s->k;
  FfnWs w;
  w.xp = static_cast<uint16_t*>(c.take(2 * Tk * s->d));
  w.h = static_cast<uint16_t*>(c.take(2 * Tk * s->f));
  w.hs = s->F ? static_cast<uint16_t*>(c.take(2 * (size_t)s->T * s->F)) : nullptr;
  w.xb = s->x_dtype == MOE_X_F32 ? static_cast<uint16_t*>(c.take(2 * (size_t)s->T * s->d)) : nullptr;
  w.dep = static_cast<int32_t*>(c.take(4 * (Tk / 256 + s->E + 1)));
  return w;
}

struct LayerWs {
  void* router;
  int32_t* active;  // [kMaxE + 1] experts with rows, count last (int4 serving path)
  int32_t* idx;
  float* gate;
  int32_t* load;
  int32_t* offsets;
  int32_t* perm_tok;
  int32_t* inv_pos;
  uint16_t* y;
  uint16_t* s_out;  // [T][d] shared-expert output (before the combine)
  void* serve;      // fused serving scratch (int4 shapes with at most kServeMaxPairs pairs)
  void* small_router;  // logits and counter of the permutation-free path's router
  PermuteWs perm;
  FfnWs ffn;
};
LayerWs carve_layer(Carver& c, const moe_shape_t* s) {
  const size_t Tk = (size_t)s->T * s->k;
  LayerWs w;
  const size_t rb = route_scratch_bytes(s);
  w.router = rb ? c.take(rb) : nullptr;
  w.active = static_cast<int32_t*>(c.take(4 * (size_t)(kMaxE + 1)));
  w.idx = static_cast<int32_t*>(c.take(4 * Tk));
  w.gate = static_cast<float*>(c.take(4 * Tk));
  w.load = nullptr;  // placed after the count table below (one memset clears both)
  w.offsets = static_cast<int32_t*>(c.take(4 * (size_t)(s->E + 1)));
  w.perm_tok = static_cast<int32_t*>(c.take(4 * Tk));
  w.inv_pos = static_cast<int32_t*>(c.take(4 * Tk));
  w.y = static_cast<uint16_t*>(c.take(2 * Tk * s->d));
  w.s_out = s->F ? static_cast<uint16_t*>(c.take(2 * (size_t)s->T * s->d)) : nullptr;
  {
    int ct;
    const int chunks = layer_chunks_of(s, &ct);
    w.perm.counts = static_cast<int32_t*>(c.take(4 * ((size_t)chunks * s->E + s->E)));
    w.load = w.perm.counts + (size_t)chunks * s->E;
  }
  w.ffn = carve_ffn(c, s);
  // The fused serving launch's logits and sync words: carved from the shape alone, so
  // the workspace size does not depend on the device.
  w.serve = (s->w_format == MOE_W_INT4_G32 && s->x_dtype == MOE_X_BF16 && Tk <= (size_t)kServeMaxPairs)
                ? c.take(serve_fused_scratch_bytes(s))
                : nullptr;
  w.small_router = (s->w_format == MOE_W_INT4_G32 && s->x_dtype == MOE_X_BF16 && Tk <= (size_t)kDirectMaxPairs)
                       ? c.take(router_small_scratch_bytes(s->T, s->E))
                       : nullptr;
  return w;
}

// The grouped-GEMM launches of the bf16 expert FFN: gate/up for routed rows
// (xp -> h) and the shared expert (x -> hs) in one launch, both down projections
// (h -> y_perm, hs -> shared_out) in another; with `comb` set, the combine kernel
// then writes out = residual + shared_out + sum_j gate_j * y_perm[inv_pos_j].
moe_status_t run_ffn(const moe_shape_t* s, const void* x_bf16, const int32_t* offsets,
                     const moe_weights_t* w, const FfnWs& ws, uint16_t* y_perm,
                     uint16_t* shared_out, const CombineInputs* comb, uint16_t* out,
                     cudaStream_t st, bool mark = false, bool shared_gate_up_done = false) {
  const long long Tk = (long long)s->T * s->k;
  int bad = 0;
  CombineInputs none{};
  GemmOperandSet r1{ws.xp, Tk, w->w_gate_up, s->E, 2 * s->f, s->d, ws.h, s->f, EPI_SWIGLU, 0};
  r1.b_stream = 1;
  GemmOperandSet sd{};
  if (s->F)
    sd = GemmOperandSet{ws.hs, s->T, w->shared_down, 1, s->d, s->F, shared_out, s->d, EPI_STORE, s->T};
  // Each launch pairs tiles that stream expert weights (memory bound) with shared-
  // expert tiles (compute bound), interleaved.  With the shared gate/up already done,
  // the routed gate/up runs beside the shared down projection and the routed down
  // projection runs alone; otherwise the two gate/up sets share one launch and the
  // two down projections the next.
  GemmOperandSet s1{};
  if (s->F && !shared_gate_up_done)
    s1 = GemmOperandSet{x_bf16, s->T, w->shared_gate_up, 1, 2 * s->F, s->d, ws.hs, s->F,
                        EPI_SWIGLU, s->T};
  else if (s->F)
    s1 = sd;
  GemmOperandSet r2{ws.h, Tk, w->w_down, s->E, s->d, s->f, y_perm, s->d, EPI_STORE, 0};
  r2.b_stream = 1;
  // With the shared gate/up done, the routed down projection is chained into the same
  // launch (its tiles follow the others and start block by block as h is written;
  // ws.dep was zeroed by the caller); otherwise it shares a second launch with the
  // shared down projection.
  const bool chained = s->F && shared_gate_up_done;
  if (mark) prof_mark(chained ? "routed_ffn_shared_down" : "gemm_gate_up", st);
  cudaError_t e = launch_grouped_gemm(r1, offsets, s->E, s1, none, Tk, st, &bad, 0, 0, 0,
                                      chained ? &r2 : nullptr, chained ? ws.dep : nullptr);
  if (bad) return MOE_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  if (!chained) {
    GemmOperandSet s2{};
    if (s->F && !shared_gate_up_done) s2 = sd;
    if (mark) prof_mark(shared_gate_up_done ? "routed_down" : "gemm_down", st);
    // The offsets come from before the gate/up launch and B is weights: the down launch
    // may start its tile table and weight copies before its dependency wait.
    e = launch_grouped_gemm(r2, offsets, s->E, s2, none, Tk, st, &bad, 0, 0, /*early=*/1);
    if (bad) return MOE_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (comb) {
    if (mark) prof_mark("combine", st);
    e = launch_combine(y_perm, s->F ? shared_out : nullptr, comb->inv_pos, comb->gate,
                       comb->residual, out, s->T, s->k, s->d, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Top-1 serving path with int4 routed experts: the shared expert's gate/up on the
// tensor cores, the routed experts' gate/up and down on the int4 dequantising warps
// (active experts only), then the shared down projection whose epilogue adds the
// gated routed rows (and the residual) and writes `out`.
// A few tokens: the shared expert streams its weights over 8-CTA clusters (weights in
// the MMA's M, tokens in N) instead of the 256-token tiles of the grouped GEMM.
bool int4_skinny(const moe_shape_t* s) {
  return s->F && skinny_supported(0, s->T, 2 * s->F, s->d, moe_gate_up_block(s->F)) &&
         skinny_supported(1, s->T, s->d, s->F, 0);
}

// shared_gate_up_on: non-null when the shared gate/up already runs on another stream;
// its completion event, waited for before the shared down projection.
// direct: the routed experts work from idx without the permutation (h and y by pair).
// shared_on_aux: the second stream also ran the shared down projection into L.s_out
// (with the residual); the routed down projection then adds it in its epilogue.
moe_status_t run_ffn_int4(const moe_shape_t* s, const void* x_bf16, const LayerWs& L,
                          const moe_weights_t* w, const void* residual, uint16_t* out,
                          cudaStream_t st, bool mark, cudaEvent_t shared_gate_up_on = nullptr,
                          bool direct = false, const int32_t* slot = nullptr, bool shared_on_aux = false) {
  const long long Tk = (long long)s->T * s->k;
  int bad = 0;
  GemmOperandSet off{};
  CombineInputs none{};
  cudaError_t e = cudaSuccess;
  if (mark) prof_mark("gate_up_and_int4_experts", st);
  const bool skinny = int4_skinny(s);
  if (shared_gate_up_on) {
    // launched beside the routing
  } else if (skinny) {
    e = launch_skinny(0, static_cast<const uint16_t*>(w->shared_gate_up), 2 * s->F, s->d,
                      static_cast<const uint16_t*>(x_bf16), s->T, L.ffn.hs, s->F, nullptr, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else if (s->F) {
    GemmOperandSet s1{x_bf16, s->T, w->shared_gate_up, 1, 2 * s->F, s->d, L.ffn.hs, s->F,
                      EPI_SWIGLU, s->T};
    e = launch_grouped_gemm(off, L.offsets, s->E, s1, none, Tk, st, &bad);
    if (bad) return MOE_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (direct) {
    e = launch_int4_direct(true, L.idx, (int)Tk, s->k, static_cast<const uint8_t*>(w->w_gate_up),
                           static_cast<const uint16_t*>(w->scale_gate_up),
                           static_cast<const uint16_t*>(x_bf16), L.ffn.h, s->d, s->f,
                           moe_gate_up_block(s->f), st, slot);
    if (e == cudaSuccess && shared_on_aux) {
      if (mark) prof_mark("int4_down_combine", st);
      if (cudaStreamWaitEvent(st, shared_gate_up_on, 0) != cudaSuccess) return MOE_ERR_CUDA;
      e = launch_int4_direct_down_combine(L.idx, (int)Tk, static_cast<const uint8_t*>(w->w_down),
                                          static_cast<const uint16_t*>(w->scale_down), L.ffn.h, L.s_out, L.gate,
                                          out, s->d, s->f, st, slot);
      return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    if (e == cudaSuccess)
      e = launch_int4_direct(false, L.idx, (int)Tk, s->k, static_cast<const uint8_t*>(w->w_down),
                             static_cast<const uint16_t*>(w->scale_down), L.ffn.h, L.y, s->d, s->f,
                             moe_gate_up_block(s->f), st, slot);
  } else {
    e = launch_int4_gate_up(L.active, L.offsets, static_cast<const uint8_t*>(w->w_gate_up),
                            static_cast<const uint16_t*>(w->scale_gate_up), L.ffn.xp, L.ffn.h, s->d,
                            s->f, moe_gate_up_block(s->f), st, slot);
    if (e == cudaSuccess)
      e = launch_int4_down(L.active, L.offsets, static_cast<const uint8_t*>(w->w_down),
                           static_cast<const uint16_t*>(w->scale_down), L.ffn.h, L.y, s->d, s->f, st, slot);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (mark) prof_mark("shared_down_combine", st);
  CombineInputs comb{L.y, direct ? nullptr : L.inv_pos, L.gate,
                     static_cast<const uint16_t*>(residual), s->k};
  if (shared_gate_up_on && cudaStreamWaitEvent(st, shared_gate_up_on, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (skinny) {
    e = launch_skinny(1, static_cast<const uint16_t*>(w->shared_down), s->d, s->F, L.ffn.hs, s->T,
                      out, s->d, &comb, st);
  } else if (s->F) {
    GemmOperandSet s2{L.ffn.hs, s->T, w->shared_down, 1, s->d, s->F, out, s->d, EPI_COMBINE, s->T};
    e = launch_grouped_gemm(off, L.offsets, s->E, s2, comb, Tk, st, &bad);
    if (bad) return MOE_ERR_UNSUPPORTED;
  } else {
    // Without the permutation comb.inv_pos is null: the routed rows are indexed by pair.
    e = launch_combine(L.y, nullptr, comb.inv_pos, L.gate, comb.residual, out, s->T, s->k, s->d, st);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

bool weights_ok(const moe_shape_t* s, const moe_weights_t* w) {
  if (!w || !w->w_gate_up || !w->w_down) return false;
  if (!aligned16(w->w_gate_up) || !aligned16(w->w_down)) return false;
  if (s->w_format == MOE_W_INT4_G32) {
    if (!w->scale_gate_up || !w->scale_down) return false;
  }
  if (s->F) {
    if (!w->shared_gate_up || !w->shared_down) return false;
    if (!aligned16(w->shared_gate_up) || !aligned16(w->shared_down)) return false;
  }
  return true;
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return 2; }

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "device check failed";
  }
  return "unknown status";
}

int32_t moe_gate_up_block(int32_t width) {
  return width % 128 == 0 ? 128 : (width % 64 == 0 ? 64 : 32);
}

size_t moe_route_workspace_size(const moe_shape_t* shape) {
  if (check_shape(shape)) return 0;
  return route_scratch_bytes(shape);
}

moe_status_t moe_route(const moe_shape_t* shape, const void* x, const float* w_router,
                       const float* logit_offset, const float* bias, float* scores, int32_t* idx,
                       float* gate, int32_t* load, void* workspace, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st) return st;
  if (!x || !w_router || !bias || !idx || !gate || !load) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || (scores && !aligned16(scores)))
    return MOE_ERR_INVALID_ARG;
  const size_t need = route_scratch_bytes(shape);
  if (need && (!workspace || !aligned16(workspace))) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(load, 0, sizeof(int32_t) * shape->E, s) != cudaSuccess) return MOE_ERR_CUDA;
  RouterArgs a{x, shape->x_dtype == MOE_X_F32, w_router, logit_offset, bias, scores, idx, gate,
               load, nullptr, kRouterTokens, shape->T, shape->d, shape->E, shape->k, shape->renorm};
  return cuda_status(run_router(a, workspace, s));
}

size_t moe_permute_workspace_size(const moe_shape_t* shape) {
  if (check_shape(shape)) return 0;
  Carver c(nullptr);
  carve_permute(c, shape);
  return c.off;
}

moe_status_t moe_permute(const moe_shape_t* shape, const int32_t* idx, int32_t* offsets,
                         int32_t* perm_tok, int32_t* inv_pos, void* workspace, size_t ws_bytes,
                         void* stream) {
  moe_status_t st = check_shape(shape);
  if (st) return st;
  if (!idx || !offsets || !perm_tok || !inv_pos || !workspace) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_permute_workspace_size(shape)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carver c(workspace);
  PermuteWs w = carve_permute(c, shape);
  int ct;
  const int chunks = chunks_of(shape, &ct);
  if (cudaMemsetAsync(w.counts, 0, sizeof(int32_t) * chunks * shape->E, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaError_t e = launch_count(idx, shape->T, shape->k, shape->E, ct, w.counts, s);
  if (e == cudaSuccess)
    e = launch_scatter(idx, w.counts, shape->T, shape->k, shape->E, ct, offsets, nullptr, nullptr,
                       0.f, 0, perm_tok, inv_pos, nullptr, 0, shape->d, nullptr, nullptr, s);
  return cuda_status(e);
}

size_t moe_expert_ffn_workspace_size(const moe_shape_t* shape) {
  if (check_shape(shape)) return 0;
  Carver c(nullptr);
  carve_ffn(c, shape);
  return c.off;
}

moe_status_t moe_expert_ffn(const moe_shape_t* shape, const void* x, const int32_t* offsets,
                            const int32_t* perm_tok, const moe_weights_t* w, void* y_perm,
                            void* shared_out, void* workspace, size_t ws_bytes, void* stream) {
  moe_status_t st = check_shape(shape);
  if (st) return st;
  if (shape->w_format != MOE_W_BF16) return MOE_ERR_UNSUPPORTED;
  if (!x || !offsets || !perm_tok || !y_perm || !workspace || !weights_ok(shape, w))
    return MOE_ERR_INVALID_ARG;
  if ((shape->F != 0) != (shared_out != nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y_perm) || (shared_out && !aligned16(shared_out)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_expert_ffn_workspace_size(shape)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carver c(workspace);
  FfnWs ws = carve_ffn(c, shape);
  const long long Tk = (long long)shape->T * shape->k;
  const int xf = shape->x_dtype == MOE_X_F32;
  cudaError_t e = launch_gather(x, xf, perm_tok, Tk, shape->d, ws.xp, s);
  if (e == cudaSuccess && xf && shape->F)
    e = launch_to_bf16(static_cast<const float*>(x), (long long)shape->T * shape->d, ws.xb, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const void* xbf = xf ? ws.xb : x;
  return run_ffn(shape, xbf, offsets, w, ws, static_cast<uint16_t*>(y_perm),
                 static_cast<uint16_t*>(shared_out), nullptr, nullptr, s);
}

moe_status_t moe_selftest_bounded_wait(int64_t limit_ns, int32_t* gave_up, void* stream) {
  if (limit_ns < 1 || limit_ns > 1000000000LL || !gave_up) return MOE_ERR_INVALID_ARG;
  int g = -1;
  const cudaError_t e = run_bounded_wait_selftest((unsigned long long)limit_ns, &g, static_cast<cudaStream_t>(stream));
  *gave_up = g;
  return cuda_status(e);
}

moe_status_t moe_gather_rows(int64_t rows, int32_t d, const void* src, const int32_t* index, void* dst,
                             void* stream) {
  if (rows < 0 || d < 8 || d % 8 || d > 8192 || (rows > 0 && (!src || !index || !dst)))
    return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!aligned16(src) || !aligned16(dst))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_gather(src, 0, index, rows, d, static_cast<uint16_t*>(dst),
                                   static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_ep_regroup(int32_t world, int32_t experts_local, const int32_t* counts, int32_t* perm,
                            int32_t* inv, int32_t* offsets, void* stream) {
  if (world < 1 || experts_local < 1 || (long long)world * experts_local > 4096) return MOE_ERR_INVALID_ARG;
  if (!counts || !perm || !inv || !offsets) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_ep_regroup(world, experts_local, counts, perm, inv, offsets,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_combine(const moe_shape_t* shape, const void* y_perm, const void* shared_out,
                         const int32_t* inv_pos, const float* gate, const void* residual, void* out,
                         void* stream) {
  moe_status_t st = check_shape(shape);
  if (st) return st;
  if (!y_perm || !inv_pos || !gate || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out) || (shared_out && !aligned16(shared_out)) ||
      (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(static_cast<const uint16_t*>(y_perm),
                                    static_cast<const uint16_t*>(shared_out), inv_pos, gate,
                                    static_cast<const uint16_t*>(residual),
                                    static_cast<uint16_t*>(out), shape->T, shape->k, shape->d,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_bias_update(int32_t E, int64_t tokens_times_k, const int32_t* load, float gamma,
                             float* bias, void* stream) {
  if (E < 1 || E > kMaxE || (tokens_times_k < 0 && tokens_times_k != MOE_TK_FROM_LOAD) || !load || !bias)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_bias_update(E, tokens_times_k, load, gamma, bias, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_load_balance(int32_t E, const int32_t* load, moe_balance_t* balance, void* stream) {
  if (E < 1 || E > kMaxE || !load || !balance || (reinterpret_cast<uintptr_t>(balance) & 7u))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_bias_update(E, 0, load, 0.f, nullptr, static_cast<cudaStream_t>(stream), balance));
}

size_t moe_layer_workspace_size(const moe_shape_t* shape) {
  if (check_shape(shape)) return 0;
  Carver c(nullptr);
  carve_layer(c, shape);
  return c.off;
}

}  // extern "C"

namespace {

// An int4 expert cache taking part in a serving call: the slots' weights stand in for
// the routed weights, filled from host memory right after the routing.
struct CacheCtx {
  CacheView view;
  CacheSegments host_src;
  long long expert_bytes;
  int slots;
};

moe_status_t layer_fwd_impl(const moe_shape_t* shape, const void* x, const float* w_router,
                            const float* logit_offset, float* bias, float gamma, int32_t update_bias,
                            const moe_weights_t* w, const void* residual, void* out, const moe_debug_t* dbg,
                            void* workspace, size_t ws_bytes, void* stream, const CacheCtx* cache);

}  // namespace

extern "C" {

moe_status_t moe_layer_fwd(const moe_shape_t* shape, const void* x, const float* w_router,
                           const float* logit_offset, float* bias, float gamma,
                           int32_t update_bias, const moe_weights_t* w, const void* residual,
                           void* out, const moe_debug_t* dbg, void* workspace, size_t ws_bytes,
                           void* stream) {
  return layer_fwd_impl(shape, x, w_router, logit_offset, bias, gamma, update_bias, w, residual, out, dbg,
                        workspace, ws_bytes, stream, nullptr);
}

}  // extern "C"

namespace {

moe_status_t layer_fwd_impl(const moe_shape_t* shape, const void* x, const float* w_router,
                            const float* logit_offset, float* bias, float gamma, int32_t update_bias,
                            const moe_weights_t* w, const void* residual, void* out, const moe_debug_t* dbg,
                            void* workspace, size_t ws_bytes, void* stream, const CacheCtx* cache) {
  moe_status_t st = check_shape(shape);
  if (st) return st;
  const bool int4 = shape->w_format == MOE_W_INT4_G32;
  if (int4 && shape->x_dtype != MOE_X_BF16) return MOE_ERR_UNSUPPORTED;
  if (cache && !int4) return MOE_ERR_UNSUPPORTED;
  if (!x || !w_router || !bias || !out || !workspace || !weights_ok(shape, w))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(out) ||
      (residual && !aligned16(residual)) || !aligned16(workspace) ||
      (dbg && dbg->scores && !aligned16(dbg->scores)) ||
      (dbg && dbg->balance && (reinterpret_cast<uintptr_t>(dbg->balance) & 7u)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_layer_workspace_size(shape)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carver c(workspace);
  LayerWs L = carve_layer(c, shape);
  if (dbg) {
    if (dbg->idx) L.idx = dbg->idx;
    if (dbg->gate) L.gate = dbg->gate;
    if (dbg->load) L.load = dbg->load;
    if (dbg->offsets) L.offsets = dbg->offsets;
    if (dbg->perm_tok) L.perm_tok = dbg->perm_tok;
    if (dbg->inv_pos) L.inv_pos = dbg->inv_pos;
  }
  const int T = shape->T, E = shape->E, k = shape->k;
  int ct;
  const int chunks = layer_chunks_of(shape, &ct);
  const int xf = shape->x_dtype == MOE_X_F32;
  // Top-1 serving of at most kServeMaxPairs pairs: one persistent launch does the whole
  // layer, the expert cache's plan and fill included (not when the caller asks for the
  // permutation).
  if (int4 && L.serve && !(dbg && (dbg->offsets || dbg->perm_tok || dbg->inv_pos)) &&
      serve_fused_supported(shape, x, w_router, w)) {
    ServeArgs a{};
    a.x = x;
    a.w_router = w_router;
    a.logit_offset = logit_offset;
    a.bias = bias;
    a.w = w;
    a.residual = residual;
    a.out = static_cast<uint16_t*>(out);
    a.scores = dbg ? dbg->scores : nullptr;
    a.idx = L.idx;
    a.gate = L.gate;
    a.load = dbg ? dbg->load : nullptr;
    a.balance = dbg ? dbg->balance : nullptr;
    a.scratch = L.serve;
    a.hs = L.ffn.hs;
    a.h = L.ffn.h;
    a.update_bias = update_bias;
    a.gamma = gamma;
    if (cache) {
      a.cache_view = &cache->view;
      a.cache_src = &cache->host_src;
      a.cache_slots = cache->slots;
      a.cache_expert_bytes = cache->expert_bytes;
    }
    const bool prof = prof_begin_call();
    if (prof) prof_mark("serve_fused", s);
    const cudaError_t e = launch_serve_fused(shape, a, s);
    if (prof) prof_mark(nullptr, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }

  const bool prof = prof_begin_call();
  const bool tc = router_tc_supported(T, E, xf);
  // Fork: the shared expert's gate/up needs only x, so it runs on the caller's stream
  // (on most SMs) while the routing runs on a second stream (on the rest).
  const bool fork = !int4 && !xf && shape->F > 0 && T >= 1024;
  AuxStream* aux = nullptr;
  std::unique_lock<std::mutex> aux_lock(g_aux_mu, std::defer_lock);
  cudaStream_t rs = s;  // stream of the routing kernels
  if (fork) {
    aux_lock.lock();
    aux = aux_for_current_device();
    if (!aux) return MOE_ERR_CUDA;
    rs = aux->s;
    if (prof) prof_mark("shared_gate_up", s);
    if (cudaEventRecord(aux->fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(rs, aux->fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    const int pairs = gemm_max_pairs();
    const int reserve = pairs >= 32 ? pairs / 6 : 0;  // SMs left for the routing
    GemmOperandSet off{}, s1{x, T, w->shared_gate_up, 1, 2 * shape->F, shape->d, L.ffn.hs,
                             shape->F, EPI_SWIGLU, T};
    CombineInputs none{};
    int bad = 0;
    // Shared-only launch: no offsets, B is the shared expert's weights (early start).
    const cudaError_t eg = launch_grouped_gemm(off, L.offsets, E, s1, none, (long long)T * k, s,
                                               &bad, pairs - reserve, 0, /*early=*/1);
    if (bad) return MOE_ERR_UNSUPPORTED;
    if (eg != cudaSuccess) return MOE_ERR_CUDA;
    if (prof) prof_mark("routing_wait", s);
  } else if (prof) {
    prof_mark("router", s);
  }
  // Top-1 serving with few tokens: the shared expert's gate/up needs only x, so it
  // runs on the second stream beside the routing and the routed int4 experts.
  const bool int4_fork = int4 && !xf && int4_skinny(shape);
  // Top-1 serving with at most kDirectMaxPairs (token, expert) pairs skips the
  // permutation: the int4 experts read the routing result directly.  The loads are
  // then counted only when the bias update or the caller needs them.
  const bool direct = int4 && !xf && (long long)T * k <= kDirectMaxPairs &&
                      (shape->F == 0 || int4_skinny(shape)) &&
                      !(dbg && (dbg->offsets || dbg->perm_tok || dbg->inv_pos));
  // With one expert per token on the tensor-core kernels, the shared down projection
  // also runs on the second stream (into s_out, residual included) and the routed down
  // projection adds it: the shared expert leaves the critical path.
  const bool shared_on_aux = int4_fork && direct && k == 1 && L.s_out &&
                             int4_direct_down_combine_supported(shape->d, shape->f, k, w->w_down, w->scale_down,
                                                                L.ffn.h);
  if (int4_fork) {
    aux_lock.lock();
    aux = aux_for_current_device();
    if (!aux) return MOE_ERR_CUDA;
    if (cudaEventRecord(aux->fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(aux->s, aux->fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (launch_skinny(0, static_cast<const uint16_t*>(w->shared_gate_up), 2 * shape->F, shape->d,
                      static_cast<const uint16_t*>(x), T, L.ffn.hs, shape->F, nullptr,
                      aux->s) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (shared_on_aux) {
      CombineInputs res_only{nullptr, nullptr, nullptr, static_cast<const uint16_t*>(residual), k};
      if (launch_skinny(1, static_cast<const uint16_t*>(w->shared_down), shape->d, shape->F, L.ffn.hs, T, L.s_out,
                        shape->d, &res_only, aux->s) != cudaSuccess)
        return MOE_ERR_CUDA;
    }
    if (cudaEventRecord(aux->join, aux->s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  moe_balance_t* balance = dbg ? dbg->balance : nullptr;
  const bool need_load = update_bias || (dbg && dbg->load) || balance;
  if (direct) {
    RouterArgs ra{x, xf, w_router, logit_offset, bias, dbg ? dbg->scores : nullptr, L.idx, L.gate,
                  need_load ? L.load : nullptr, nullptr, ct, T, shape->d, E, k, shape->renorm};
    cudaError_t e = cudaSuccess;
    if (L.small_router && router_small_supported(ra)) {
      e = launch_router_small(ra, L.small_router, rs);  // writes the loads outright
    } else {
      if (need_load && cudaMemsetAsync(L.load, 0, sizeof(int32_t) * E, rs) != cudaSuccess)
        return MOE_ERR_CUDA;
      e = run_router(ra, L.router, rs);
    }
    if (e == cudaSuccess && (update_bias || balance))
      e = launch_bias_update(E, (long long)T * k, L.load, gamma, update_bias ? bias : nullptr, rs, balance);
    if (e == cudaSuccess && cache) {
      if (prof) prof_mark("cache_fetch", rs);
      e = launch_cache_fetch(L.idx, T * k, E, cache->slots, cache->view, cache->host_src,
                             cache->expert_bytes, rs);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const moe_status_t st2 = run_ffn_int4(shape, x, L, w, residual, static_cast<uint16_t*>(out), s,
                                          prof, int4_fork ? aux->join : nullptr, true,
                                          cache ? cache->view.expert_slot : nullptr, shared_on_aux);
    if (prof) prof_mark(nullptr, s);
    return st2;
  }
  // The tensor-core router's first kernel zeroes load and counts itself.
  if (!tc) {
    // The load vector follows the count table in the workspace: one memset for both,
    // unless the caller asked for the loads in a buffer of its own.
    const bool adjacent = L.load == L.perm.counts + (size_t)chunks * E;
    if (cudaMemsetAsync(L.perm.counts, 0, sizeof(int32_t) * ((size_t)chunks * E + (adjacent ? E : 0)),
                        rs) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (!adjacent && cudaMemsetAsync(L.load, 0, sizeof(int32_t) * E, rs) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  // The chained down projection's block counters (run_ffn after the fork).
  if (fork && cudaMemsetAsync(L.ffn.dep, 0, sizeof(int32_t) * ((size_t)T * k / 256 + E + 1), rs) !=
                  cudaSuccess)
    return MOE_ERR_CUDA;
  RouterArgs ra{x, xf, w_router, logit_offset, bias, dbg ? dbg->scores : nullptr, L.idx, L.gate,
                L.load, L.perm.counts, ct, T, shape->d, E, k, shape->renorm};
  cudaError_t e = run_router(ra, L.router, rs);
  if (prof && !fork) prof_mark("permute_gather", s);
  // The scatter launch derives the offsets from the counts and applies the bias
  // update (after the router has read the bias).
  if (e == cudaSuccess)
    e = launch_scatter(L.idx, L.perm.counts, T, k, E, ct, L.offsets, nullptr,
                       update_bias ? bias : nullptr, gamma, (long long)T * k, L.perm_tok,
                       L.inv_pos, x, xf, shape->d, L.ffn.xp, (xf && shape->F) ? L.ffn.xb : nullptr,
                       rs, int4 ? L.active : nullptr, balance);
  if (e == cudaSuccess && cache) {
    if (prof) prof_mark("cache_fetch", rs);
    e = launch_cache_fetch(L.idx, T * k, E, cache->slots, cache->view, cache->host_src, cache->expert_bytes,
                           rs);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (fork) {
    if (cudaEventRecord(aux->join, rs) != cudaSuccess ||
        cudaStreamWaitEvent(s, aux->join, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    aux_lock.unlock();
  }
  const void* xbf = xf ? L.ffn.xb : x;
  CombineInputs comb{L.y, L.inv_pos, L.gate, static_cast<const uint16_t*>(residual), k};
  const moe_status_t st2 =
      int4 ? run_ffn_int4(shape, xbf, L, w, residual, static_cast<uint16_t*>(out), s, prof,
                          int4_fork ? aux->join : nullptr, false, cache ? cache->view.expert_slot : nullptr)
           : run_ffn(shape, xbf, L.offsets, w, L.ffn, L.y, L.s_out, &comb,
                     static_cast<uint16_t*>(out), s, prof, fork);
  if (prof) prof_mark(nullptr, s);
  return st2;
}

// ---------------------------------------------------------------- int4 expert cache

// Bytes per expert of the four int4 weight segments: gate/up codes, gate/up scales,
// down codes, down scales.
long long cache_seg_bytes(const moe_shape_t* s, int i) {
  switch (i) {
    case 0: return 2LL * s->f * (s->d / 2);
    case 1: return 2LL * s->f * (s->d / 32) * 2;
    case 2: return (long long)s->d * (s->f / 2);
    default: return (long long)s->d * (s->f / 32) * 2;
  }
}

bool cache_shape_ok(const moe_shape_t* s, int slots) {
  if (check_shape(s) != MOE_OK || s->w_format != MOE_W_INT4_G32) return false;
  // Every step must fit: at least as many slots as a step can use distinct experts.
  if (slots < std::min<long long>(s->E, (long long)s->T * s->k) || slots > kMaxCacheSlots) return false;
  for (int i = 0; i < 4; ++i)
    if (cache_seg_bytes(s, i) % 16) return false;
  return true;
}

CacheView carve_cache(Carver& c, const moe_shape_t* s, int slots) {
  CacheView v;
  v.state = static_cast<CacheState*>(c.take(sizeof(CacheState)));
  v.slot_expert = static_cast<int32_t*>(c.take(4 * (size_t)slots));
  v.stamp = static_cast<int32_t*>(c.take(4 * (size_t)slots));
  v.expert_slot = static_cast<int32_t*>(c.take(4 * (size_t)s->E));
  v.jobs = static_cast<int2*>(c.take(8 * (size_t)std::max(s->E, slots)));
  for (int i = 0; i < 4; ++i) {
    v.slots_w.bytes[i] = cache_seg_bytes(s, i);
    v.slots_w.base[i] = static_cast<uint8_t*>(c.take((size_t)slots * cache_seg_bytes(s, i)));
  }
  return v;
}

void* align_up(void* p) {
  return reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(p) + kAlign - 1) / kAlign * kAlign);
}

// Device-accessible address of caller memory holding the experts (pinned or managed
// host memory, or device memory); null when the GPU cannot read it directly.
const void* device_view(const void* p) {
  cudaPointerAttributes a;
  if (!p || cudaPointerGetAttributes(&a, p) != cudaSuccess) return nullptr;
  if (a.type == cudaMemoryTypeUnregistered) return nullptr;
  return a.devicePointer;
}

}  // namespace

extern "C" {

size_t moe_expert_cache_bytes(const moe_shape_t* shape, int32_t slots) {
  if (!cache_shape_ok(shape, slots)) return 0;
  Carver c(nullptr);
  carve_cache(c, shape, slots);
  return c.off + kAlign;
}

moe_status_t moe_expert_cache_init(const moe_shape_t* shape, int32_t slots, void* cache, size_t bytes,
                                   void* stream) {
  if (!cache_shape_ok(shape, slots)) return MOE_ERR_UNSUPPORTED;
  if (!cache) return MOE_ERR_INVALID_ARG;
  if (bytes < moe_expert_cache_bytes(shape, slots)) return MOE_ERR_WORKSPACE;
  Carver c(align_up(cache));
  const CacheView v = carve_cache(c, shape, slots);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(v.state, 0, sizeof(CacheState), s) != cudaSuccess ||
      cudaMemsetAsync(v.slot_expert, 0xFF, 4 * (size_t)slots, s) != cudaSuccess ||
      cudaMemsetAsync(v.stamp, 0xFF, 4 * (size_t)slots, s) != cudaSuccess ||
      cudaMemsetAsync(v.expert_slot, 0xFF, 4 * (size_t)shape->E, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_expert_cache_read(const moe_shape_t* shape, int32_t slots, const void* cache,
                                   moe_cache_stats_t* stats, int32_t* slot_expert, int32_t* expert_slot,
                                   int32_t* stamp, void* stream) {
  if (!cache_shape_ok(shape, slots)) return MOE_ERR_UNSUPPORTED;
  if (!cache) return MOE_ERR_INVALID_ARG;
  Carver c(align_up(const_cast<void*>(cache)));
  const CacheView v = carve_cache(c, shape, slots);
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  if (stats) {
    CacheState h;
    if (cudaMemcpy(&h, v.state, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    stats->steps = h.step;
    stats->hits = h.hits;
    stats->misses = h.misses;
    stats->evictions = h.evictions;
    stats->bytes = h.bytes;
    stats->overflow = h.overflow;
  }
  if (slot_expert && cudaMemcpy(slot_expert, v.slot_expert, 4 * (size_t)slots, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (expert_slot && cudaMemcpy(expert_slot, v.expert_slot, 4 * (size_t)shape->E, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (stamp && cudaMemcpy(stamp, v.stamp, 4 * (size_t)slots, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_layer_fwd_cached(const moe_shape_t* shape, const void* x, const float* w_router,
                                  const float* logit_offset, float* bias, float gamma, int32_t update_bias,
                                  const moe_weights_t* host_w, int32_t slots, void* cache, size_t cache_bytes,
                                  const void* residual, void* out, const moe_debug_t* dbg, void* workspace,
                                  size_t ws_bytes, void* stream) {
  if (!cache_shape_ok(shape, slots)) return MOE_ERR_UNSUPPORTED;
  if (!host_w || !cache) return MOE_ERR_INVALID_ARG;
  if (cache_bytes < moe_expert_cache_bytes(shape, slots)) return MOE_ERR_WORKSPACE;
  const void* src[4] = {device_view(host_w->w_gate_up), device_view(host_w->scale_gate_up),
                        device_view(host_w->w_down), device_view(host_w->scale_down)};
  CacheCtx ctx;
  Carver c(align_up(cache));
  ctx.view = carve_cache(c, shape, slots);
  ctx.slots = slots;
  ctx.expert_bytes = 0;
  for (int i = 0; i < 4; ++i) {
    if (!src[i] || !aligned16(src[i])) return MOE_ERR_INVALID_ARG;
    ctx.host_src.base[i] = static_cast<uint8_t*>(const_cast<void*>(src[i]));
    ctx.host_src.bytes[i] = cache_seg_bytes(shape, i);
    ctx.expert_bytes += cache_seg_bytes(shape, i);
  }
  moe_weights_t wc = *host_w;  // the routed weights come from the slots; shared as given
  wc.w_gate_up = ctx.view.slots_w.base[0];
  wc.scale_gate_up = ctx.view.slots_w.base[1];
  wc.w_down = ctx.view.slots_w.base[2];
  wc.scale_down = ctx.view.slots_w.base[3];
  return layer_fwd_impl(shape, x, w_router, logit_offset, bias, gamma, update_bias, &wc, residual, out, dbg,
                        workspace, ws_bytes, stream, &ctx);
}

}  // extern "C"

// ---------------------------------------------------------------- layer backward

namespace {

moe_status_t check_bwd_shape(const moe_shape_t* s) {
  const moe_status_t st = check_shape(s);
  if (st != MOE_OK) return st;
  if (s->x_dtype != MOE_X_BF16 || s->w_format != MOE_W_BF16) return MOE_ERR_UNSUPPORTED;
  // MN-major operands of the backward GEMMs: whole 128-element halves of a tile.
  if (s->d % 128 || s->f % 128 || s->F % 128) return MOE_ERR_UNSUPPORTED;
  if ((long long)s->T * s->k + 63LL * s->E > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Rows of the padded permuted layout: every pair plus up to 63 padding rows per expert.
long long bwd_rows(const moe_shape_t* s) { return (long long)s->T * s->k + 63LL * s->E; }

// Column tiles of the routed dgrad-through-down GEMM: partial sums of dL/dgate per row.
int bwd_parts(const moe_shape_t* s) { return 2 * s->f / gemm_tile_n(EPI_SWIGLU_BWD, 2 * s->f); }

// The shared expert's input gradient dxs = (das, dbs) Sgu runs over K = 2F: with
// 2F >= 2048 its tiles are split into two K halves (a K = 4096 tile alone took four
// times a routed tile and left the launch's end to the pairs holding two of them);
// the router backward adds the halves.
int bwd_dxs_parts(const moe_shape_t* s) { return (s->F && 2 * s->F >= 2048 && (2 * s->F) % 128 == 0) ? 2 : 1; }

// The shared expert's down-projection weight gradient runs over K = T tokens in few
// output tiles ([d][F]: 32 for Nano, so most pairs had none and the launch ended with
// the K = 8192 tiles): split into up to four parts of >= 2048 tokens, added in order
// into the fp32 output.  The gate/up one ([2F][d], 64 tiles, one for most pairs) gains
// less from balance than the extra tiles and reductions cost, and is not split.
int bwd_wgrad_parts(const moe_shape_t* s) {
  int ks = std::min(4, s->T / 2048);
  while (ks > 1 && s->T % (64 * ks) != 0) --ks;
  return std::max(ks, 1);
}
// Output tiles of the shared down-projection weight gradient [d][F].
int bwd_wgrad_tiles_down(const moe_shape_t* s) {
  return s->F ? (s->d + 255) / 256 * (s->F / gemm_tile_n(EPI_STORE_F32, s->F)) : 0;
}


struct BwdWs {
  int32_t* poff;     // [E+1] padded expert offsets
  int32_t* inv_pad;  // [T*k] padded row of each pair
  float* gperm;      // [Q] gate of each padded row
  float* dgp;        // [Q][f / tile width] partial dL/dgate of each padded row
  float* dzp;        // [Q] dL/dlogit of each padded row
  uint16_t* xp;      // [Q][d] gathered tokens
  uint16_t* dp;      // [Q][d] gathered output gradients
  uint16_t* ab;      // [Q][2f] gradients of the gate/up pre-activations
  uint16_t* dh;      // [Q][f] dout Wd, then gate * h
  uint16_t* dxp;     // [Q][d] routed input gradient of each row
  uint16_t* abs;     // [T][2F] shared expert: as ab
  uint16_t* dhs;     // [T][F] as dh (gate 1)
  uint16_t* dxs;     // [bwd_dxs_parts][T][d] shared expert's input gradient (K parts)
  int32_t* kdep;     // per output tile of dS_down: its K parts added so far
};
BwdWs carve_bwd(Carver& c, const moe_shape_t* s) {
  const size_t Q = (size_t)bwd_rows(s), Tk = (size_t)s->T * s->k, T = (size_t)s->T;
  BwdWs w;
  w.poff = static_cast<int32_t*>(c.take(4 * (size_t)(s->E + 1)));
  w.inv_pad = static_cast<int32_t*>(c.take(4 * Tk));
  w.gperm = static_cast<float*>(c.take(4 * Q));
  w.dgp = static_cast<float*>(c.take(4 * Q * bwd_parts(s)));
  w.dzp = static_cast<float*>(c.take(4 * Q));
  w.xp = static_cast<uint16_t*>(c.take(2 * Q * s->d));
  w.dp = static_cast<uint16_t*>(c.take(2 * Q * s->d));
  w.ab = static_cast<uint16_t*>(c.take(2 * Q * 2 * s->f));
  w.dh = static_cast<uint16_t*>(c.take(2 * Q * s->f));
  w.dxp = static_cast<uint16_t*>(c.take(2 * Q * s->d));
  w.abs = s->F ? static_cast<uint16_t*>(c.take(2 * T * 2 * s->F)) : nullptr;
  w.dhs = s->F ? static_cast<uint16_t*>(c.take(2 * T * s->F)) : nullptr;
  w.dxs = s->F ? static_cast<uint16_t*>(c.take(2 * T * s->d * bwd_dxs_parts(s))) : nullptr;
  w.kdep = static_cast<int32_t*>(c.take(4 * (size_t)(bwd_wgrad_tiles_down(s) + 1)));
  return w;
}

}  // namespace

extern "C" {

size_t moe_layer_bwd_workspace_size(const moe_shape_t* shape) {
  if (check_bwd_shape(shape) != MOE_OK) return 0;
  Carver c(nullptr);
  carve_bwd(c, shape);
  return c.off + kAlign;
}

moe_status_t moe_layer_bwd(const moe_shape_t* shape, const void* x, const float* w_router,
                           const moe_weights_t* w, const moe_debug_t* saved, const void* dout,
                           int32_t residual, const moe_grads_t* g, void* workspace, size_t ws_bytes,
                           void* stream) {
  const moe_status_t st = check_bwd_shape(shape);
  if (st != MOE_OK) return st;
  if (!x || !w_router || !w || !saved || !dout || !g || !workspace) return MOE_ERR_INVALID_ARG;
  if (residual != 0 && residual != 1) return MOE_ERR_INVALID_ARG;
  if (!w->w_gate_up || !w->w_down || !saved->scores || !saved->idx || !saved->gate ||
      !saved->offsets || !saved->perm_tok || !saved->inv_pos || !g->dx || !g->dw_router ||
      !g->dw_gate_up || !g->dw_down)
    return MOE_ERR_INVALID_ARG;
  const bool has_shared = shape->F > 0;
  if (has_shared != (w->shared_gate_up && w->shared_down && g->ds_gate_up && g->ds_down))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w_router, w->w_gate_up, w->w_down, dout, g->dx, g->dw_router,
                        g->dw_gate_up, g->dw_down, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (has_shared && (!aligned16(w->shared_gate_up) || !aligned16(w->shared_down) ||
                     !aligned16(g->ds_gate_up) || !aligned16(g->ds_down)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_layer_bwd_workspace_size(shape)) return MOE_ERR_WORKSPACE;

  const int T = shape->T, d = shape->d, E = shape->E, k = shape->k, f = shape->f, F = shape->F;
  const long long P = (long long)T * k, Q = bwd_rows(shape);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(workspace) + kAlign - 1) / kAlign * kAlign);
  Carver c(base);
  const BwdWs b = carve_bwd(c, shape);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  const uint16_t* db = static_cast<const uint16_t*>(dout);
  int bad = 0;
  CombineInputs none{};
  cudaError_t e;
  const bool prof = prof_begin_call();
  if (prof) prof_mark("bwd_pad_gather", s);
  const int ksw = has_shared ? bwd_wgrad_parts(shape) : 1;
  if (ksw > 1 && cudaMemsetAsync(b.kdep, 0, 4 * (size_t)bwd_wgrad_tiles_down(shape), s) != cudaSuccess) {
    if (prof) prof_mark(nullptr, s);
    return MOE_ERR_CUDA;
  }

  // Padded permuted layout and the gathered tokens and output gradients.
  e = launch_pad_gather(saved->offsets, saved->perm_tok, saved->idx, saved->inv_pos, saved->gate, E, P, Q, xb,
                        db, d, b.poff, b.inv_pad, b.gperm, b.xp, b.dp, s);
  if (e != cudaSuccess) {
    if (prof) prof_mark(nullptr, s);
    return MOE_ERR_CUDA;
  }
  if (prof) prof_mark("bwd_dgrad_down", s);
  // (1) dh = dout Wd_e (B = the stored [d][f] weights, MN-major), dhs = dout Sd.
  {
    GemmOperandSet r{b.dp, Q, w->w_down, E, f, d, b.dh, f, EPI_STORE, 0, 0, 1};
    GemmOperandSet sh{};
    if (has_shared) sh = GemmOperandSet{dout, T, w->shared_down, 1, F, d, b.dhs, F, EPI_STORE, T, 0, 1};
    e = launch_grouped_gemm(r, b.poff, E, sh, none, Q, s, &bad);
  }
  if (prof && e == cudaSuccess) prof_mark("bwd_recompute_swiglu", s);
  // (2-3) Gate/up pre-activations recomputed on the tensor cores (xp Wgu_e^T, x Sgu^T)
  // with the SwiGLU backward in the epilogue: ab <- (da, db), dh <- gate * h,
  // dgp <- partial <dh, h> (= <dout, y>) per column tile.
  if (e == cudaSuccess) {
    GemmOperandSet r{b.xp, Q, w->w_gate_up, E, 2 * f, d, b.ab, 2 * f, EPI_SWIGLU_BWD, 0, 0, 0,
                     b.dh, b.gperm, b.dgp};
    GemmOperandSet sh{};
    if (has_shared)
      sh = GemmOperandSet{x, T, w->shared_gate_up, 1, 2 * F, d, b.abs, 2 * F, EPI_SWIGLU_BWD, T, 0, 0,
                          b.dhs, nullptr, nullptr};
    e = launch_grouped_gemm(r, b.poff, E, sh, none, Q, s, &bad, 0, 0, /*early=*/1);
  }
  if (prof && e == cudaSuccess) prof_mark("bwd_dgrad_gate_up", s);
  // (4) dxp = (da, db) Wgu_e (B = the stored [2f][d] weights, MN-major), dxs likewise.
  if (e == cudaSuccess) {
    GemmOperandSet r{b.ab, Q, w->w_gate_up, E, d, 2 * f, b.dxp, d, EPI_STORE, 0, 0, 1};
    GemmOperandSet sh{};
    if (has_shared)
      sh = GemmOperandSet{b.abs, T, w->shared_gate_up, 1, d, 2 * F, b.dxs, d, EPI_STORE, T, 0, 1,
                          nullptr, nullptr, nullptr, bwd_dxs_parts(shape), (long long)T * d};
    e = launch_grouped_gemm(r, b.poff, E, sh, none, Q, s, &bad, 0, 0, /*early=*/1);
  }
  if (prof && e == cudaSuccess) prof_mark("bwd_router_dx", s);
  // (5) Router backward and dx = sum of the pairs' rows + shared + router (+ dout).
  if (e == cudaSuccess)
    e = launch_router_bwd_dx(saved->idx, saved->gate, saved->scores, b.inv_pad, b.dgp, bwd_parts(shape),
                             w_router, b.dxp,
                             has_shared ? b.dxs : nullptr,
                             has_shared && bwd_dxs_parts(shape) > 1 ? b.dxs + (size_t)T * d : nullptr,
                             residual ? db : nullptr, T, d, E, k,
                             shape->renorm, b.dzp, g->dgate, static_cast<uint16_t*>(g->dx), s);
  if (prof && e == cudaSuccess) prof_mark("bwd_wgrad_down", s);
  // (6) dWd_e = dp^T (gate * h) over the expert's rows (K-grouped), dSd = dout^T hs.
  if (e == cudaSuccess) {
    GemmOperandSet r{b.dp, Q, b.dh, 1, f, (int)Q, g->dw_down, f, EPI_STORE_F32, d, 1, 1};
    GemmOperandSet sh{};
    if (has_shared)
      sh = GemmOperandSet{dout, T, b.dhs, 1, F, T, g->ds_down, F, EPI_STORE_F32, d, 1, 1,
                          nullptr, nullptr, nullptr, ksw, 0};
    e = launch_grouped_gemm(r, b.poff, E, sh, none, Q, s, &bad, 0, (long long)d * f, /*early=*/1, nullptr,
                            nullptr, b.kdep);
  }
  if (prof && e == cudaSuccess) prof_mark("bwd_wgrad_gate_up", s);
  // (7) dWgu_e = (da, db)^T xp (rows interleaved as w_gate_up), dSgu = (das, dbs)^T x.
  if (e == cudaSuccess) {
    GemmOperandSet r{b.ab, Q, b.xp, 1, d, (int)Q, g->dw_gate_up, d, EPI_STORE_F32, 2 * f, 1, 1};
    GemmOperandSet sh{};
    if (has_shared)
      sh = GemmOperandSet{b.abs, T, x, 1, d, T, g->ds_gate_up, d, EPI_STORE_F32, 2 * F, 1, 1};
    e = launch_grouped_gemm(r, b.poff, E, sh, none, Q, s, &bad, 0, (long long)2 * f * d, /*early=*/1);
  }
  if (prof && e == cudaSuccess) prof_mark("bwd_router_wgrad", s);
  // (8) dW_r[e] = sum over the expert's rows of dz * x.
  if (e == cudaSuccess) e = launch_router_wgrad(b.dzp, saved->offsets, b.poff, b.xp, d, E, g->dw_router, s);
  if (prof) prof_mark(nullptr, s);
  if (bad) return MOE_ERR_UNSUPPORTED;
  return cuda_status(e);
}

}  // extern "C"

extern "C" {

moe_status_t moe_pack_gate_up(int32_t G, int32_t width, int32_t d, const void* w_gate,
                              const void* w_up, void* w_gate_up, void* stream) {
  if (G < 1 || width < 32 || width % 32 || d < 8 || d % 8 || !w_gate || !w_up || !w_gate_up)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_gate_up)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_gate_up(G, width, d, moe_gate_up_block(width),
                                         static_cast<const uint16_t*>(w_gate),
                                         static_cast<const uint16_t*>(w_up),
                                         static_cast<uint16_t*>(w_gate_up),
                                         static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quantize_int4(int64_t rows, int32_t K, const void* w, void* q, void* scale,
                               void* stream) {
  if (rows < 1 || K < 32 || K % 32 || !w || !q || !scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_int4(rows, K, static_cast<const uint16_t*>(w),
                                          static_cast<uint8_t*>(q), static_cast<uint16_t*>(scale),
                                          static_cast<cudaStream_t>(stream)));
}

int32_t moe_profile_stage_count(void) { return kMaxNames; }

const char* moe_profile_stage_name(int32_t stage) {
  if (stage < 0 || stage >= kMaxNames) return "";
  const char* n = g_prof.names[stage];
  return n ? n : "";
}

int32_t moe_profile_stage_calls(int32_t stage) {
  if (stage < 0 || stage >= kMaxNames) return 0;
  return g_prof.name_calls[stage];
}

moe_status_t moe_profile_start(int32_t max_calls, int32_t period) {
  if (max_calls < 1 || max_calls > (1 << 20) || period < 1) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  for (cudaEvent_t ev : g_prof.ev) cudaEventDestroy(ev);
  g_prof.ev.assign((size_t)max_calls * kMarks, nullptr);
  g_prof.call_names.assign((size_t)max_calls * kMarks, nullptr);
  for (auto& ev : g_prof.ev)
    if (cudaEventCreate(&ev) != cudaSuccess) return MOE_ERR_CUDA;
  for (auto& n : g_prof.names) n = nullptr;
  for (auto& c : g_prof.name_calls) c = 0;
  g_prof.max_calls = max_calls;
  g_prof.calls = 0;
  g_prof.period = period;
  g_prof.seen = 0;
  g_prof.on = true;
  return MOE_OK;
}

moe_status_t moe_profile_stop(float* ms_per_stage, int32_t* calls) {
  if (!ms_per_stage || !calls) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.on = false;
  for (int i = 0; i < kMaxNames; ++i) ms_per_stage[i] = 0.f;
  *calls = g_prof.calls;
  for (int c = 0; c < g_prof.calls; ++c) {
    cudaEvent_t* ev = &g_prof.ev[(size_t)c * kMarks];
    const char* const* nm = &g_prof.call_names[(size_t)c * kMarks];
    if (cudaEventSynchronize(ev[kMarks - 1]) != cudaSuccess) return MOE_ERR_CUDA;
    for (int i = 0; i + 1 < kMarks; ++i) {
      if (!nm[i]) break;
      int slot = 0;
      while (slot < kMaxNames && g_prof.names[slot] && g_prof.names[slot] != nm[i]) ++slot;
      if (slot == kMaxNames) continue;  // more distinct stages than slots: not reported
      if (!g_prof.names[slot]) g_prof.names[slot] = nm[i];
      ++g_prof.name_calls[slot];
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, ev[i], ev[i + 1]) == cudaSuccess) ms_per_stage[slot] += ms;
    }
  }
  return MOE_OK;
}

moe_status_t moe_device_status(void* stream, int32_t* device_status) {
  if (!device_status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int* p = device_status_ptr();
  if (!p) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
  *device_status = (v & kDevTimeout) ? MOE_ERR_TIMEOUT : ((v & kDevCheck) ? MOE_ERR_DEVICE : MOE_OK);
  return MOE_OK;
}

moe_status_t moe_last_device_status(void* stream) {
  int32_t st = MOE_OK;
  const moe_status_t e = moe_device_status(stream, &st);
  return e != MOE_OK ? e : static_cast<moe_status_t>(st);
}

size_t moe_workspace_size(const moe_shape_t* shape) { return moe_layer_workspace_size(shape); }

}  // extern "C"

namespace {

moe_status_t check_attn(const moe_attn_shape_t* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->batch < 1 || s->seq < 1 || s->d < 1 || s->n_head < 1 || s->n_kv_head < 1 || !(s->eps > 0.f))
    return MOE_ERR_INVALID_ARG;
  if (s->head_dim != kAttnHeadDim || s->n_head % s->n_kv_head || s->n_head * kAttnHeadDim > 8192 ||
      s->d % 64 || s->d > 8192 || (long long)s->batch * s->seq > (1LL << 24))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

struct AttnWs {
  uint16_t* qkv;  // [T][C]
  uint16_t* o;    // [T][n_head * 128]
};
AttnWs carve_attn(Carver& c, const moe_attn_shape_t* s) {
  const size_t T = (size_t)s->batch * s->seq;
  AttnWs w;
  w.qkv = static_cast<uint16_t*>(c.take(2 * T * (size_t)(s->n_head + 2 * s->n_kv_head) * kAttnHeadDim));
  w.o = static_cast<uint16_t*>(c.take(2 * T * (size_t)s->n_head * kAttnHeadDim));
  return w;
}

}  // namespace

extern "C" {

size_t moe_attention_workspace_size(const moe_attn_shape_t* shape) {
  if (check_attn(shape)) return 0;
  Carver c(nullptr);
  carve_attn(c, shape);
  return c.off;
}

moe_status_t moe_attention_core(const moe_attn_shape_t* shape, const void* qkv, void* o, void* stream) {
  const moe_status_t st = check_attn(shape);
  if (st) return st;
  if (!qkv || !o || !aligned16(qkv) || !aligned16(o)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_attention(static_cast<const uint16_t*>(qkv), shape->batch, shape->seq, shape->n_head,
                                      shape->n_kv_head, static_cast<uint16_t*>(o), static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_attention_fwd(const moe_attn_shape_t* shape, const void* x, const void* w_qkv, const void* w_o,
                               int32_t residual, void* out, void* workspace, size_t ws_bytes, void* stream) {
  const moe_status_t st = check_attn(shape);
  if (st) return st;
  if (!x || !w_qkv || !w_o || !out || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(w_o) || !aligned16(out) || !aligned16(workspace))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_attention_workspace_size(shape)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carver c(workspace);
  const AttnWs w = carve_attn(c, shape);
  const int T = shape->batch * shape->seq, hd = kAttnHeadDim;
  const int C = (shape->n_head + 2 * shape->n_kv_head) * hd, HO = shape->n_head * hd;
  int bad = 0;
  CombineInputs none{};
  // qkv = x w_qkv^T on the tensor cores (one group over all tokens).
  const GemmOperandSet off{};
  const GemmOperandSet proj{x, T, w_qkv, 1, C, shape->d, w.qkv, C, EPI_STORE, T};
  cudaError_t e = launch_grouped_gemm(off, nullptr, 1, proj, none, 0, s, &bad);
  if (bad) return MOE_ERR_UNSUPPORTED;
  if (e == cudaSuccess) e = launch_qk_norm(w.qkv, T, C, shape->n_head + shape->n_kv_head, shape->eps, s);
  if (e == cudaSuccess) e = launch_attention(w.qkv, shape->batch, shape->seq, shape->n_head, shape->n_kv_head, w.o, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  // out = o w_o^T; with the residual, the projection goes to the q, k, v region (free
  // after the attention) and the combine kernel adds x (no routed rows: k = 0).
  uint16_t* proj_out = residual ? w.qkv : static_cast<uint16_t*>(out);
  const GemmOperandSet oproj{w.o, T, w_o, 1, shape->d, HO, proj_out, shape->d, EPI_STORE, T};
  e = launch_grouped_gemm(off, nullptr, 1, oproj, none, 0, s, &bad);
  if (bad) return MOE_ERR_UNSUPPORTED;
  if (e == cudaSuccess && residual)
    e = launch_combine(nullptr, proj_out, nullptr, nullptr, static_cast<const uint16_t*>(x),
                       static_cast<uint16_t*>(out), T, 0, shape->d, s);
  return cuda_status(e);
}

}  // extern "C"
