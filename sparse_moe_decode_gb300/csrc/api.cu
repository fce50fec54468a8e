// api.cu -- the extern "C" entry points of libmoe_gb300.so: argument checks,
// workspace carving, and the order of kernel launches on the caller's stream.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "moe_gb300.h"

namespace moe {
namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status check_dims(const moe_dims *d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->num_experts != kE || d->top_k != kK || d->group != kG) return MOE_ERR_UNSUPPORTED;
  if (d->hidden <= 0 || d->hidden % kG || d->hidden > kMaxH) return MOE_ERR_UNSUPPORTED;
  if (d->expert_inter <= 0 || d->expert_inter % kG || d->expert_inter > kMaxI)
    return MOE_ERR_UNSUPPORTED;
  if (d->shared_inter < 0 || d->shared_inter % kG || d->shared_inter > kMaxI)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_weights(const moe_dims *d, const moe_weights *w, bool router, bool experts) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (router && (!w->w_router || !aligned(w->w_router, 16))) return MOE_ERR_INVALID_ARG;
  if (experts) {
    const void *p[4] = {w->w13_q, w->w13_s, w->w2_q, w->w2_s};
    for (const void *q : p)
      if (!q || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
  }
  if (d->shared_inter > 0) {
    if (router && (!w->w_shared_gate || !aligned(w->w_shared_gate, 16)))
      return MOE_ERR_INVALID_ARG;
    if (experts) {
      const void *p[4] = {w->ws13_q, w->ws13_s, w->ws2_q, w->ws2_s};
      for (const void *q : p)
        if (!q || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
    }
  }
  return MOE_OK;
}

bool ptr_ok(const void *p) { return p != nullptr && aligned(p, 16); }
bool opt_ok(const void *p) { return p == nullptr || aligned(p, 16); }

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// candidate selection: run length (the largest k), widest row, most lists
constexpr int kTopkRun = 16;
constexpr int kTopkMaxN = 1 << 24;
constexpr int kTopkMaxLists = 65536;

// Workspace carving for a call with T tokens; offsets are 256-byte aligned
// and grow monotonically with T, so a workspace sized for T_max serves every
// T <= T_max.
struct Layout {
  size_t status, logits, gate_logit, ids, weights, sgate;
  size_t counts, offsets, active, perm, slot_of;
  size_t h_routed, h_shared, h16, y, rpart, x16, xscale, hscale, xstage, ostage;
  size_t xs, acc, items, counters, total;
};

// Token count from which moe_block_forward runs the tcgen05 grouped GEMMs
// instead of the weight-streaming kernels: measured on GB300 at H = 2048,
// I = 512, the grouped GEMMs take 271 us at T = 128 and about as long down
// to T = 65, where the separate weight-streaming kernels took 761 us (and
// 1064 us at T = 127).
constexpr int kTcMinT = 65;

// Routes of moe_block_forward, chosen by sizes only (so that workspace sizes
// never depend on the device): the fused persistent decode kernel, the
// separate GEMV kernels, or the tcgen05 grouped GEMMs.  MOE_DECODE_ROUTE=gemv
// in the environment forces the GEMV kernels below kTcMinT (diagnostics).
enum Route { kRouteFused, kRouteGemv, kRouteTc };

bool force_gemv() {
  static int v = -1;
  if (v < 0) {
    const char *e = getenv("MOE_DECODE_ROUTE");
    v = (e && strcmp(e, "gemv") == 0) ? 1 : 0;
  }
  return v == 1;
}

Route route_of(const moe_dims *d, int T) {
  if (T >= kTcMinT) return kRouteTc;
  if (!force_gemv() && T <= kFusedMaxT && d->hidden <= kFusedMaxH && d->hidden % 512 == 0 &&
      d->expert_inter <= kFusedMaxI && d->shared_inter <= kFusedMaxI)
    return kRouteFused;
  return kRouteGemv;
}

Layout layout(const moe_dims *d, int T) {
  Layout L{};
  const size_t H = d->hidden, I = d->expert_inter, Is = d->shared_inter;
  const size_t t = static_cast<size_t>(T);
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += up256(bytes); return at; };
  L.status = take(256);
  L.logits = take(4 * t * kE);
  L.gate_logit = take(4 * t);
  L.ids = take(4 * t * kK);
  L.weights = take(4 * t * kK);
  L.sgate = take(4 * t);
  L.counts = take(4 * kE);
  L.offsets = take(4 * (kE + 1));
  L.active = take(4 * (kE + 1));
  L.perm = take(4 * t * kK);
  L.slot_of = take(4 * t * kK);
  L.h_routed = take(2 * t * kK * I);
  L.h_shared = take(2 * t * (Is ? Is : 1));
  const Route r = route_of(d, T);
  if (r == kRouteGemv || r == kRouteFused) L.y = take(4 * t * (kK + 1) * H);
  if (r == kRouteFused) {
    L.rpart = take(4 * t * 260 * (H / 512));
    L.h16 = take(2 * t * (kK * I + Is));
  }
  if (r == kRouteFused || r == kRouteTc) {
    L.x16 = take(2 * t * H);
    L.xscale = take(4 * t);
  }
  if (r == kRouteTc) {
    L.hscale = take(4 * t * (kK + 1));
  }
  L.xstage = take(2 * t * H);
  L.ostage = take(2 * t * H);
  if (r == kRouteTc) {
    L.xs = take(2 * t * kK * H);
    L.acc = take(4 * t * H);
    L.items = take(tc_items_bytes(T, static_cast<int>(I), static_cast<int>(Is),
                                  static_cast<int>(H)));
    L.counters = take(16);
  }
  L.total = o;
  return L;
}

template <typename P>
P *at(void *ws, size_t off) {
  return reinterpret_cast<P *>(static_cast<uint8_t *>(ws) + off);
}

Lists lists_in(void *ws, const Layout &L) {
  return Lists{at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.perm),
               at<int32_t>(ws, L.slot_of), at<int32_t>(ws, L.active)};
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                                  \
  do {                                                 \
    cudaError_t e_ = (expr);                           \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;        \
  } while (0)

moe_status check_ws(const moe_dims *d, int T, const void *ws, size_t ws_bytes, Layout &L) {
  if (!ws || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  L = layout(d, T);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// Kernel sequences of moe_block_forward: decode/verify route (GEMV kernels)
// and prefill route (tcgen05 grouped GEMMs).
const char *const kStageNames[] = {"router_gemv", "select_top8", "expert_lists",
                                   "gateup_swiglu", "down", "combine"};
constexpr int kStages = 6;
const char *const kFusedStageNames[] = {"decode_fused"};
const char *const kTcStageNames[] = {"router_tc", "select_top8", "lists_items",
                                     "scale_gather", "gateup_swiglu_tc", "h_scale",
                                     "down_combine_tc", "acc_to_bf16"};
constexpr int kTcStages = 8;

// Records `ev[i]` after kernel i-1 when profiling (ev[0] before the first).
struct Rec : StageRecorder {
  cudaEvent_t const *ev;
  cudaStream_t s;
  int i = 0;
  Rec(cudaEvent_t const *e, cudaStream_t st) : ev(e), s(st) {}
  cudaError_t operator()() override { return ev ? cudaEventRecord(ev[i++], s) : cudaSuccess; }
};

// The steps after the block in a decoder layer (moe_block_forward_residual):
// the residual added in the combine epilogue, then the next layer's input.
struct Residual {
  const moe_bf16 *resid;  // [T][H], added to the block's output before its rounding
  const moe_bf16 *gamma;  // [H]
  float eps;
  moe_bf16 *x_next;       // [T][H]
};

// The decode/verify path: router -> select -> lists -> gate|up -> down -> combine.
moe_status block_forward_device(const moe_dims *d, const moe_weights *w, const moe_bf16 *x,
                                int T, moe_bf16 *out, int32_t *ids_out, float *weights_out,
                                float *logits_out, float *gate_logit_out, void *ws,
                                const Layout &L, cudaStream_t s,
                                cudaEvent_t const *events = nullptr,
                                const Residual *res = nullptr) {
  const int H = d->hidden, I = d->expert_inter, Is = d->shared_inter;
  Rec rec{events, s};
  uint32_t *status = at<uint32_t>(ws, L.status);
  float *logits = logits_out ? logits_out : at<float>(ws, L.logits);
  float *glog = gate_logit_out ? gate_logit_out : at<float>(ws, L.gate_logit);
  int32_t *ids = ids_out ? ids_out : at<int32_t>(ws, L.ids);
  float *wts = weights_out ? weights_out : at<float>(ws, L.weights);
  float *sg = at<float>(ws, L.sgate);
  const moe_bf16 *wg = Is > 0 ? w->w_shared_gate : nullptr;
  const Lists lists = lists_in(ws, L);
  moe_bf16 *hr = at<moe_bf16>(ws, L.h_routed);
  moe_bf16 *hs = at<moe_bf16>(ws, L.h_shared);
  MOE_TRY(rec());
  const Route route = route_of(d, T);
  if (route == kRouteFused) {
    if (!fused_decode_supported(T, H, I, Is)) return MOE_ERR_UNSUPPORTED;
    unsigned *grid_bar = reinterpret_cast<unsigned *>(at<uint8_t>(ws, L.status) + 4);
    MOE_TRY(launch_decode_fused(x, T, H, I, Is, *w, at<uint16_t>(ws, L.x16),
                                at<float>(ws, L.xscale), at<float>(ws, L.rpart),
                                at<int32_t>(ws, L.ids), at<float>(ws, L.weights),
                                at<float>(ws, L.sgate), hr, hs, out, ids_out, weights_out,
                                logits_out, gate_logit_out, status, grid_bar, grid_bar + 1,
                                grid_bar + 2, at<float>(ws, L.y), at<uint16_t>(ws, L.h16),
                                grid_bar + 3, res ? res->resid : nullptr, s));
    MOE_TRY(rec());
    if (res) MOE_TRY(launch_rmsnorm(out, T, H, res->gamma, res->eps, res->x_next, s));
    return MOE_OK;
  }
  if (route == kRouteGemv) {
    MOE_TRY(launch_router_gemv(x, T, H, w->w_router, wg, logits, wg ? glog : nullptr, s));
    MOE_TRY(rec());
    MOE_TRY(launch_select(logits, T, kE, wg ? glog : nullptr, ids, wts, wg ? sg : nullptr,
                          status, s));
    MOE_TRY(rec());
    MOE_TRY(launch_lists(ids, T, lists, status, s));
    MOE_TRY(rec());
    float *y = at<float>(ws, L.y);
    MOE_TRY(launch_gateup_simt(x, T, H, I, Is, *w, lists, hr, hs, s));
    MOE_TRY(rec());
    MOE_TRY(launch_down_simt(T, H, I, Is, *w, lists, hr, hs, y, s));
    MOE_TRY(rec());
    MOE_TRY(launch_combine(T, H, y, wts, wg ? sg : nullptr, out, s, res ? res->resid : nullptr));
    MOE_TRY(rec());
    if (res) MOE_TRY(launch_rmsnorm(out, T, H, res->gamma, res->eps, res->x_next, s));
    return MOE_OK;
  }
  int4 *items = at<int4>(ws, L.items);
  int *counters = at<int>(ws, L.counters);
  MOE_TRY(launch_router_tc(x, T, H, w->w_router, logits, status, s, lists.counts));
  MOE_TRY(rec());
  MOE_TRY(launch_select(logits, T, kE, nullptr, ids, wts, wg ? sg : nullptr, status, s, x, wg,
                        H, glog, lists.counts));
  MOE_TRY(rec());
  MOE_TRY(launch_experts_tc(x, T, H, I, Is, *w, ids, lists, wts, wg ? sg : nullptr,
                            at<uint16_t>(ws, L.xs), at<uint16_t>(ws, L.x16),
                            at<float>(ws, L.xscale), at<float>(ws, L.hscale), hr, hs, at<float>(ws, L.acc), out, items,
                            counters, status, s, rec, nullptr, res ? res->resid : nullptr));
  if (res) MOE_TRY(launch_rmsnorm(out, T, H, res->gamma, res->eps, res->x_next, s));
  return MOE_OK;
}

}  // namespace

moe_status block_forward_check(const moe_dims *d, const moe_weights *w, const moe_bf16 *x, int T,
                               const moe_bf16 *out) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > kMaxT) return MOE_ERR_UNSUPPORTED;
  if ((st = check_weights(d, w, true, true)) != MOE_OK) return st;
  if (T > 0 && (!ptr_ok(x) || !ptr_ok(out))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null, misaligned or negative)";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch or copy failed";
  }
  return "unknown status";
}

size_t moe_workspace_bytes(const moe_dims *dims, int T_max) {
  if (check_dims(dims) != MOE_OK || T_max < 0 || T_max > kMaxT) return 0;
  if (T_max < 1) T_max = 1;
  // sizes grow with T inside a route; take the largest route boundary <= T_max
  size_t need = layout(dims, T_max).total;
  const int cands[2] = {kTcMinT - 1, kFusedMaxT};
  for (int c : cands)
    if (c < T_max) {
      const size_t v = layout(dims, c).total;
      if (v > need) need = v;
    }
  return need;
}

moe_status moe_router_logits(const moe_dims *dims, const moe_weights *w, const moe_bf16 *x,
                             int T, float *logits, float *shared_gate_logit, void *stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > kMaxT) return MOE_ERR_UNSUPPORTED;
  if ((st = check_weights(dims, w, true, false)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!ptr_ok(x) || !ptr_ok(logits) || !opt_ok(shared_gate_logit)) return MOE_ERR_INVALID_ARG;
  const moe_bf16 *wg = dims->shared_inter > 0 ? w->w_shared_gate : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T < kTcMinT)
    return cuda_status(launch_router_gemv(x, T, dims->hidden, w->w_router, wg, logits,
                                          wg ? shared_gate_logit : nullptr, s));
  MOE_TRY(launch_router_tc(x, T, dims->hidden, w->w_router, logits, nullptr, s));
  if (wg && shared_gate_logit)
    MOE_TRY(launch_router_gemv(x, T, dims->hidden, w->w_router, wg, logits, shared_gate_logit,
                               s, true));
  return MOE_OK;
}

moe_status moe_select_top8(const float *logits, int T, int ld, int E,
                           const float *shared_gate_logit, int32_t *ids, float *weights,
                           float *shared_gate, void *workspace, size_t ws_bytes, void *stream) {
  if (T < 0 || ld < E) return MOE_ERR_INVALID_ARG;
  if (E != kE || T > kMaxT) return MOE_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < 256) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  if (!ptr_ok(logits) || ld % 4 || !ptr_ok(ids) || !ptr_ok(weights) ||
      !opt_ok(shared_gate_logit) || !opt_ok(shared_gate))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_select(logits, T, ld, shared_gate_logit, ids, weights,
                                   shared_gate_logit ? shared_gate : nullptr,
                                   static_cast<uint32_t *>(workspace),
                                   static_cast<cudaStream_t>(stream)));
}

moe_status moe_build_expert_lists(const int32_t *ids, int T, int E, int32_t *counts,
                                  int32_t *offsets, int32_t *perm, void *workspace,
                                  size_t ws_bytes, void *stream) {
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (E != kE || T > kMaxT) return MOE_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  // status word + the active list
  if (ws_bytes < 256 + up256(4 * (kE + 1))) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  if (!ptr_ok(ids) || !ptr_ok(counts) || !ptr_ok(offsets) || !ptr_ok(perm))
    return MOE_ERR_INVALID_ARG;
  Lists L{counts, offsets, perm, nullptr, at<int32_t>(workspace, 256)};
  return cuda_status(launch_lists(ids, T, L, static_cast<uint32_t *>(workspace),
                                  static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_swiglu_w8(const moe_dims *dims, const moe_weights *w, const moe_bf16 *x,
                                int T, const int32_t *ids, float *y, void *workspace,
                                size_t ws_bytes, void *stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > kMaxT) return MOE_ERR_UNSUPPORTED;
  if ((st = check_weights(dims, w, false, true)) != MOE_OK) return st;
  Layout L;
  if ((st = check_ws(dims, T, workspace, ws_bytes, L)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!ptr_ok(x) || !ptr_ok(ids) || !ptr_ok(y)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = dims->hidden, I = dims->expert_inter, Is = dims->shared_inter;
  uint32_t *status = at<uint32_t>(workspace, L.status);
  const Lists lists = lists_in(workspace, L);
  moe_bf16 *hr = at<moe_bf16>(workspace, L.h_routed);
  moe_bf16 *hs = at<moe_bf16>(workspace, L.h_shared);
  if (Is == 0) {
    // slot K is defined as zeros when there is no shared expert
    MOE_TRY(cudaMemset2DAsync(y + static_cast<size_t>(kK) * H, sizeof(float) * (kK + 1) * H, 0,
                              sizeof(float) * H, T, s));
  }
  if (T >= kTcMinT) {
    // the tcgen05 grouped GEMMs of the block's prefill route, with the down
    // kernel storing every slot's unweighted output instead of combining
    Rec none{nullptr, s};
    MOE_TRY(launch_expert_counts(ids, T, lists.counts, status, s));
    MOE_TRY(launch_experts_tc(x, T, H, I, Is, *w, ids, lists, nullptr, nullptr,
                              at<uint16_t>(workspace, L.xs), at<uint16_t>(workspace, L.x16),
                              at<float>(workspace, L.xscale), at<float>(workspace, L.hscale), hr,
                              hs, nullptr, nullptr, at<int4>(workspace, L.items),
                              at<int>(workspace, L.counters), status, s, none, y));
    return MOE_OK;
  }
  MOE_TRY(launch_lists(ids, T, lists, status, s));
  MOE_TRY(launch_gateup_simt(x, T, H, I, Is, *w, lists, hr, hs, s));
  MOE_TRY(launch_down_simt(T, H, I, Is, *w, lists, hr, hs, y, s));
  return MOE_OK;
}

moe_status moe_combine(const moe_dims *dims, int T, const float *y, const float *weights,
                       const float *shared_gate, moe_bf16 *out, void *stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > kMaxT) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!ptr_ok(y) || !ptr_ok(weights) || !opt_ok(shared_gate) || !ptr_ok(out))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(T, dims->hidden, y, weights, shared_gate, out,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_block_forward(const moe_dims *dims, const moe_weights *w, const moe_bf16 *x,
                             int T, moe_bf16 *out, int32_t *ids_out, float *weights_out,
                             float *logits_out, float *gate_logit_out, void *workspace,
                             size_t ws_bytes, void *stream) {
  moe_status st = block_forward_check(dims, w, x, T, out);
  if (st != MOE_OK) return st;
  Layout L;
  if ((st = check_ws(dims, T, workspace, ws_bytes, L)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!opt_ok(ids_out) || !opt_ok(weights_out) || !opt_ok(logits_out) ||
      !opt_ok(gate_logit_out))
    return MOE_ERR_INVALID_ARG;
  return block_forward_device(dims, w, x, T, out, ids_out, weights_out, logits_out,
                              gate_logit_out, workspace, L, static_cast<cudaStream_t>(stream));
}

moe_status moe_block_forward_residual(const moe_dims *dims, const moe_weights *w,
                                      const moe_bf16 *x, int T, const moe_bf16 *resid_in,
                                      const moe_bf16 *gamma, float eps, moe_bf16 *resid_out,
                                      moe_bf16 *x_next, void *workspace, size_t ws_bytes,
                                      void *stream) {
  moe_status st = block_forward_check(dims, w, x, T, resid_out);
  if (st != MOE_OK) return st;
  Layout L;
  if ((st = check_ws(dims, T, workspace, ws_bytes, L)) != MOE_OK) return st;
  if (!(eps >= 0.0f) || eps > 3.0e38f) return MOE_ERR_INVALID_ARG;  // also NaN
  if (T == 0) return MOE_OK;
  if (!ptr_ok(resid_in) || !ptr_ok(gamma) || !ptr_ok(x_next)) return MOE_ERR_INVALID_ARG;
  // x_next is written after everything else has read the buffers, but it
  // must not overlap the residual rows it is computed from
  const uintptr_t bytes = sizeof(moe_bf16) * static_cast<uintptr_t>(T) * dims->hidden;
  const uintptr_t a = reinterpret_cast<uintptr_t>(x_next), b = reinterpret_cast<uintptr_t>(resid_out);
  const uintptr_t c = reinterpret_cast<uintptr_t>(resid_in);
  if ((a < b + bytes && b < a + bytes) || (a < c + bytes && c < a + bytes))
    return MOE_ERR_INVALID_ARG;
  // in place (resid_out == resid_in) or disjoint; a partial overlap would
  // let one row's sum read another row's result
  if (b != c && b < c + bytes && c < b + bytes) return MOE_ERR_INVALID_ARG;
  const Residual res{resid_in, gamma, eps, x_next};
  return block_forward_device(dims, w, x, T, resid_out, nullptr, nullptr, nullptr, nullptr,
                              workspace, L, static_cast<cudaStream_t>(stream), nullptr, &res);
}

moe_status moe_block_forward_host(const moe_dims *dims, const moe_weights *w,
                                  const moe_bf16 *x_host, int T, moe_bf16 *out_host,
                                  void *workspace, size_t ws_bytes, void *stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > kMaxT) return MOE_ERR_UNSUPPORTED;
  if ((st = check_weights(dims, w, true, true)) != MOE_OK) return st;
  Layout L;
  if ((st = check_ws(dims, T, workspace, ws_bytes, L)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = sizeof(moe_bf16) * static_cast<size_t>(T) * dims->hidden;
  moe_bf16 *xd = at<moe_bf16>(workspace, L.xstage);
  moe_bf16 *od = at<moe_bf16>(workspace, L.ostage);
  MOE_TRY(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s));
  st = block_forward_device(dims, w, xd, T, od, nullptr, nullptr, nullptr, nullptr, workspace,
                            L, s);
  if (st != MOE_OK) return st;
  MOE_TRY(cudaMemcpyAsync(out_host, od, bytes, cudaMemcpyDeviceToHost, s));
  MOE_TRY(cudaStreamSynchronize(s));
  return MOE_OK;
}

moe_status moe_block_forward_profiled(const moe_dims *dims, const moe_weights *w,
                                      const moe_bf16 *x, int T, moe_bf16 *out, void *workspace,
                                      size_t ws_bytes, void *const *events, int n_events,
                                      void *stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > kMaxT) return MOE_ERR_UNSUPPORTED;
  if ((st = check_weights(dims, w, true, true)) != MOE_OK) return st;
  Layout L;
  if ((st = check_ws(dims, T, workspace, ws_bytes, L)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  const int nk = moe_block_kernel_count(dims, T);
  if (!ptr_ok(x) || !ptr_ok(out) || !events || n_events < 1 + nk) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 1 + nk; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return block_forward_device(dims, w, x, T, out, nullptr, nullptr, nullptr, nullptr, workspace,
                              L, static_cast<cudaStream_t>(stream),
                              reinterpret_cast<cudaEvent_t const *>(events));
}

int moe_block_kernel_count(const moe_dims *dims, int T) {
  if (check_dims(dims) != MOE_OK || T < 1 || T > kMaxT) return 0;
  const Route r = route_of(dims, T);
  if (r == kRouteFused) return 1;
  if (r == kRouteGemv) return kStages;
  return kTcStages;
}

const char *moe_block_kernel_name(const moe_dims *dims, int T, int i) {
  const int n = moe_block_kernel_count(dims, T);
  if (i < 0 || i >= n) return nullptr;
  const Route r = route_of(dims, T);
  if (r == kRouteFused) return kFusedStageNames[i];
  if (r == kRouteGemv) return kStageNames[i];
  return kTcStageNames[i];
}

size_t moe_topk_workspace_bytes(int T, int N) {
  if (T < 0 || T > kMaxT || N < 1 || N > kTopkMaxN) return 0;
  return 256 + up256(static_cast<size_t>(T) * topk_chunks(N) * kTopkRun * sizeof(uint64_t));
}

moe_status moe_topk_candidates(const float *logits, int T, int ld, int N, int k, int32_t *ids,
                               float *values, void *workspace, size_t ws_bytes, void *stream) {
  if (T < 0 || N < 1 || ld < N || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kTopkRun || T > kMaxT || N > kTopkMaxN) return MOE_ERR_UNSUPPORTED;
  if (k > N) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_topk_workspace_bytes(T, N)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  if (!ptr_ok(logits) || ld % 4 || !ptr_ok(ids) || !ptr_ok(values)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_topk(logits, T, ld, N, k, ids, values,
                                 at<uint64_t>(workspace, 256), static_cast<uint32_t *>(workspace),
                                 static_cast<cudaStream_t>(stream)));
}

moe_status moe_topk_merge(const int32_t *ids, const float *values, int T, int n_lists, int k,
                          int32_t *ids_out, float *values_out, void *workspace, size_t ws_bytes,
                          void *stream) {
  if (T < 0 || n_lists < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kTopkRun || T > kMaxT || n_lists > kTopkMaxLists) return MOE_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < 256) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  if (!ptr_ok(ids) || !ptr_ok(values) || !ptr_ok(ids_out) || !ptr_ok(values_out))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_topk_merge(ids, values, T, n_lists, k, ids_out, values_out,
                                       static_cast<uint32_t *>(workspace),
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_read_status(const void *workspace, void *stream, uint32_t *bits) {
  if (!workspace || !aligned(workspace, 256) || !bits) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_TRY(cudaMemcpyAsync(bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
  MOE_TRY(cudaStreamSynchronize(s));
  return MOE_OK;
}

moe_status moe_clear_status(void *workspace, void *stream) {
  if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(cudaMemsetAsync(workspace, 0, 256, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

}  // extern "C"
