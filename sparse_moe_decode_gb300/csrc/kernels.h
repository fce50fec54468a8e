// kernels.h -- host-side launchers of the sm_103a kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

// Records a profiling event after each kernel launch (no-op when not profiling).
struct StageRecorder {
  virtual cudaError_t operator()() = 0;
};

// Token -> expert lists as the expert kernels consume them.
struct Lists {
  int32_t *counts;   // [E]
  int32_t *offsets;  // [E+1]
  int32_t *perm;     // [T*K] entries t*K+j sorted by (e, t, j)
  int32_t *slot_of;  // [T*K] inverse of perm (position of entry t*K+j), or -1
  int32_t *active;   // [1+E]: active[0] = number of active experts, then ids
};

// The host-side checks of a moe_block_forward call other than its
// workspace and optional outputs (dims, T, weights, x, out); no side effect.
moe_status block_forward_check(const moe_dims *d, const moe_weights *w, const moe_bf16 *x, int T,
                               const moe_bf16 *out);

// A1: router GEMV for any T (SIMT, fp32 accumulate).
cudaError_t launch_router_gemv(const moe_bf16 *x, int T, int H, const moe_bf16 *w_router,
                               const moe_bf16 *w_gate, float *logits, float *gate_logit,
                               cudaStream_t s, bool gate_only = false);

// A2: one warp per token.  With x and w_gate given, the shared gate's logit
// is computed here (written to gate_out when that is given) instead of read
// from gate_logit; counts (optional, zero on entry) receives per-expert token
// counts.
cudaError_t launch_select(const float *logits, int T, int ld, const float *gate_logit,
                          int32_t *ids, float *weights, float *sgate, uint32_t *status,
                          cudaStream_t s, const moe_bf16 *x = nullptr,
                          const moe_bf16 *w_gate = nullptr, int H = 0,
                          float *gate_out = nullptr, int32_t *counts = nullptr);

// Wide-row top-k candidates (topk.cu): runs holds T * topk_chunks(N) runs
// of 16 keys.  The merge takes caller lists of (id, value) pairs.
int topk_chunks(int N);
cudaError_t launch_topk(const float *logits, int T, int ld, int N, int k, int32_t *ids,
                        float *values, uint64_t *runs, uint32_t *status, cudaStream_t s);
cudaError_t launch_topk_merge(const int32_t *ids, const float *values, int T, int n_lists,
                              int k, int32_t *ids_out, float *values_out, uint32_t *status,
                              cudaStream_t s);

// A3: deterministic counting sort of the T*K entries (single CTA).
cudaError_t launch_lists(const int32_t *ids, int T, Lists L, uint32_t *status, cudaStream_t s);

// A4/A6: gate|up + SwiGLU, weight-streaming SIMT kernel.  h_routed [T*K][I]
// in list order, h_shared [T][Is].
cudaError_t launch_gateup_simt(const moe_bf16 *x, int T, int H, int I, int Is,
                               const moe_weights &w, Lists L, moe_bf16 *h_routed,
                               moe_bf16 *h_shared, cudaStream_t s);

// A5/A6: down projection into per-slot rows y [T][K+1][H] (fp32).
cudaError_t launch_down_simt(int T, int H, int I, int Is, const moe_weights &w, Lists L,
                             const moe_bf16 *h_routed, const moe_bf16 *h_shared, float *y,
                             cudaStream_t s);

// A7: out[t] = bf16(sum_j w[t][j] y[t][j] + sg[t] y[t][K] (+ resid[t])).
cudaError_t launch_combine(int T, int H, const float *y, const float *weights,
                           const float *sgate, moe_bf16 *out, cudaStream_t s,
                           const moe_bf16 *resid = nullptr);

// The next layer's input from the residual sum r [T][H] (bf16): x_next =
// bf16(r / sqrt(mean(r^2) + eps) * gamma), one warp per token, the sum of
// squares in a fixed order.
cudaError_t launch_rmsnorm(const moe_bf16 *r, int T, int H, const moe_bf16 *gamma, float eps,
                           moe_bf16 *x_next, cudaStream_t s);

// ---- decode-size T: the fused persistent kernel (decode_fused.cu)

constexpr int kFusedMaxT = 64;    // tokens
constexpr int kFusedMaxH = 2048;  // hidden (multiple of 512)
constexpr int kFusedMaxI = 2048;  // expert / shared intermediate

// Whether the fused kernel runs these sizes on the current device (one CTA
// per SM must fit, and the SMs must cover the Is / 8 shared gate|up units
// and the router rows in groups of 16 per 512-wide K-slice).
bool fused_decode_supported(int T, int H, int I, int Is);
size_t fused_smem_bytes();

// A1..A7 in one cooperative launch (resid, nullable: a residual [T][H] added
// to out before its rounding).  x16 [T][H] fp16 and xscale [T] (the
// tokens' scaled fp16 copies), rpart [T][H/512][260] fp32, sel_ids [T][K],
// sel_w [T][K], sel_sg [T], h_routed [T*K][I], h_shared [T][Is],
// y [T*K + T][H] fp32, h16 [T*K*I + T*Is] fp16, unit_claims, down_claims
// and h_wide (one word each) scratch; grid_bar is a 32-bit counter whose low 31 bits must be zero before the first launch
// (each grid barrier leaves them unchanged).
cudaError_t launch_decode_fused(const moe_bf16 *x, int T, int H, int I, int Is,
                                const moe_weights &w, uint16_t *x16, float *xscale,
                                float *rpart, int32_t *sel_ids, float *sel_w,
                                float *sel_sg, moe_bf16 *h_routed,
                                moe_bf16 *h_shared, moe_bf16 *out, int32_t *ids_out,
                                float *weights_out, float *logits_out, float *gate_logit_out,
                                uint32_t *status, unsigned *grid_bar, unsigned *unit_claims,
                                unsigned *down_claims, float *y, uint16_t *h16,
                                unsigned *h_wide, const moe_bf16 *resid, cudaStream_t s);

// ---- prefill-size T: tcgen05 GEMMs (tc_gemm.cu: router; tc_expert.cu: experts)

// 2-D row-major tensor [rows][cols] of `esize`-byte elements, box
// [box_rows][box_cols], 128-byte swizzle, zero fill out of bounds.
bool tc_make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
                 uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols);
// 3-D tensor of `esize`-byte elements: dims innermost first, strides (bytes)
// of dims 1 and 2, box innermost first; 128-byte swizzle, zero fill.
bool tc_make_map3(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
                  const uint64_t dims[3], const uint64_t strides[2], const uint32_t box[3]);
// Tensor of rank 1..5, dims innermost first, byte strides of dims 1..rank-1,
// box innermost first; no swizzle (rows land in shared memory as they lie in
// global memory), no fill.
bool tc_make_map_nd(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int rank,
                    const uint64_t *dims, const uint64_t *strides, const uint32_t *box);
int tc_sm_count();
// Budget of every bounded wait in the tcgen05 kernels (MOE_WAIT_BUDGET_NS, default 2 s).
unsigned long long tc_wait_budget_ns();

// Bytes of the work-item lists for T tokens.
size_t tc_items_bytes(int T, int I, int Is, int H);

// A1 router logits [T][E] as a tcgen05 GEMM (the gate row is left to the
// selection kernel or to the GEMV launcher with gate_only = true).  `status`
// may be NULL; zero_counts (optional, kE ints) is zeroed by the kernel.
cudaError_t launch_router_tc(const moe_bf16 *x, int T, int H, const moe_bf16 *w_router,
                             float *logits, uint32_t *status, cudaStream_t s,
                             int32_t *zero_counts = nullptr);

// A3..A7 for prefill-size T: builds the token -> expert lists of ids [T][K]
// into L (offsets, perm, slot_of from the per-expert counts that the
// selection left in L.counts; not active) with the work items,
// the tokens' scaled fp16 copies (xs16 [T*K][H] in list order, x16 [T][H],
// xscale [T]), runs gate|up + SwiGLU (h in bf16), converts h in place to
// per-row scaled fp16 (2^s of each row in hscale [T*K + T]), runs down + weighted combine into out_acc [T][H] (fp32, zeroed
// here), then rounds out_acc to bf16.  With y_slots given (per-slot mode),
// the down kernel instead stores each slot's unweighted fp32 output in
// y_slots [T][K+1][H] (the shared expert in slot K); out_acc, out, weights
// and sgate are then unused.
cudaError_t launch_experts_tc(const moe_bf16 *x, int T, int H, int I, int Is,
                              const moe_weights &w, const int32_t *ids, const Lists &L,
                              const float *weights,
                              const float *sgate, uint16_t *xs16, uint16_t *x16, float *xscale,
                              float *hscale,
                              moe_bf16 *h_routed, moe_bf16 *h_shared, float *out_acc,
                              moe_bf16 *out, int4 *items, int *counters, uint32_t *status,
                              cudaStream_t s, StageRecorder &rec, float *y_slots = nullptr,
                              const moe_bf16 *resid = nullptr);

// Per-expert entry counts of ids [T][K] into counts [E] (zeroed here); ids
// >= E set MOE_DEV_BAD_EXPERT.
cudaError_t launch_expert_counts(const int32_t *ids, int T, int32_t *counts, uint32_t *status,
                                 cudaStream_t s);

}  // namespace moe
