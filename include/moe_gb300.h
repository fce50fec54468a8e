/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) sparse-MoE block.
 *
 * The block is the MoE layer of a hybrid Qwen-style model at serving time:
 *   A1  router GEMV: 256 expert logits plus one shared-expert gate logit
 *       per token (the T x 257 rows of the S1/S2 router kernels in
 *       ninfer-windows PR #8, roofline paragraph);
 *   A2  per-token top-8 under a total order (the larger logit first, the
 *       lower expert id first among equal logits), softmax over the 8
 *       selected logits, sigmoid
 *       of the shared gate logit (PR #8, paragraphs on the warp merge network,
 *       sparse_moe_ranked_better and the untouched selector tail);
 *   A3  token -> expert lists (PR #8, the prefill select_count kernel);
 *   A4  int8 group-128 expert gate|up GEMV + SwiGLU, activations in bf16
 *       (ninfer 0.9.0 release notes, the W8 SwiGLU row of the route table;
 *       ninfer-tp2 v0.2.3, 16-bit activations in the SwiGLU and down
 *       projections);
 *   A5  int8 group-128 expert down projection;
 *   A6  the shared expert (A4 + A5 on every token) scaled by the gate;
 *   A7  weighted combine into a bf16 output row per token.
 * Beside the block: exact top-k (k <= 16) candidates over wide rows and the
 * exact merge of per-shard candidate lists (the drafter's candidate
 * selector: lucebox commit list; ninfer-tp2 v0.4.0, the vocabulary split
 * with an exact top-16 merge).
 *
 * Conventions (all entry points):
 *   - extern "C", no C++ or CUDA types: device pointers are plain pointers,
 *     a stream is passed as `void *` holding a cudaStream_t (NULL = legacy
 *     default stream).
 *   - Every call is asynchronous on that stream and never synchronises it,
 *     except moe_read_status and moe_block_forward_host (documented there).
 *   - The caller owns all memory.  Weights, inputs, outputs and the workspace
 *     are caller-allocated device buffers; the library never allocates,
 *     frees, or keeps a pointer after a call returns.
 *   - Host-detectable problems return a moe_status at once and launch nothing.
 *     A launch failure returns MOE_ERR_CUDA.
 *   - Problems only the device can see (non-finite logits, an expert id out
 *     of range, a bounded wait that ran out) set bits in a 32-bit status word
 *     at the start of the workspace; read it with moe_read_status.  The bits
 *     are sticky until moe_clear_status.
 *   - T == 0 is a no-op returning MOE_OK.
 *   - One workspace per concurrently running stream: two calls in flight on
 *     different streams must not share a workspace.
 *   - The first 256 bytes of a workspace (the device status word and the
 *     decode kernel's grid-barrier counter) must be zero before its first
 *     use, e.g. by moe_clear_status; the library keeps them consistent after
 *     that, except after a MOE_DEV_TIMEOUT, when moe_clear_status must be
 *     called again before the workspace is reused.
 *   - Supported shapes: num_experts == 256, top_k == 8, group == 128, hidden
 *     and expert_inter multiples of 128 (hidden <= 8192, expert_inter <= 2048),
 *     shared_inter 0 or a multiple of 128 (<= 2048), 1 <= T <= 65536.
 *     Anything else returns MOE_ERR_UNSUPPORTED; there is no fallback path.
 *   - Alignment: every device pointer 16-byte aligned, the workspace
 *     256-byte aligned; otherwise MOE_ERR_INVALID_ARG.
 *   - Layouts are row-major.  bf16 values are IEEE bfloat16 bit patterns.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

typedef uint16_t moe_bf16; /* IEEE bfloat16 bit pattern */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null / misaligned pointer, negative size      */
  MOE_ERR_UNSUPPORTED = 2, /* a shape outside the supported set above       */
  MOE_ERR_WORKSPACE = 3,   /* workspace smaller than moe_workspace_bytes    */
  MOE_ERR_CUDA = 4         /* a CUDA launch or copy failed                  */
} moe_status;

/* Device status bits, OR-ed into the status word at workspace + 0. */
#define MOE_DEV_NONFINITE 0x1u  /* a token's logits held NaN/inf (A2)       */
#define MOE_DEV_BAD_EXPERT 0x2u /* an expert id >= num_experts was given    */
#define MOE_DEV_TIMEOUT 0x4u    /* a bounded device-side wait gave up       */

typedef struct {
  int32_t hidden;       /* H                                              */
  int32_t num_experts;  /* E (256)                                        */
  int32_t top_k;        /* K (8)                                          */
  int32_t expert_inter; /* I: routed expert intermediate size             */
  int32_t shared_inter; /* Is: shared expert intermediate size, 0 = none  */
  int32_t group;        /* G (128): quantisation group along the K dim    */
} moe_dims;

/* All weights: device pointers, row-major, caller-owned, read-only.
 * Quantised matrices are int8 q with one bf16 scale per row per group of G
 * consecutive reduction elements: W[r][k] = q[r][k] * s[r][k / G]. */
typedef struct {
  const moe_bf16 *w_router;      /* [E][H]                                 */
  const moe_bf16 *w_shared_gate; /* [H]; NULL iff shared_inter == 0        */
  const int8_t *w13_q;           /* [E][2I][H]: rows 0..I-1 gate, I..2I-1 up */
  const moe_bf16 *w13_s;         /* [E][2I][H/G]                           */
  const int8_t *w2_q;            /* [E][H][I]                              */
  const moe_bf16 *w2_s;          /* [E][H][I/G]                            */
  const int8_t *ws13_q;          /* shared [2Is][H]  (NULL iff Is == 0)    */
  const moe_bf16 *ws13_s;        /* shared [2Is][H/G]                      */
  const int8_t *ws2_q;           /* shared [H][Is]                         */
  const moe_bf16 *ws2_s;         /* shared [H][Is/G]                       */
} moe_weights;

/* Bytes of workspace any call with T <= T_max needs (0 on bad dims). */
size_t moe_workspace_bytes(const moe_dims *dims, int T_max);

/* A1.  logits[t][e] = sum_k x[t][k] * w_router[e][k] (fp32 accumulate of
 * exact bf16 products) for e < E; shared_gate_logit[t] likewise with
 * w_shared_gate when both are non-NULL.  x [T][H] bf16, logits [T][E] fp32,
 * shared_gate_logit [T] fp32 (nullable). */
moe_status moe_router_logits(const moe_dims *dims, const moe_weights *w,
                             const moe_bf16 *x, int T, float *logits,
                             float *shared_gate_logit, void *stream);

/* A2.  For each token t (row t at logits + t*ld, ld >= E, E == 256):
 * ids[t][0..7] = the 8 best experts under "greater value wins, lower id
 * breaks a tie" (-0 == +0 is a tie) in rank order; weights[t][j] =
 * softmax over those 8 logits; shared_gate[t] = sigmoid(shared_gate_logit[t])
 * when both are non-NULL.  The ids and their order are bit-exact functions of
 * the fp32 inputs.  A row holding NaN/inf gets ids -1 and weights 0 and sets
 * MOE_DEV_NONFINITE.  The workspace holds only the status word here
 * (ws_bytes >= 256). */
moe_status moe_select_top8(const float *logits, int T, int ld, int E,
                           const float *shared_gate_logit, int32_t *ids,
                           float *weights, float *shared_gate, void *workspace,
                           size_t ws_bytes, void *stream);

/* A3 (exposed for testing).  counts[e] = number of entries (t, j) with
 * ids[t][j] == e; offsets[0..E] = exclusive scan of counts; perm[p] = t*8+j
 * for the entries sorted by (expert, t, j).  Negative ids are skipped; ids
 * >= E are skipped and set MOE_DEV_BAD_EXPERT.  ids [T][8]. */
moe_status moe_build_expert_lists(const int32_t *ids, int T, int E,
                                  int32_t *counts, int32_t *offsets,
                                  int32_t *perm, void *workspace,
                                  size_t ws_bytes, void *stream);

/* A4 + A5 + A6 without the combine.  For every token t and slot j < 8 with
 * e = ids[t][j] >= 0: h = bf16(silu(a_gate) * a_up) with a = W13_e x_t, and
 * y[t][j][:] = W2_e h (fp32).  Slot 8 holds the shared expert's output,
 * unscaled by its gate (zeros if shared_inter == 0).  Rows y[t][j] whose id
 * is negative are left unwritten; an id >= E sets MOE_DEV_BAD_EXPERT and
 * its row is left unwritten.  y [T][9][H] fp32.  Routes by T as
 * moe_block_forward does: weight-streaming kernels for T <= 64, the tcgen05
 * grouped GEMMs (each slot's output stored once, no atomics) from T = 65. */
moe_status moe_expert_swiglu_w8(const moe_dims *dims, const moe_weights *w,
                                const moe_bf16 *x, int T, const int32_t *ids,
                                float *y, void *workspace, size_t ws_bytes,
                                void *stream);

/* A7.  out[t][n] = bf16( sum_{j<8} weights[t][j] * y[t][j][n]
 *                        + shared_gate[t] * y[t][8][n] ), fp32 sums in slot
 * order, one round to nearest even.  Slots whose weight is exactly 0 are
 * skipped (their y rows need not be initialised).  shared_gate may be NULL
 * (no shared term).  y [T][9][H], weights [T][8], out [T][H]. */
moe_status moe_combine(const moe_dims *dims, int T, const float *y,
                       const float *weights, const float *shared_gate,
                       moe_bf16 *out, void *stream);

/* A1..A7 in one call: out [T][H] bf16 from x [T][H] bf16.  Optional outputs
 * (each nullable): ids_out [T][8], weights_out [T][8], logits_out [T][E],
 * gate_logit_out [T].  Routes, chosen by sizes only: T <= 64 with
 * hidden <= 2048 (a multiple of 512) and intermediate sizes <= 2048 runs one
 * persistent cooperative kernel (one CTA per SM, bounded grid barriers);
 * other T <= 64 run separate weight-streaming kernels; T >= 65 runs tcgen05
 * grouped GEMMs.  All routes meet the same tolerance and route on the same
 * fp32 logits.  The environment variable MOE_DECODE_ROUTE=gemv (read once
 * per process) forces the separate kernels for T <= 64, for diagnostics.
 * For large T the routed terms are summed
 * with fp32 atomics, so the last fp32 bit of an unrounded sum (and, rarely,
 * the bf16 rounding of out) may vary between runs. */
moe_status moe_block_forward(const moe_dims *dims, const moe_weights *w,
                             const moe_bf16 *x, int T, moe_bf16 *out,
                             int32_t *ids_out, float *weights_out,
                             float *logits_out, float *gate_logit_out,
                             void *workspace, size_t ws_bytes, void *stream);

/* The block and the steps either side of it in a decoder layer (lucebox
 * commit list: the residual add, RMS norm and weight multiply fused, with
 * the residual sum kept beside the normalised output):
 *   resid_out[t] = bf16(resid_in[t] + block(x)[t])   (the block's fp32 sum
 *                  plus the residual, one round to nearest even), and
 *   x_next[t]    = bf16(resid_out[t] / sqrt(mean(resid_out[t]^2) + eps)
 *                  * gamma)                           (the next layer's input).
 * x, resid_in, resid_out, x_next [T][H] bf16; gamma [H] bf16; eps >= 0 and
 * finite.  resid_out may be resid_in (in place) and x_next may be x;
 * x_next must not overlap either residual buffer, and the two residual
 * buffers are the same or disjoint (otherwise MOE_ERR_INVALID_ARG).  Same
 * routes, tolerance and workspace as moe_block_forward; one more kernel (the
 * norm, one warp per token, its sum of squares in a fixed order, so the
 * result does not depend on the batch). */
moe_status moe_block_forward_residual(const moe_dims *dims, const moe_weights *w,
                                      const moe_bf16 *x, int T, const moe_bf16 *resid_in,
                                      const moe_bf16 *gamma, float eps, moe_bf16 *resid_out,
                                      moe_bf16 *x_next, void *workspace, size_t ws_bytes,
                                      void *stream);

/* moe_block_forward with HOST x and out (ordinary or pinned host memory):
 * copies x in, runs the block, copies out back, then synchronises the stream
 * so that out is valid on return.  The staging buffers live in the workspace
 * (size it with moe_workspace_bytes as usual). */
moe_status moe_block_forward_host(const moe_dims *dims, const moe_weights *w,
                                  const moe_bf16 *x_host, int T,
                                  moe_bf16 *out_host, void *workspace,
                                  size_t ws_bytes, void *stream);

/* Profiling form of moe_block_forward: identical work and results, plus a
 * cudaEvent_t record on the stream before the first kernel (events[0]) and
 * after each kernel i (events[i + 1]).  `events` holds n_events >= 1 +
 * moe_block_kernel_count(dims, T) cudaEvent_t handles (created by the
 * caller, timing enabled); fewer returns MOE_ERR_INVALID_ARG. */
moe_status moe_block_forward_profiled(const moe_dims *dims, const moe_weights *w,
                                      const moe_bf16 *x, int T, moe_bf16 *out,
                                      void *workspace, size_t ws_bytes,
                                      void *const *events, int n_events,
                                      void *stream);
/* Number of kernels moe_block_forward launches for this T (0 on bad dims),
 * and the name of kernel i (NULL if out of range). */
int moe_block_kernel_count(const moe_dims *dims, int T);
const char *moe_block_kernel_name(const moe_dims *dims, int T, int i);

/* moe_block_forward for callers that cannot allocate device memory (a
 * plugin in a runtime that owns all device memory, a process with a fixed
 * device-memory budget, a latency-critical path that cannot take
 * cudaMalloc's implicit synchronisation).  There is no counterpart on the
 * pages: this is a packaging variant of the same block.  The caller passes
 * only inputs and outputs; the scratch is a 4 MiB array that the library
 * holds on every GPU that loads it, until the process exits.
 *   - A (dims, T) whose moe_workspace_bytes(dims, T) exceeds 4 MiB is
 *     rejected with MOE_ERR_WORKSPACE (at H = 2048, I = Is = 512 that
 *     admits T <= 38; at H = 512, I = Is = 128, T <= 247).
 *   - Every other check of moe_block_forward (dims, T, weights, x, out) runs
 *     first: a rejected call enqueues nothing and leaves the array as it was.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - Every call shares the one array, which keeps the last call's contents:
 *     calls that overlap on the GPU (other streams, other threads) race.
 *   - The device status word lives in the array and is cleared at the start
 *     of each call; it is not reported. */
moe_status moe_block_forward_noalloc(const moe_dims *dims, const moe_weights *w,
                                     const moe_bf16 *x, int T, moe_bf16 *out,
                                     void *stream);

/* Candidate selection over wide rows (the drafter's top-k lm_head
 * candidates, k raised from 8 to 16: lucebox commit list, "candidate
 * selector head"), and the exact merge that joins vocabulary shards
 * (ninfer-tp2 v0.4.0 notes: the proposal head split by vocabulary, "exact
 * top-16 merge").  Same order as moe_select_top8: greater value wins, the
 * lower index breaks a tie, -0 ties +0.  Every k in 1..16 is served; other
 * k return MOE_ERR_UNSUPPORTED (never a silent default).
 *
 * moe_topk_candidates: for each row t (at logits + t*ld, N fp32 entries,
 * ld >= N, ld a multiple of 4, logits 16-byte aligned), ids[t][0..k-1] =
 * the k best column indices in rank order and values[t][j] =
 * logits[t][ids[t][j]] (bit for bit).  k <= N <= 2^24.  A row holding NaN
 * or +-inf gets ids -1 and values 0 and sets MOE_DEV_NONFINITE.  The
 * workspace (moe_topk_workspace_bytes) holds the status word and one run of
 * 16 keys per 1024 columns of each row.  ids [T][k] int32, values [T][k]. */
size_t moe_topk_workspace_bytes(int T, int N);
moe_status moe_topk_candidates(const float *logits, int T, int ld, int N, int k,
                               int32_t *ids, float *values, void *workspace,
                               size_t ws_bytes, void *stream);

/* moe_topk_merge: row t holds n_lists candidate lists of k (id, value)
 * pairs at ids/values + t*n_lists*k (any order inside a list; the ids of a
 * row distinct and >= 0, e.g. the per-shard results of moe_topk_candidates
 * with each shard's column offset added).  ids_out[t][0..k-1] / values_out =
 * the k best pairs of the row's union in rank order, exact whenever each
 * list holds its shard's top k.  A row with any id < 0 gets ids -1 and
 * values 0 and sets MOE_DEV_NONFINITE.  The workspace holds only the status
 * word (ws_bytes >= 256).  1 <= n_lists <= 65536. */
moe_status moe_topk_merge(const int32_t *ids, const float *values, int T, int n_lists,
                          int k, int32_t *ids_out, float *values_out,
                          void *workspace, size_t ws_bytes, void *stream);

/* Copy the device status word to *bits (synchronises the stream). */
moe_status moe_read_status(const void *workspace, void *stream, uint32_t *bits);
/* Zero the first 256 bytes of the workspace: the device status word and the
 * decode kernel's grid-barrier counter (asynchronous). */
moe_status moe_clear_status(void *workspace, void *stream);

const char *moe_status_string(moe_status s);
int moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
