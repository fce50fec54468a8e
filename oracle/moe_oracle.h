/*
 * moe_oracle.h -- plain, slow CPU statement of the sparse-MoE block.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  The
 * product path (sparse_moe_decode_gb300) never links, imports or calls it,
 * and it shares no code, header, table or helper with the CUDA sources.
 *
 * Everything is computed in fp64 from the bf16 / int8 inputs, except the
 * points where the method itself fixes a precision:
 *   - router logits are rounded to fp32 ("the fp32 logits" the selector and
 *     its bit-exact contract are defined on);
 *   - the SwiGLU activation h is rounded to bf16 before the down projection
 *     (the down projections consume 16-bit activations);
 *   - the block output is rounded to bf16 (round to nearest, ties to even).
 *
 * Sources (ninfer-windows PR #8, the commit that swaps eight dependent
 * selection rounds for a warp merge network):
 *   router + 257th shared-gate row ......... the S1/S2 description and its
 *                                            roofline paragraph (T x 257 rows)
 *   total order "greater value, lower id" .. the bit-identity paragraph
 *                                            (sparse_moe_ranked_better)
 *   softmax over the 8 selected logits,
 *   shared-expert sigmoid .................. same paragraph (the selector tail)
 *   per-expert counting ..................... the prefill select_count kernel
 *   int8 groupwise experts, stacked gate|up,
 *   fused SwiGLU, A16 down projections ..... ninfer release notes ("W8 SwiGLU"),
 *                                            ninfer-tp2 v0.2.3 notes (A16 SwiGLU
 *                                            and down), lucebox "stacked
 *                                            projections" commit (swiglu_split)
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int oracle_version(void);

/* bf16 <-> fp64.  bf16 is the upper 16 bits of an IEEE binary32. */
double   oracle_bf16_to_f64(uint16_t b);
/* Round an fp64 value directly to the nearest bf16, ties to even
 * (no intermediate rounding through fp32).  NaN -> 0x7FC0. */
uint16_t oracle_f64_to_bf16(double v);

/* Elementwise array forms of the two conversions above (n elements). */
void oracle_bf16_to_f64_array(int64_t n, const uint16_t *in, double *out);
void oracle_f64_to_bf16_array(int64_t n, const double *in, uint16_t *out);

/* A1 router: logits[t][e] = fp32( sum_k x[t][k] * Wr[e][k] ), e < E, and
 * gate_logit[t] = fp32( sum_k x[t][k] * wg[k] ) when wg != NULL.
 * x [T][H] bf16, Wr [E][H] bf16, wg [H] bf16. */
void oracle_router_logits(int T, int H, int E, const uint16_t *x,
                          const uint16_t *w_router, const uint16_t *w_gate,
                          float *logits, float *gate_logit);

/* A2 selection: for each token the K best (value, id) pairs of its E fp32
 * logits under the total order "greater value wins, lower id breaks a tie"
 * (IEEE ==, so -0 and +0 tie), in rank order; softmax over the K selected
 * values (fp64, max-subtracted); shared gate sigmoid(gate_logit[t]).
 * logits row t starts at logits + t*ld.  A row holding any NaN/inf gets
 * ids = -1 and weights = 0.  gate_logit and sgate may be NULL.
 * Returns the number of non-finite rows. */
int oracle_select_topk(int T, int E, int K, int ld, const float *logits,
                       const float *gate_logit, int32_t *ids, double *weights,
                       double *sgate);

/* The steps either side of the block (lucebox commit list, the fused
 * DeltaNet decode kernels entry: an ADD + RMS_NORM + MUL fusion that keeps
 * the residual sum beside the normalised output).  For each token t, with
 * block[t] the block's unrounded output:
 *   resid_out[t][i] = bf16(resid_in[t][i] + block[t][i])   (one rounding)
 *   ms              = mean over i of resid_out[t][i]^2      (the bf16 values)
 *   x_next[t][i]    = bf16(resid_out[t][i] / sqrt(ms + eps) * gamma[i])
 * All in fp64.  resid_in, gamma, resid_out, x_next: bf16 bits. */
void oracle_add_rmsnorm(int T, int H, const uint16_t *resid_in, const double *block,
                        const uint16_t *gamma, double eps, uint16_t *resid_out,
                        uint16_t *x_next);

/* Wide top-k candidates and their exact merge (the candidate selector of
 * the DFlash2 drafter: GPU top-k with at most 16 candidates, lucebox
 * commit list, "candidate selector head"; a vocabulary split across two
 * GPUs joined by an exact top-16 merge, ninfer-tp2 v0.4.0 notes).  The
 * selection itself is oracle_select_topk on rows of any width (ids only are
 * used; the values are the row's entries at those ids).
 *
 * oracle_merge_topk: row t holds n_lists candidate lists of K (value, id)
 * pairs each, at values/ids + t*n_lists*K; the output is the K best pairs of
 * their union under the selector's total order, in rank order.  An id < 0
 * anywhere in the row (a list from a non-finite row) makes the output row
 * ids -1, values 0.  Returns the number of such rows. */
int oracle_merge_topk(int T, int n_lists, int K, const int32_t *ids,
                      const float *values, int32_t *ids_out, float *values_out);

/* A3 token -> expert lists: counts[e] = #(t,j) with ids[t][j]==e,
 * offsets[0..E] exclusive scan of counts, perm = the entries t*K+j sorted by
 * (expert, t, j).  Entries with id < 0 are skipped. */
void oracle_expert_lists(int T, int E, int K, const int32_t *ids,
                         int32_t *counts, int32_t *offsets, int32_t *perm);

/* Groupwise int8 GEMV: out[r] = sum_k q[r][k] * s[r][k/G] * v[k], with
 * q [R][C] int8, s [R][C/G] bf16, v [C] bf16 (fp64 accumulate). */
void oracle_w8_gemv(int R, int C, int G, const int8_t *q, const uint16_t *s,
                    const uint16_t *v, double *out);

/* A4 SwiGLU of a stacked pre-activation a[0..2I): gate rows 0..I-1, up rows
 * I..2I-1.  h_exact[i] = silu(a[i]) * a[I+i], silu(z) = z / (1 + e^-z);
 * h_bf16[i] = bf16(h_exact[i]).  Either output may be NULL. */
void oracle_swiglu(int I, const double *a, double *h_exact, uint16_t *h_bf16);

/* A7 combine of one token: out[n] = sum_{j<K} w[j]*y[j][n] + sg*ys[n],
 * ys may be NULL (no shared expert).  out_bf16 may be NULL. */
void oracle_combine(int H, int K, const double *y, const double *w,
                    const double *ys, double sg, double *out,
                    uint16_t *out_bf16);

/* The whole block, A1..A7, for the tokens in `tokens` (all T if NULL).
 * Expert weights: w13_q [E][2I][H] int8, w13_s [E][2I][H/G] bf16,
 * w2_q [E][H][I] int8, w2_s [E][H][I/G] bf16; shared expert likewise with
 * Is in place of I and no leading E (all shared pointers NULL iff Is == 0).
 * If route_logits is given ([T][E] fp32, row stride E), selection runs on
 * those values (and route_gate, [T] fp32, for the shared gate) instead of
 * the oracle's own router output.  Outputs are indexed by token t (not by
 * position in `tokens`); any output pointer may be NULL.
 *   out_bf16 [T][H], out_f64 [T][H], ids [T][K], weights [T][K],
 *   sgate [T], logits [T][E] (the oracle's own fp32 logits),
 *   gate_logit [T], y [T][K+1][H] (slot K = shared expert, unscaled),
 *   h [T][K+1][I'] bf16 with I' = max(I, Is).
 * nthreads <= 1 runs on the calling thread.  Returns the number of
 * non-finite routing rows among the computed tokens, or -1 on bad args. */
typedef struct {
  int32_t T, H, E, K, I, Is, G;
} oracle_dims;

typedef struct {
  const uint16_t *w_router, *w_gate;
  const int8_t *w13_q; const uint16_t *w13_s;
  const int8_t *w2_q;  const uint16_t *w2_s;
  const int8_t *ws13_q; const uint16_t *ws13_s;
  const int8_t *ws2_q;  const uint16_t *ws2_s;
} oracle_weights;

int oracle_block_forward(const oracle_dims *d, const oracle_weights *w,
                         const uint16_t *x, const int32_t *tokens,
                         int n_tokens, const float *route_logits,
                         const float *route_gate, uint16_t *out_bf16,
                         double *out_f64, int32_t *ids, double *weights,
                         double *sgate, float *logits, float *gate_logit,
                         double *y, uint16_t *h, int nthreads);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */
