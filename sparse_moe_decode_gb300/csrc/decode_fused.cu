// decode_fused.cu -- the whole block (A1..A7) for decode-size T in one
// persistent cooperative kernel: one CTA per SM, 16 warps (the producer
// warp and three reducer warps on one SM sub-partition, twelve consumer
// warps in three quads on the other three), phases separated by bounded
// grid barriers (two, one more when T > 24 for the shared selection, one
// more when T > 8 for the item-mode combine).
//
//   R  router: each CTA stages one 512-wide K-slice of every token and of
//      up to 16 of the 257 rows (256 experts + the shared gate) in shared
//      memory and forms fp32 partials with bf16 tensor-core MMAs (the
//      pages' split of the router into K-slices); the last warp of CTA t
//      scales token t into fp16 for phase W;
//   -- grid barrier 1 --
//   S  one warp per token folds the partials in a fixed order and selects
//      the top-8 (8 warp-max rounds over lane-sorted keys; softmax, shared
//      sigmoid); for T <= 24 every CTA selects every token itself, so every
//      CTA holds the same selection; for larger T each token is selected
//      once in the grid and a grid barrier publishes the selections;
//   L  every CTA builds the token -> expert lists in shared memory;
//   W  gate|up + SwiGLU: work unit = 8 gate rows + their 8 up rows of one
//      expert (16 rows x H int8); the first Is / 8 CTAs take one shared
//      unit each before routing is known, and the routed units are claimed
//      from a grid-wide counter, so that faster CTAs take more of them; the
//      producer streams each unit's rows and group scales with two
//      tensor-map copies into a 6-stage shared-memory ring; quad q consumes
//      ring stages q, q + 3, ..., each warp a quarter of K, as m16n8k16
//      fp16 tensor-core MMAs: the int8 weights become fp16 exactly in
//      registers, the activations are each token's copy scaled by a power
//      of two into fp16 (exact for every element within 2^29 of the
//      token's largest), the group scales are promoted per 128-wide K group
//      in fp32; the quad's reducer warp adds the four K quarters in a fixed
//      order and writes h = bf16(silu(gate) * up), with an fp16 copy;
//   -- grid barrier 2 --
//   D  down + combine, two modes chosen by T (the same in every CTA); each
//      quad's down stages continue its own ring sequence past its gate|up
//      end marker.  Item mode (T > kFRowOwnerT): work item = R consecutive
//      output rows (R * max(I, Is) = one 32 KB stage) of one expert,
//      claimed from a second grid-wide counter by the producer as soon as
//      its gate|up claims run out, so the down weights stream in while the
//      gate|up tail is still computing; each warp of the consuming quad
//      takes 16 of the rows over the full K (fp16 MMAs on the fp16 h, bf16
//      ones on the bf16 h when some |h| >= 2^15), and y for every (slot,
//      row) goes to global memory (fp32); after a third grid barrier every
//      thread of the grid forms two output elements.  Row-owner mode (small
//      T, where the extra barrier would cost more than the even split of
//      the bytes gains): CTA c owns output rows 16c .. 16c+15 of every
//      expert, its y stays in shared memory and the CTA writes its combined
//      rows itself.  Both combine the 8 routed y in rank order, then the
//      shared expert's, with one bf16 rounding.
//
// The producer's time per stage bounds the stream once the consumers keep
// up, so it issues as few copy operations per stage as the layout allows
// and forms addresses before its waits.  The tensor cores here are the
// register-fragment form (mma.sync): at decode sizes each weight meets
// 1..~10 tokens, the kernel is bound by HBM, and register fragments avoid a
// shared-memory round trip for the converted weights.  Every wait
// (mbarrier, grid barrier) is bounded by a %globaltimer budget; a wait that
// gives up sets MOE_DEV_TIMEOUT and the kernel runs to its end without
// waiting again.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "select.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

constexpr int kFQuads = 3;
constexpr int kFConsumerWarps = 4 * kFQuads;
constexpr int kFConsumers = kFConsumerWarps * 32;
// 16 warps, 128 registers: warp 0 is the producer, on an SM sub-partition
// with no consumer warp, so that the consumers' issue does not delay its
// copies; warps w with w mod 4 != 0 are consumer warps; warps 4, 8 and 12
// (the producer's sub-partition) reduce the gate|up passes of quads 0, 1, 2.
constexpr int kFThreads = 512;

// consumer warp index (0 .. 11) of warp w (w mod 4 != 0)
__device__ __forceinline__ int consumer_warp(int w) { return w - (w >> 2) - 1; }
__device__ __forceinline__ int consumer_tid() {
  return consumer_warp(threadIdx.x >> 5) * 32 + (threadIdx.x & 31);
}
#ifndef MOE_FUSED_BULK_COPIES
#define MOE_FUSED_BULK_COPIES 0
#endif

constexpr int kFStages = 6;
constexpr int kFRedBufs = 2;  // buffers of each quad's reduction exchange
constexpr int kFStageBytes = 16 * kFusedMaxH;  // one gate|up unit, or packed down units
constexpr int kFScaleBytes = 512;              // the group scales of a stage's rows
constexpr int kFPass = 8;                    // gate|up tokens per pass (one n8 tile)
constexpr int kFDownPass = 16;               // down tokens per pass (two n8 tiles)
constexpr int kRP = 260;                     // router partial row: 257 used, 16-byte rows
// Up to this T every CTA selects every token itself (at most two per warp),
// which costs less than a grid-shared selection's extra grid barrier and
// read-back; above it each token is selected once in the grid.
constexpr int kFLocalSelT = 2 * kFConsumerWarps;
constexpr int kFClaim = 4;  // routed gate|up units per claim when there are many
constexpr int kFRowOwnerT = 8;  // down phase in row-owner mode up to this T

struct FusedParams {
  const moe_bf16 *x;
  uint16_t *x16;        // [T][H] fp16: x * 2^-xexp[t], exact (see scale_token)
  float *xscale;        // [T] 2^xexp[t]
  int T, H, I, Is, KS;  // KS = H / 512 router K-slices
  const moe_bf16 *w_router, *w_gate;
  const int8_t *w13_q;
  const moe_bf16 *w13_s;
  const int8_t *w2_q;
  const moe_bf16 *w2_s;
  const int8_t *ws13_q;
  const moe_bf16 *ws13_s;
  const int8_t *ws2_q;
  const moe_bf16 *ws2_s;
  float *rpart;        // [T][KS][kRP] router partial sums
  int32_t *sel_ids;    // [T][K] selection of every token (T > kFLocalSelT)
  float *sel_w;        // [T][K]
  float *sel_sg;       // [T]
  moe_bf16 *h_routed;  // [T*K][I], rows in list order
  moe_bf16 *h_shared;  // [T][Is]
  uint16_t *h16_routed;  // [T*K][I] fp16 copies of h (exact while every |h| < 2^15)
  uint16_t *h16_shared;  // [T][Is]
  unsigned *h_wide;      // nonzero: some |h| >= 2^15 (or not finite); zeroed in phase R
  float *y;            // [T*K + T][H] down outputs: routed slots in list order, then shared
  moe_bf16 *out;       // [T][H]
  const moe_bf16 *resid;  // [T][H] residual added before the rounding of out, or NULL
  int32_t *ids_out;
  float *weights_out, *logits_out, *gate_logit_out;
  uint32_t *status;
  unsigned *grid_bar;
  unsigned *unit_claims;  // routed gate|up units claimed so far (zeroed in phase R)
  unsigned *down_claims;  // down items claimed so far (zeroed in phase R)
  unsigned long long budget_ns;
};

// Tensor maps of the gate|up rows and their scales ([0] routed, [1] shared):
// one copy fetches a unit's 8 gate and 8 up rows (two blocks I rows apart),
// another their scales, so a stage costs the copy engine two operations
// rather than four.  Rows: (256 bytes, H/256 chunks, row, gate|up, expert),
// box (256, H/256, 8, 2, 1).  Scales: (the 8 * H/128 scales of 8 rows, row
// block, gate|up, expert), box (8 * H/128, 1, 2, 1).  ok = 0: bulk copies.
struct FusedMaps {
  CUtensorMap w[2];
  CUtensorMap s[2];
  int ok;
};

struct FusedSmem {
  uint8_t ring[kFStages][kFStageBytes];
  uint8_t ring_s[kFStages][kFScaleBytes];  // bf16 scales of each stage's rows
  union {
    float red[kFQuads][kFRedBufs][4][32][4];     // gate|up: quad reduction exchange
    float ys[16][kFRowOwnerT * (kK + 1)];      // row-owner down: y of this CTA's 16 rows
  } u;
  int32_t ids[kFusedMaxT][kK];
  float wts[kFusedMaxT][kK];
  float sg[kFusedMaxT];
  float xs[kFusedMaxT];
  int32_t slot_of[kFusedMaxT][kK];
  int32_t perm[kFusedMaxT * kK];
  int32_t counts[kE];
  int32_t offsets[kE + 1];
  int32_t active[kE + 1];
  uint64_t full[kFStages], empty[kFStages], routed;
  int2 stage_unit[kFStages];  // (expert, first row pair | first output row); x < 0: end
  uint64_t red_full[kFQuads][kFRedBufs];   // the quad's four quarters are stored
  uint64_t red_empty[kFQuads][kFRedBufs];  // the reducer has read them
  uint64_t red_done[kFQuads];              // the reducer wrote its last h
  int4 red_meta[kFQuads][kFRedBufs];       // the pass: (expert | -1 = end, i0, tb, 0)
  int abort;
};

// ------------------------------------------------------------ helpers

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate (register fragments).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, f16 inputs, fp32 accumulate (register fragments).
__device__ __forceinline__ void mma16816_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                             uint32_t a2, uint32_t a3, uint32_t b0,
                                             uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 1-D bulk copy global -> shared completing on an mbarrier, L2 evict-first.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(ptx::smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(ptx::smem_u32(bar)), "l"(policy)
      : "memory");
}

// Loads of data written earlier in this launch by other CTAs: L2 only.

__device__ __forceinline__ uint4 ld_ca16(const void *p) {
  return __ldca(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ float ld_cg_f32(const float *p) { return __ldcg(p); }

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ bool aborted(FusedSmem &S) {
  return *reinterpret_cast<volatile int *>(&S.abort) != 0;
}

// Bounded wait used by consumers and the producer: after an abort it no
// longer waits, so control flow (and every named barrier) still completes.
// The first wait of the grid to give up records where: status words 5, 6
// and 7 = site (1: mbarrier, 2: grid barrier), detail (the mbarrier's
// shared-memory offset, the barrier's arrival count) and the CTA.
__device__ __forceinline__ void record_give_up(uint32_t *status, unsigned site, unsigned detail) {
  if (atomicCAS(status + 5, 0u, site) == 0u) {
    status[6] = detail;
    status[7] = blockIdx.x;
  }
}

__device__ __forceinline__ void fwait(uint64_t *bar, uint32_t parity, FusedSmem &S,
                                      uint64_t budget, uint32_t *status) {
  if (aborted(S)) return;
  if (!ptx::mbar_wait(bar, parity, &S.abort, budget))
    record_give_up(status, 1u, static_cast<unsigned>(reinterpret_cast<const uint8_t *>(bar) -
                                                     reinterpret_cast<const uint8_t *>(&S)));
}

// Grid-wide barrier of the consumer threads of every CTA.  Self-resetting:
// CTA 0 adds 2^31 - (G - 1), the others 1, so each barrier flips bit 31 of the
// counter and leaves its low bits unchanged.  The arrival is a release
// reduction (no round trip to wait for); `phase` (consumer thread 0 only) is
// the value bit 31 takes when the barrier completes: the bit read at the
// start of the launch, which every CTA reads alike (no barrier completes
// before every CTA has arrived), flipped at each barrier.  The polling
// thread's acquire load and the CTA barrier after it order the reads that
// follow after every CTA's writes before its arrival.  Bounded by the wait
// budget.
__device__ __forceinline__ void grid_sync(unsigned *bar, unsigned &phase, FusedSmem &S,
                                          uint64_t budget, uint32_t *status) {
  ptx::named_barrier(1, kFConsumers);
  if (consumer_tid() == 0) {
    phase ^= 0x80000000u;
    const unsigned inc = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1) : 1u;
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(bar), "r"(inc) : "memory");
    const uint64_t t0 = ptx::globaltimer();
    unsigned v;
    while (((v = ld_acquire_u32(bar)) & 0x80000000u) != phase) {
      if (aborted(S) || ptx::globaltimer() - t0 > budget) {
        if (!aborted(S)) record_give_up(status, 2u, v & 0x7FFFFFFFu);
        *reinterpret_cast<volatile int *>(&S.abort) = 1;
        break;
      }
      __nanosleep(32);
    }
  }
  ptx::named_barrier(1, kFConsumers);
}

// Routing-derived work sizes (identical in every thread of the CTA; the
// mode and the item sizes are identical in every CTA).
struct Work {
  int nSb, nIb;         // gate|up units of the shared expert, per routed expert
  int n_exp;            // experts with down work: the shared one (if any) + the active ones
  int row_owner;        // down mode (see the file comment)
  // item mode
  int down_rows;        // R: output rows of one down item (a multiple of 16)
  int nrb;              // down items per expert: ceil(H / R)
  // row-owner mode
  int n0;               // first output row of this CTA (-1: none)
  int unit_stride;      // bytes of one 16-row unit in a ring stage
  int scale_stride;     // bytes of one unit's scales in the stage's scale area
  int units_per_stage;
  int n_down_stages;    // of this CTA
};

__device__ __forceinline__ Work make_work(const FusedSmem &S, const FusedParams &p) {
  Work wk;
  wk.nSb = p.Is / 8;
  wk.nIb = p.I / 8;
  wk.n_exp = (p.Is > 0 ? 1 : 0) + S.active[0];
  wk.row_owner = p.T <= kFRowOwnerT ? 1 : 0;
  const int imax = p.I > p.Is ? p.I : p.Is;
  // R rows of K <= imax fill at most one stage; their scales (R * imax/128
  // bf16) then fit the stage's 512-byte scale area
  wk.down_rows = min(p.H, (kFStageBytes / imax) & ~15);
  wk.nrb = (p.H + wk.down_rows - 1) / wk.down_rows;
  wk.n0 = 16 * static_cast<int>(blockIdx.x) < p.H ? 16 * static_cast<int>(blockIdx.x) : -1;
  wk.unit_stride = 16 * imax;
  wk.scale_stride = 2 * 16 * (imax / kG);
  wk.units_per_stage = kFStageBytes / wk.unit_stride;
  const int nu = wk.n0 >= 0 ? wk.n_exp : 0;
  wk.n_down_stages = (nu + wk.units_per_stage - 1) / wk.units_per_stage;
  return wk;
}

// down expert a (0 .. n_exp - 1): the shared expert (kE) first, then the active ones
__device__ __forceinline__ int down_expert(const FusedSmem &S, const FusedParams &p, int a) {
  return p.Is > 0 ? (a == 0 ? kE : S.active[a]) : S.active[1 + a];
}

// down item b (item mode): the expert and its first output row
__device__ __forceinline__ int2 down_item(const FusedSmem &S, const FusedParams &p,
                                          const Work &wk, unsigned b) {
  const int a = static_cast<int>(b) / wk.nrb, rb = static_cast<int>(b) % wk.nrb;
  return make_int2(down_expert(S, p, a), rb * wk.down_rows);
}

// Producer: issue gate|up unit j (expert e, row pairs i0..i0+7) into ring
// stage j % kFStages; false if the stage was not issued (abort).
__device__ __forceinline__ bool produce_gu(FusedSmem &S, const FusedParams &p,
                                           const FusedMaps &maps, int j, int e, int i0,
                                           uint64_t pol, uint64_t budget, int lane) {
  const int s = j % kFStages;
  int go = 0;  // lane 0 decides for the whole warp (the flag may be set meanwhile)
  if (lane == 0) {
    fwait(&S.empty[s], ((j / kFStages) & 1) ^ 1, S, budget, p.status);
    go = aborted(S) ? 0 : 1;
    if (go) {
      S.stage_unit[s] = make_int2(e, i0);  // published by the arrival below
      ptx::mbar_expect_tx(&S.full[s], 16u * p.H + 2u * 8 * 2 * (p.H / kG));
    }
  }
  if (!__shfl_sync(0xFFFFFFFFu, go, 0)) return false;
  if (maps.ok) {
    if (lane == 0) {
      const int sh = e == kE ? 1 : 0;
      ptx::tma_load_5d(S.ring[s], &maps.w[sh], 0, 0, i0, 0, sh ? 0 : e, &S.full[s], pol);
      ptx::tma_load_4d(S.ring_s[s], &maps.s[sh], 0, i0 / 8, 0, sh ? 0 : e, &S.full[s], pol);
    }
  } else if (lane < 4) {
    // lanes 0/1: 8 consecutive gate / up rows, one contiguous copy of 8 * H
    // bytes each (bulk copies of >= 8 KB stream at full rate); lanes 2/3:
    // the bf16 group scales of those rows (8 * H/128 each)
    const int half = e == kE ? p.Is : p.I;
    const int ng = p.H / kG;
    const int row = (lane & 1) == 0 ? i0 : half + i0;
    if (lane < 2) {
      const int8_t *src = e == kE ? p.ws13_q + static_cast<size_t>(row) * p.H
                                  : p.w13_q + (static_cast<size_t>(e) * 2 * p.I + row) * p.H;
      bulk_g2s(S.ring[s] + lane * 8 * p.H, src, 8u * p.H, &S.full[s], pol);
    } else {
      const moe_bf16 *src = e == kE ? p.ws13_s + static_cast<size_t>(row) * ng
                                    : p.w13_s + (static_cast<size_t>(e) * 2 * p.I + row) * ng;
      bulk_g2s(S.ring_s[s] + (lane - 2) * 8 * ng * 2, src, 2u * 8 * ng, &S.full[s], pol);
    }
  }
  __syncwarp();
  return true;
}

// Producer, row-owner mode: issue this CTA's down stage k into ring stage
// j % kFStages: the 16 output rows n0 of down experts k * U .. k * U + U - 1
// (one contiguous copy of 16 * K bytes each, at a fixed stride in the stage)
// and their group scales.  False if the stage was not issued (abort).
__device__ __forceinline__ bool produce_rows(FusedSmem &S, const FusedParams &p, const Work &wk,
                                             int j, int k, uint64_t pol, uint64_t budget,
                                             int lane) {
  const int s = j % kFStages;
  const int a0 = k * wk.units_per_stage;
  const int nu = min(wk.units_per_stage, wk.n_exp - a0);
  int go = 0;  // lane 0 decides for the whole warp (the flag may be set meanwhile)
  if (lane == 0) {
    fwait(&S.empty[s], ((j / kFStages) & 1) ^ 1, S, budget, p.status);
    uint32_t tx = 0;
    for (int u = 0; u < nu; ++u) {
      const int Ii = down_expert(S, p, a0 + u) == kE ? p.Is : p.I;
      tx += 16u * Ii + 2u * 16 * (Ii / kG);
    }
    go = aborted(S) ? 0 : 1;
    if (go) {
      S.stage_unit[s] = make_int2(kE + 1, k);  // published by the arrival below
      ptx::mbar_expect_tx(&S.full[s], tx);
    }
  }
  if (!__shfl_sync(0xFFFFFFFFu, go, 0)) return false;
  if (lane < 2 * nu) {
    // lane u < nu: unit u's rows; lane nu + u: their group scales
    const int u = lane < nu ? lane : lane - nu;
    const int e = down_expert(S, p, a0 + u);
    const int Ii = e == kE ? p.Is : p.I;
    const int ng = Ii / kG;
    const int n0 = wk.n0;
    if (lane < nu) {
      const int8_t *src = e == kE ? p.ws2_q + static_cast<size_t>(n0) * p.Is
                                  : p.w2_q + (static_cast<size_t>(e) * p.H + n0) * p.I;
      bulk_g2s(S.ring[s] + u * wk.unit_stride, src, 16u * Ii, &S.full[s], pol);
    } else {
      const moe_bf16 *src = e == kE ? p.ws2_s + static_cast<size_t>(n0) * ng
                                    : p.w2_s + (static_cast<size_t>(e) * p.H + n0) * ng;
      bulk_g2s(S.ring_s[s] + u * wk.scale_stride, src, 2u * 16 * ng, &S.full[s], pol);
    }
  }
  __syncwarp();
  return true;
}

// Producer, item mode: issue down item (e, n0) = rows n0 .. n0 + nr - 1 of
// expert e's down matrix (nr * K contiguous bytes, lane 0) and their group
// scales (lane 1) into ring stage j % kFStages.  The addresses are formed
// before the wait and both copies go out in one instruction: the producer's
// time per stage bounds the stream.  False if the stage was not issued.
__device__ __forceinline__ bool produce_item(FusedSmem &S, const FusedParams &p, const Work &wk,
                                             int j, int e, int n0, uint64_t pol,
                                             uint64_t budget, int lane) {
  const int s = j % kFStages;
  const bool sh = e == kE;
  const int Ii = sh ? p.Is : p.I;
  const int ng = Ii / kG;
  const int nr = min(wk.down_rows, p.H - n0);
  const uint32_t wbytes = static_cast<uint32_t>(nr) * Ii, sbytes = 2u * nr * ng;
  const size_t row0 = sh ? static_cast<size_t>(n0) : static_cast<size_t>(e) * p.H + n0;
  const void *src = lane == 0 ? static_cast<const void *>((sh ? p.ws2_q : p.w2_q) + row0 * Ii)
                              : static_cast<const void *>((sh ? p.ws2_s : p.w2_s) + row0 * ng);
  void *dst = lane == 0 ? static_cast<void *>(S.ring[s]) : static_cast<void *>(S.ring_s[s]);
  const uint32_t bytes = lane == 0 ? wbytes : sbytes;
  int go = 0;  // lane 0 decides for the whole warp (the flag may be set meanwhile)
  if (lane == 0) {
    fwait(&S.empty[s], ((j / kFStages) & 1) ^ 1, S, budget, p.status);
    go = aborted(S) ? 0 : 1;
    if (go) {
      S.stage_unit[s] = make_int2(e, n0);  // published by the arrival below
      ptx::mbar_expect_tx(&S.full[s], wbytes + sbytes);
    }
  }
  if (!__shfl_sync(0xFFFFFFFFu, go, 0)) return false;
  if (lane < 2) bulk_g2s(dst, src, bytes, &S.full[s], pol);
  __syncwarp();
  return true;
}

// Token scaling for the fp16 tensor-core path: token t becomes x * 2^-s in
// fp16 with s = exponent(max |x_t|) - 14, so the largest magnitude lands in
// [2^14, 2^15).  A bf16 value (8 significant bits) is exact in fp16 whenever
// the scaled value is a normal fp16, i.e. for every element within 2^29 of
// the token's largest; smaller ones are off by less than 2^-40 of that
// largest.  2^s is undone on the fp32 results.  One warp.
__device__ __forceinline__ void scale_token(const FusedParams &p, int t, int lane) {
  const moe_bf16 *xr = p.x + static_cast<size_t>(t) * p.H;
  float m = 0.0f;
  for (int k = lane * 8; k < p.H; k += 256) {
    const uint4 v = ld_nc(xr + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  int sexp = 0;
  if (m > 0.0f && isfinite(m)) {
    sexp = static_cast<int>((__float_as_uint(m) >> 23) & 0xFF) - 127 - 14;
    sexp = max(-110, min(110, sexp));
  }
  const float down = __uint_as_float(static_cast<uint32_t>(127 - sexp) << 23);  // 2^-s
  for (int k = lane * 8; k < p.H; k += 256) {
    const uint4 v = ld_nc(xr + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(bf16_lo(w[i]) * down, bf16_hi(w[i]) * down);
      o[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p.x16 + static_cast<size_t>(t) * p.H + k) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) p.xscale[t] = __uint_as_float(static_cast<uint32_t>(127 + sexp) << 23);
}

// Phase R: router partials (the pages' split of the router GEMV into
// K-slices).  CTA c takes K-slice ks = c mod KS (512 wide) of a group of at
// most 16 rows (256 expert rows, row 256 = the shared gate): it stages the
// slices of every token and of its rows in shared memory (ring stages 1..,
// unused until routing is known; rows padded to 1040 bytes so that the
// fragment loads below hit distinct banks), all loads in flight at once.
// Task (nt, kq) is one warp: bf16 m16n8k16 tensor-core MMAs (products
// exact, fp32 accumulation) of tokens 8nt .. 8nt+7 over the slice's K
// quarter kq; the four quarters are then added in order.  Every token's
// partials are formed the same way whatever T is, so a token's routing
// does not depend on the batch it rides in.  The last warp of CTA t (t < T)
// scales token t instead.
constexpr int kRStride = 520;  // bf16 per staged row

__device__ __forceinline__ void phase_router(FusedSmem &S, const FusedParams &p, int cwarp,
                                             int lane) {
  if (blockIdx.x == 0 && consumer_tid() == 0) {  // claimed / set after barrier 1
    *p.unit_claims = 0u;
    *p.down_claims = 0u;
    *p.h_wide = 0u;
  }
  const int G = static_cast<int>(gridDim.x);
  const bool scales = static_cast<int>(blockIdx.x) < p.T;
  if (scales && cwarp == kFConsumerWarps - 1) {
    for (int t = blockIdx.x; t < p.T; t += G) scale_token(p, t, lane);
    return;
  }
  const int n_rw = kFConsumerWarps - (scales ? 1 : 0);  // router warps of this CTA
  const int rows_total = kE + (p.Is > 0 ? 1 : 0);
  const int n_rg = G / p.KS;  // row groups
  const int rpg = min(16, (rows_total + n_rg - 1) / n_rg);
  const int rg = static_cast<int>(blockIdx.x) / p.KS, ks = static_cast<int>(blockIdx.x) % p.KS;
  const int r0 = rg * rpg;
  const int nr = rg < n_rg ? max(0, min(rpg, rows_total - r0)) : 0;
  if (nr == 0) return;  // (the size check makes the groups cover every row)
  // staged slices: the T token rows from ring stage 1 (up to 65 KB), then the
  // 16 weight rows (rows nr.. zero)
  moe_bf16 *xs = reinterpret_cast<moe_bf16 *>(S.ring[1]);
  moe_bf16 *ws = xs + p.T * kRStride;
  const int n_x = p.T * 64;  // uint4 per token slice: 64
  for (int i = cwarp * 32 + lane; i < n_x + 16 * 64; i += n_rw * 32) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    moe_bf16 *dst;
    if (i < n_x) {
      v = ld_nc(p.x + static_cast<size_t>(i >> 6) * p.H + ks * 512 + (i & 63) * 8);
      dst = xs + (i >> 6) * kRStride + (i & 63) * 8;
    } else {
      const int ri = (i - n_x) >> 6;
      if (ri < nr) {
        const int r = r0 + ri;
        const moe_bf16 *wrow = r < kE ? p.w_router + static_cast<size_t>(r) * p.H : p.w_gate;
        v = ld_nc(wrow + ks * 512 + (i & 63) * 8);
      }
      dst = ws + ri * kRStride + (i & 63) * 8;
    }
    *reinterpret_cast<uint4 *>(dst) = v;
  }
  ptx::named_barrier(5, n_rw * 32);
  const int g = lane >> 2, c = lane & 3;
  const int n_nt = (p.T + 7) / 8;
  float *part = reinterpret_cast<float *>(ws + 16 * kRStride);  // [n_nt * 4][4][32]
  for (int task = cwarp; task < 4 * n_nt; task += n_rw) {
    const int nt = task >> 2, kq = task & 3;
    const int t = nt * 8 + g;  // this lane's B column (token)
    const uint32_t *xr = reinterpret_cast<const uint32_t *>(xs + min(t, p.T - 1) * kRStride);
    const uint32_t *wlo = reinterpret_cast<const uint32_t *>(ws + g * kRStride);
    const uint32_t *whi = reinterpret_cast<const uint32_t *>(ws + (g + 8) * kRStride);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k2 = 64 * kq; k2 < 64 * kq + 64; k2 += 8) {  // k2: bf16 pairs, 8 per k16 step
      const uint32_t b0 = t < p.T ? xr[k2 + c] : 0u, b1 = t < p.T ? xr[k2 + 4 + c] : 0u;
      mma16816(d, wlo[k2 + c], whi[k2 + c], wlo[k2 + 4 + c], whi[k2 + 4 + c], b0, b1);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) part[(task * 4 + i) * 32 + lane] = d[i];
  }
  ptx::named_barrier(5, n_rw * 32);
  // d0, d1 of lane l: row g, tokens 8nt + 2c, +1; d2, d3: row g + 8
  for (int idx = cwarp * 32 + lane; idx < n_nt * 128; idx += n_rw * 32) {
    const int nt = idx >> 7, i = (idx >> 5) & 3, ln = idx & 31;
    const float *q = part + (nt * 16 + i) * 32 + ln;  // quarter kq at q[kq * 128]
    const float v = ((q[0] + q[128]) + q[256]) + q[384];
    const int row = (ln >> 2) + (i >> 1) * 8, tok = nt * 8 + 2 * (ln & 3) + (i & 1);
    if (row < nr && tok < p.T)
      p.rpart[(static_cast<size_t>(tok) * p.KS + ks) * kRP + r0 + row] = v;
  }
  // the staged slices were written and read by the generic proxy; the ring
  // is next written by bulk copies (async proxy)
  ptx::fence_proxy_async_smem();
}

// Token t's selection: fold the K-slice partials (fixed order), select the
// top-8, softmax, shared gate.  Local: into this CTA's shared memory (every
// CTA selects every token; CTA 0 writes the optional outputs).  Otherwise
// into the global selection arrays, by the one warp that owns token t.
__device__ __forceinline__ void select_token(FusedSmem &S, const FusedParams &p, int t,
                                             int lane, bool local) {
  const bool first = !local || blockIdx.x == 0;  // writes the optional outputs
  const float *rp = p.rpart + static_cast<size_t>(t) * p.KS * kRP;
  float4 a0[kFusedMaxH / 512], a1[kFusedMaxH / 512];
  float gp[kFusedMaxH / 512];
#pragma unroll
  for (int ks = 0; ks < kFusedMaxH / 512; ++ks) {  // all loads in flight at once
    if (ks < p.KS) {
      const float4 *row = reinterpret_cast<const float4 *>(rp + ks * kRP + 8 * lane);
      a0[ks] = __ldcg(row);
      a1[ks] = __ldcg(row + 1);
      gp[ks] = p.Is > 0 ? ld_cg_f32(rp + ks * kRP + kE) : 0.0f;
    }
  }
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float g = 0.0f;
#pragma unroll
  for (int ks = 0; ks < kFusedMaxH / 512; ++ks) {  // fixed K-slice order
    if (ks < p.KS) {
      v[0] += a0[ks].x; v[1] += a0[ks].y; v[2] += a0[ks].z; v[3] += a0[ks].w;
      v[4] += a1[ks].x; v[5] += a1[ks].y; v[6] += a1[ks].z; v[7] += a1[ks].w;
      g += gp[ks];
    }
  }
  int id[8];
  float w[8];
  const bool ok = select_top8_rounds(v, lane, id, w);
  if (lane < 8) {
    int myid = id[0];
    float myw = w[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
      if (lane == i) { myid = id[i]; myw = w[i]; }
    if (local) {
      S.ids[t][lane] = myid;
      S.wts[t][lane] = myw;
    } else {
      p.sel_ids[t * kK + lane] = myid;
      p.sel_w[t * kK + lane] = myw;
    }
    if (first && p.ids_out) p.ids_out[t * kK + lane] = myid;
    if (first && p.weights_out) p.weights_out[t * kK + lane] = myw;
  }
  if (lane == 0) {
    const float sg = p.Is > 0 ? sigmoidf_(g) : 0.0f;
    if (local) S.sg[t] = sg;
    else p.sel_sg[t] = sg;
    if (first && p.gate_logit_out && p.Is > 0) p.gate_logit_out[t] = g;
    if (first && !ok) set_status(p.status, MOE_DEV_NONFINITE);
  }
  if (first && p.logits_out) {
    float4 *dst = reinterpret_cast<float4 *>(p.logits_out + static_cast<size_t>(t) * kE + 8 * lane);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// Phases S and L.  T <= kFLocalSelT: every CTA selects all T tokens itself
// (warp w takes tokens w, w + 12, ..., with the same fold order and
// selection in every CTA, so every CTA holds the same selection), with no
// grid barrier between selection and lists.  Larger T: one warp of the grid
// per token (one token per CTA), a grid barrier, and every CTA reads all
// selections.  Then every CTA builds the token -> expert lists in shared
// memory.
__device__ __forceinline__ void phase_select_lists(FusedSmem &S, const FusedParams &p, int cwarp,
                                                   int lane, unsigned &phase, uint64_t budget) {
  const int tid = consumer_tid();
  // independent of the selection, so done first, by the last warps
  for (int t2 = kFConsumers - 1 - tid; t2 < p.T; t2 += kFConsumers)
    S.xs[t2] = __ldcg(p.xscale + t2);
  if (p.T <= kFLocalSelT) {
    for (int t = cwarp; t < p.T; t += kFConsumerWarps) select_token(S, p, t, lane, true);
  } else {
    // one token per CTA (consumer warp 0): the merge network is bound by
    // issue, so tokens that share an SM sub-partition take turns
    const int t = blockIdx.x + gridDim.x * cwarp;
    if (t < p.T) select_token(S, p, t, lane, false);
    grid_sync(p.grid_bar, phase, S, budget, p.status);
    for (int i = tid; i < p.T * kK; i += kFConsumers) {
      S.ids[i / kK][i % kK] = __ldcg(p.sel_ids + i);
      S.wts[i / kK][i % kK] = __ldcg(p.sel_w + i);
    }
    for (int t2 = tid; t2 < p.T; t2 += kFConsumers) S.sg[t2] = __ldcg(p.sel_sg + t2);
  }
  ptx::named_barrier(1, kFConsumers);
  // Lists, in (expert, t, j) order.  Warp 0 walks the entries in batches of
  // 32 in entry order: the lanes naming one expert (__match_any_sync) take
  // consecutive places after that expert's earlier entries, so each entry
  // learns its rank within its expert (kept in slot_of for now); warp 0 then
  // scans the counts into offsets and the active list, and every thread
  // places its entries.
  const int n = p.T * kK;
  if (cwarp == 0) {
    for (int e = lane; e < kE; e += 32) S.counts[e] = 0;
    __syncwarp();
    for (int b = 0; b < n; b += 32) {
      const int i = b + lane;
      const int e = i < n ? S.ids[i / kK][i % kK] : -1;
      const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
      const int lead = __ffs(same) - 1;
      int before = 0;
      if (lane == lead && e >= 0) {
        before = S.counts[e];
        S.counts[e] = before + __popc(same);
      }
      before = __shfl_sync(0xFFFFFFFFu, before, lead);
      if (i < n) S.slot_of[i / kK][i % kK] = e >= 0 ? before + __popc(same & ((1u << lane) - 1u)) : -1;
      __syncwarp();
    }
    // offsets: exclusive scan of the counts (8 experts per lane), and the
    // active list (experts with entries, ascending)
    int c[kE / 32], run = 0, act = 0;
#pragma unroll
    for (int k = 0; k < kE / 32; ++k) {
      c[k] = S.counts[8 * lane + k];
      run += c[k];
      act += c[k] > 0 ? 1 : 0;
    }
    int incl = run, aincl = act;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      const int y = __shfl_up_sync(0xFFFFFFFFu, aincl, o);
      if (lane >= o) { incl += x; aincl += y; }
    }
    int off = incl - run, a = aincl - act;
#pragma unroll
    for (int k = 0; k < kE / 32; ++k) {
      S.offsets[8 * lane + k] = off;
      off += c[k];
      if (c[k] > 0) S.active[1 + a++] = 8 * lane + k;
    }
    if (lane == 31) {
      S.offsets[kE] = incl;
      S.active[0] = aincl;
    }
  }
  ptx::named_barrier(1, kFConsumers);
  for (int i = tid; i < n; i += kFConsumers) {
    const int t = i / kK, jj = i % kK, e = S.ids[t][jj];
    if (e >= 0) {
      const int pos = S.offsets[e] + S.slot_of[t][jj];
      S.perm[pos] = i;
      S.slot_of[t][jj] = pos;
    }
  }
  ptx::named_barrier(1, kFConsumers);
}

// One 64-wide K slice of a 16-row unit against one n8 token tile: A rows g
// and g+8 from the staged rows (int8 -> bf16 in registers), B fragments xw.
// Logical k (2c, 2c+1 | 2c+8, 2c+9) of MMA jj maps to physical k
// 16c + 4jj + (0, 1 | 2, 3) for A and B alike.
__device__ __forceinline__ void mma_slice(const uint8_t *rows, int stride, int k0, int g, int c,
                                          const uint32_t (&xw)[8], float (&part)[4]) {
  const uint4 qa = *reinterpret_cast<const uint4 *>(rows + g * stride + k0 + 16 * c);
  const uint4 qb = *reinterpret_cast<const uint4 *>(rows + (g + 8) * stride + k0 + 16 * c);
  const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    // bytes 4jj..4jj+3 of rows g and g+8, converted just before their MMA
    const f4 fa = i8x4_to_f32(wa[jj]), fb = i8x4_to_f32(wb[jj]);
    const uint32_t a0 = __byte_perm(__float_as_uint(fa.x), __float_as_uint(fa.y), 0x7632);
    const uint32_t a2 = __byte_perm(__float_as_uint(fa.z), __float_as_uint(fa.w), 0x7632);
    const uint32_t a1 = __byte_perm(__float_as_uint(fb.x), __float_as_uint(fb.y), 0x7632);
    const uint32_t a3 = __byte_perm(__float_as_uint(fb.z), __float_as_uint(fb.w), 0x7632);
    mma16816(part, a0, a1, a2, a3, xw[2 * jj], xw[2 * jj + 1]);
  }
}

// As mma_slice with f16 operands: the int8 rows convert exactly to f16 and
// the B fragments hold the token's scaled fp16 activations.
__device__ __forceinline__ void mma_slice_f16(const uint8_t *rows, int stride, int k0, int g,
                                              int c, const uint32_t (&xw)[8],
                                              float (&part)[4]) {
  const uint4 qa = *reinterpret_cast<const uint4 *>(rows + g * stride + k0 + 16 * c);
  const uint4 qb = *reinterpret_cast<const uint4 *>(rows + (g + 8) * stride + k0 + 16 * c);
  const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    uint32_t a0, a1, a2, a3;
    i8x4_to_f16x2(wa[jj], a0, a2);
    i8x4_to_f16x2(wb[jj], a1, a3);
    mma16816_f16(part, a0, a1, a2, a3, xw[2 * jj], xw[2 * jj + 1]);
  }
}

// The K range [kb, kb + kn) (a multiple of 64) of a 16-row unit for one n8
// token tile, bf16 operands.  The B fragments of up to four slices (256 of
// K) are fetched together before their MMAs, so each batch pays one memory
// latency; each slice's partial sums are promoted with its group's scales
// (lo: rows 0..7, hi: rows 8..15).  brow = this lane's token row or NULL:
// rows of h, written before the grid barrier that precedes the down phase
// and read by no SM earlier in the launch, so L1 holds no stale copy and
// caching them there serves the other warps and items of the same expert.
template <bool F16>
__device__ __forceinline__ void unit_gemm(const uint8_t *rows, int stride, int kb, int kn,
                                          const uint16_t *brow, int g, int c,
                                          const moe_bf16 *s_lo, const moe_bf16 *s_hi,
                                          float (&acc)[4]) {
  for (int kk = kb; kk < kb + kn; kk += 256) {
    const int ns = min(4, (kb + kn - kk) / 64);
    uint32_t xw[4][8];
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      if (brow && sl < ns) {
        const uint16_t *src = brow + kk + 64 * sl + 16 * c;
        const uint4 x0 = ld_ca16(src), x1 = ld_ca16(src + 8);
        xw[sl][0] = x0.x; xw[sl][1] = x0.y; xw[sl][2] = x0.z; xw[sl][3] = x0.w;
        xw[sl][4] = x1.x; xw[sl][5] = x1.y; xw[sl][6] = x1.z; xw[sl][7] = x1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xw[sl][i] = 0u;
      }
    }
    if (ns == 4) {
      // a full batch with no branch between its slices, so that their
      // independent MMA chains interleave
      float part[4][4];
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
#pragma unroll
        for (int i = 0; i < 4; ++i) part[sl][i] = 0.0f;
        if (F16) mma_slice_f16(rows, stride, kk + 64 * sl, g, c, xw[sl], part[sl]);
        else mma_slice(rows, stride, kk + 64 * sl, g, c, xw[sl], part[sl]);
      }
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        const int k0 = kk + 64 * sl;
        const float slo = bf16_to_f32(s_lo[k0 / kG]), shi = bf16_to_f32(s_hi[k0 / kG]);
        acc[0] = fmaf(slo, part[sl][0], acc[0]);
        acc[1] = fmaf(slo, part[sl][1], acc[1]);
        acc[2] = fmaf(shi, part[sl][2], acc[2]);
        acc[3] = fmaf(shi, part[sl][3], acc[3]);
      }
    } else {
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        if (sl >= ns) break;
        const int k0 = kk + 64 * sl;
        const float slo = bf16_to_f32(s_lo[k0 / kG]), shi = bf16_to_f32(s_hi[k0 / kG]);
        float part[4] = {0.f, 0.f, 0.f, 0.f};
        if (F16) mma_slice_f16(rows, stride, k0, g, c, xw[sl], part);
        else mma_slice(rows, stride, k0, g, c, xw[sl], part);
        acc[0] = fmaf(slo, part[0], acc[0]);
        acc[1] = fmaf(slo, part[1], acc[1]);
        acc[2] = fmaf(shi, part[2], acc[2]);
        acc[3] = fmaf(shi, part[3], acc[3]);
      }
    }
  }
}

// One consumer warp's K quarter of gate|up pass u of quad q into the quad's
// exchange buffer; warp 0 of the quad also stores the pass (m.x = -1: the
// quad's gate|up units are done).
__device__ __forceinline__ void hand_off(FusedSmem &S, const FusedParams &p, int q, int wq,
                                         int lane, uint32_t u, int4 m, const float (&acc)[4],
                                         uint64_t budget) {
  const int b = u % kFRedBufs;
  fwait(&S.red_empty[q][b], ((u / kFRedBufs) & 1) ^ 1, S, budget, p.status);
  *reinterpret_cast<float4 *>(S.u.red[q][b][wq][lane]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  if (wq == 0 && lane == 0) S.red_meta[q][b] = m;
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(&S.red_full[q][b]);
}

// Reducer warp of quad q: for each gate|up pass, the four K quarters added in
// a fixed order, 2^s undone, h = bf16(silu(gate) * up) and its fp16 copy
// (r17) written.  A bf16 value (8 significant bits) below 2^15 in magnitude
// is exact in fp16 down to 2^-17; smaller ones land on fp16's subnormal grid
// (error < 2^-25); a larger one sets h_wide.
__device__ __forceinline__ void reduce_gu(FusedSmem &S, const FusedParams &p, int q, int lane,
                                          uint64_t budget) {
  const int g = lane >> 2, c = lane & 3;
  bool wide = false;
  for (uint32_t u = 0;; ++u) {
    const int b = u % kFRedBufs;
    fwait(&S.red_full[q][b], (u / kFRedBufs) & 1, S, budget, p.status);
    if (aborted(S)) break;
    const int4 m = S.red_meta[q][b];
    if (m.x < 0) break;
    const int e = m.x, i0 = m.y, tb = m.z;
    const bool sh = e == kE;
    const int n_tok = sh ? p.T : S.counts[e];
    const int p0 = sh ? 0 : S.offsets[e];
    float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w2 = 0; w2 < 4; ++w2) {  // fixed order
      const float4 v = *reinterpret_cast<const float4 *>(S.u.red[q][b][w2][lane]);
      r4[0] += v.x; r4[1] += v.y; r4[2] += v.z; r4[3] += v.w;
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&S.red_empty[q][b]);
#pragma unroll
    for (int col = 0; col < 2; ++col) {
      const int idx = tb + 2 * c + col;
      if (idx < n_tok) {
        const float xsv = S.xs[sh ? idx : S.perm[p0 + idx] / kK];  // undo 2^-s
        const uint16_t hv = f32_to_bf16(silu_mul(r4[col] * xsv, r4[2 + col] * xsv));
        const float hf = __uint_as_float(static_cast<uint32_t>(hv) << 16);
        const uint16_t h16 = __half_as_ushort(__float2half_rn(hf));
        wide |= !(fabsf(hf) < 32768.0f);
        const size_t o = sh ? static_cast<size_t>(idx) * p.Is + i0 + g
                            : static_cast<size_t>(p0 + idx) * p.I + i0 + g;
        (sh ? p.h_shared : p.h_routed)[o] = hv;
        (sh ? p.h16_shared : p.h16_routed)[o] = h16;
      }
    }
  }
  if (__any_sync(0xFFFFFFFFu, wide) && lane == 0) atomicOr(p.h_wide, 1u);
  // Every h of this quad (and the flag) reaches the other CTAs through a
  // chain that needs no fence here: this release arrival (after the warp
  // barrier), the consumers' acquire wait for red_done, the CTA barrier of
  // their grid barrier and its gpu-scope release reduction, whose acquire
  // load in every other CTA precedes the reads of h (causality order is
  // transitive across these scopes).
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(&S.red_done[q]);
}

// Phase W consumer: gate|up unit j of this CTA, by quad q (warp wq of 4
// takes K quarter wq).
// Returns false at the stage that marks the end of the gate|up units (after
// releasing it).
__device__ __forceinline__ bool consume_gu(FusedSmem &S, const FusedParams &p, int j, int q,
                                           int wq, int lane, uint64_t budget, uint32_t &npass) {
  const int s = j % kFStages;
  fwait(&S.full[s], (j / kFStages) & 1, S, budget, p.status);
  if (aborted(S)) return false;
  const int2 un = S.stage_unit[s];
  if (un.x < 0) {
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&S.empty[s]);
    const float none[4] = {0.f, 0.f, 0.f, 0.f};
    hand_off(S, p, q, wq, lane, npass++, make_int4(-1, 0, 0, 0), none, budget);
    return false;
  }
  const int e = un.x, i0 = un.y;
  const bool sh = e == kE;
  const int n_tok = sh ? p.T : S.counts[e];
  const int p0 = sh ? 0 : S.offsets[e];
  const int g = lane >> 2, c = lane & 3;
  const int ng = p.H / kG;
  // the stage's scale area holds the 8 gate rows' then the 8 up rows' scales
  const moe_bf16 *s_gate = reinterpret_cast<const moe_bf16 *>(S.ring_s[s]) + g * ng;
  const moe_bf16 *s_up = reinterpret_cast<const moe_bf16 *>(S.ring_s[s]) + (8 + g) * ng;
  const int kq = p.H / 4, kb = wq * kq;
  const uint8_t *rows = S.ring[s];
  const int stride = p.H;
  for (int tb = 0; tb < n_tok; tb += kFPass) {
    const moe_bf16 *brow = nullptr;  // this lane's B column (token) of the n8 tile
    if (tb + g < n_tok) {
      const int t = sh ? tb + g : S.perm[p0 + tb + g] / kK;
      brow = reinterpret_cast<const moe_bf16 *>(p.x16) + static_cast<size_t>(t) * p.H;
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kk = kb; kk < kb + kq; kk += 256) {  // batches of 4 slices (2 groups)
      const int ns4 = min(4, (kb + kq - kk) / 64);
      uint32_t xw[4][8];
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        if (brow && sl < ns4) {
          // fp16 rows written before grid barrier 1 of this launch: no SM
          // reads them earlier, so L1 holds no stale copy, and caching
          // them in L1 serves this CTA's many units of the same expert
          const moe_bf16 *src = brow + kk + 64 * sl + 16 * c;
          const uint4 x0 = ld_ca16(src), x1 = ld_ca16(src + 8);
          xw[sl][0] = x0.x; xw[sl][1] = x0.y; xw[sl][2] = x0.z; xw[sl][3] = x0.w;
          xw[sl][4] = x1.x; xw[sl][5] = x1.y; xw[sl][6] = x1.z; xw[sl][7] = x1.w;
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) xw[sl][i] = 0u;
        }
      }
      const int g0 = gateup_scale_group(kk / kG, ng), g1 = gateup_scale_group(kk / kG + 1, ng);
      const float slo0 = bf16_to_f32(s_gate[g0]), shi0 = bf16_to_f32(s_up[g0]);
      const float slo1 = ns4 > 2 ? bf16_to_f32(s_gate[g1]) : 0.0f;
      const float shi1 = ns4 > 2 ? bf16_to_f32(s_up[g1]) : 0.0f;
      if (ns4 == 4) {
        // a full batch with no branch between its slices, so that their
        // independent MMA chains interleave
        float part[4][4];
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
#pragma unroll
          for (int i = 0; i < 4; ++i) part[sl][i] = 0.0f;
          mma_slice_f16(rows, stride, kk + 64 * sl, g, c, xw[sl], part[sl]);
        }
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          const float slo = sl < 2 ? slo0 : slo1, shi = sl < 2 ? shi0 : shi1;
          acc[0] = fmaf(slo, part[sl][0], acc[0]);
          acc[1] = fmaf(slo, part[sl][1], acc[1]);
          acc[2] = fmaf(shi, part[sl][2], acc[2]);
          acc[3] = fmaf(shi, part[sl][3], acc[3]);
        }
      } else {
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          if (sl >= ns4) break;
          float part[4] = {0.f, 0.f, 0.f, 0.f};
          mma_slice_f16(rows, stride, kk + 64 * sl, g, c, xw[sl], part);
          const float slo = sl < 2 ? slo0 : slo1, shi = sl < 2 ? shi0 : shi1;
          acc[0] = fmaf(slo, part[0], acc[0]);
          acc[1] = fmaf(slo, part[1], acc[1]);
          acc[2] = fmaf(shi, part[2], acc[2]);
          acc[3] = fmaf(shi, part[3], acc[3]);
        }
      }
    }
    if (tb + kFPass >= n_tok) {  // the stage's rows are no longer needed
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.empty[s]);
    }
    // Hand the K quarter to the quad's reducer warp (kFRedBufs buffers), which
    // adds the four quarters in a fixed order, applies SwiGLU and writes h.
    hand_off(S, p, q, wq, lane, npass++, make_int4(e, i0, tb, 0), acc, budget);
  }
  if (n_tok == 0) {
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&S.empty[s]);
  }
  return true;
}

// One 16-row down unit of expert e over its full K (rows: the unit's int8
// rows at stride K, sbase: their scales, row by row) against every token of
// the expert; y goes to shared memory (ys != NULL: row-owner mode, rows
// 0..15 of this CTA) or to global row n0 of each slot.
__device__ __forceinline__ void down_unit_gemm(const FusedSmem &S, const FusedParams &p, int e,
                                               const uint8_t *rows, const moe_bf16 *sbase,
                                               float (*ys)[kFRowOwnerT * (kK + 1)], int n0,
                                               bool f16, int lane) {
  const bool sh = e == kE;
  const int Ii = sh ? p.Is : p.I;
  const int ng = Ii / kG;
  const int n_tok = sh ? p.T : S.counts[e];
  const int p0 = sh ? p.T * kK : S.offsets[e];  // first y slot of the expert
  const int g = lane >> 2, c = lane & 3;
  const moe_bf16 *s_lo = sbase + g * ng;
  const moe_bf16 *s_hi = sbase + (g + 8) * ng;
  for (int tb = 0; tb < n_tok; tb += kFDownPass) {
    const int ntiles = min(2, (n_tok - tb + 7) / 8);
    const uint16_t *brow[2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int idx = tb + 8 * nt + g;
      brow[nt] = nullptr;
      if (idx < n_tok) {
        const size_t o = sh ? static_cast<size_t>(idx) * p.Is : static_cast<size_t>(p0 + idx) * p.I;
        brow[nt] = f16 ? (sh ? p.h16_shared : p.h16_routed) + o
                       : reinterpret_cast<const uint16_t *>(sh ? p.h_shared : p.h_routed) + o;
      }
    }
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int nt = 0; nt < ntiles; ++nt) {
      if (f16) unit_gemm<true>(rows, Ii, 0, Ii, brow[nt], g, c, s_lo, s_hi, acc[nt]);
      else unit_gemm<false>(rows, Ii, 0, Ii, brow[nt], g, c, s_lo, s_hi, acc[nt]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int col = 0; col < 2; ++col) {
        const int idx = tb + 8 * nt + 2 * c + col;
        if (nt < ntiles && idx < n_tok) {
          if (ys) {
            ys[g][p0 + idx] = acc[nt][col];
            ys[g + 8][p0 + idx] = acc[nt][2 + col];
          } else {
            float *yr = p.y + static_cast<size_t>(p0 + idx) * p.H + n0;
            yr[g] = acc[nt][col];
            yr[g + 8] = acc[nt][2 + col];
          }
        }
      }
  }
}

// Phase D consumer: the down stage in ring stage j, by one quad: warp wq
// takes the stage's 16-row units wq, wq + 4, ....  Returns false at the
// stage that marks the end of the down stages (after releasing it).
__device__ __forceinline__ bool consume_down(FusedSmem &S, const FusedParams &p, const Work &wk,
                                             int j, int wq, bool f16, int lane, uint64_t budget) {
  const int s = j % kFStages;
  fwait(&S.full[s], (j / kFStages) & 1, S, budget, p.status);
  if (aborted(S)) return false;
  const int2 it = S.stage_unit[s];
  if (it.x > kE) {  // row-owner stage k = it.y
    const int a0 = it.y * wk.units_per_stage;
    const int nu = min(wk.units_per_stage, wk.n_exp - a0);
    for (int u = wq; u < nu; u += 4)
      down_unit_gemm(S, p, down_expert(S, p, a0 + u), S.ring[s] + u * wk.unit_stride,
                     reinterpret_cast<const moe_bf16 *>(S.ring_s[s] + u * wk.scale_stride),
                     S.u.ys, 0, f16, lane);
  } else if (it.x >= 0) {  // item (e, n0)
    const int e = it.x, n0 = it.y;
    const int Ii = e == kE ? p.Is : p.I;
    const int nu = min(wk.down_rows, p.H - n0) / 16;
    for (int u = wq; u < nu; u += 4)
      down_unit_gemm(S, p, e, S.ring[s] + static_cast<size_t>(16 * u) * Ii,
                     reinterpret_cast<const moe_bf16 *>(S.ring_s[s]) + 16 * u * (Ii / kG),
                     nullptr, n0 + 16 * u, f16, lane);
  }
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(&S.empty[s]);
  return it.x >= 0;
}

// Row-owner mode: this CTA's 16 output rows from the y in shared memory:
// slots in rank order, then the shared expert, fp32, one bf16 rounding.
__device__ __forceinline__ void combine_rows(FusedSmem &S, const FusedParams &p, const Work &wk) {
  if (wk.n0 < 0) return;
  for (int i = consumer_tid(); i < 16 * p.T; i += kFConsumers) {
    const int r = i & 15, t = i >> 4;
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < kK; ++j) {
      const int slot = S.slot_of[t][j];
      const float w = S.wts[t][j];
      if (slot >= 0 && w != 0.0f) acc = fmaf(w, S.u.ys[r][slot], acc);
    }
    if (p.Is > 0 && S.sg[t] != 0.0f) acc = fmaf(S.sg[t], S.u.ys[r][p.T * kK + t], acc);
    const size_t o = static_cast<size_t>(t) * p.H + wk.n0 + r;
    if (p.resid) acc += bf16_to_f32(p.resid[o]);
    p.out[o] = f32_to_bf16(acc);
  }
}

// Item mode: out[t][n] = sum over token t's slots in rank order of w * y, then
// the shared expert's sg * y, in fp32 with one bf16 rounding; two adjacent
// n per thread, spread over the consumer threads of the whole grid.
__device__ __forceinline__ void phase_combine(FusedSmem &S, const FusedParams &p) {
  const int half = p.H / 2;
  const int n_all = p.T * half;
  for (int i = blockIdx.x * kFConsumers + consumer_tid(); i < n_all;
       i += gridDim.x * kFConsumers) {
    const int t = i / half, n = 2 * (i - t * half);
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int j = 0; j < kK; ++j) {
      const int slot = S.slot_of[t][j];
      const float w = S.wts[t][j];
      if (slot >= 0 && w != 0.0f) {
        const float2 v = __ldcg(reinterpret_cast<const float2 *>(p.y + static_cast<size_t>(slot) * p.H + n));
        a0 = fmaf(w, v.x, a0);
        a1 = fmaf(w, v.y, a1);
      }
    }
    if (p.Is > 0 && S.sg[t] != 0.0f) {
      const float2 v = __ldcg(reinterpret_cast<const float2 *>(
          p.y + static_cast<size_t>(p.T * kK + t) * p.H + n));
      a0 = fmaf(S.sg[t], v.x, a0);
      a1 = fmaf(S.sg[t], v.y, a1);
    }
    if (p.resid) {
      const uint32_t r2 =
          *reinterpret_cast<const uint32_t *>(p.resid + static_cast<size_t>(t) * p.H + n);
      a0 += bf16_lo(r2);
      a1 += bf16_hi(r2);
    }
    const uint32_t o = static_cast<uint32_t>(f32_to_bf16(a0)) |
                       (static_cast<uint32_t>(f32_to_bf16(a1)) << 16);
    *reinterpret_cast<uint32_t *>(p.out + static_cast<size_t>(t) * p.H + n) = o;
  }
}

__global__ void __launch_bounds__(kFThreads, 1)
    decode_fused_kernel(const __grid_constant__ FusedMaps maps, const FusedParams p) {
  extern __shared__ __align__(128) uint8_t fsmem_raw[];
  FusedSmem &S = *reinterpret_cast<FusedSmem *>(fsmem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t budget = p.budget_ns;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFStages; ++s) {
      ptx::mbar_init(&S.full[s], 1);
      ptx::mbar_init(&S.empty[s], 4);  // the four warps of the consuming quad
    }
    ptx::mbar_init(&S.routed, 1);
    for (int q = 0; q < kFQuads; ++q) {
      for (int b = 0; b < kFRedBufs; ++b) {
        ptx::mbar_init(&S.red_full[q][b], 4);   // the quad's four warps
        ptx::mbar_init(&S.red_empty[q][b], 1);  // the reducer
      }
      ptx::mbar_init(&S.red_done[q], 1);
    }
    S.abort = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = ptx::policy_evict_first();
    // the shared expert's unit needs no routing: fetch it at once
    const bool early = p.Is > 0 && static_cast<int>(blockIdx.x) < p.Is / 8;
    // per ring slot, the latest stage whose copies were issued: after an
    // abort only those can still be in flight (a slot is reused only after
    // its previous copies landed and were consumed)
    int last_use[kFStages];
#pragma unroll
    for (int i = 0; i < kFStages; ++i) last_use[i] = -1;
    auto issued_at = [&](int jj) {
#pragma unroll
      for (int i = 0; i < kFStages; ++i)
        if (jj % kFStages == i) last_use[i] = jj;
    };
    if (early && produce_gu(S, p, maps, 0, kE, 8 * blockIdx.x, pol, budget, lane)) issued_at(0);
    if (lane == 0) fwait(&S.routed, 0, S, budget, p.status);
    __syncwarp();
    const Work wk = make_work(S, p);
    // Routed gate|up units are claimed from a grid-wide counter, one claim
    // ahead, so that CTAs that run faster take more of them.  When there are
    // many, a claim takes kFClaim consecutive units (rows of one expert), so
    // that the counter's round trip overlaps the issue of the units already
    // claimed; when there are few, single units keep the split even.
    const unsigned n_routed = static_cast<unsigned>(S.active[0] * wk.nIb);
    const unsigned G = gridDim.x;
    int j = early ? 1 : 0;  // ring index of the next stage
    // Few units (few tokens, so nearly equal costs): a static round-robin
    // split with no claims, in which the shared units of the first Is / 8
    // CTAs count as the first slots, so every CTA streams its units at once.
    const bool static_gu = n_routed < 24u * G;
    if (static_gu) {
      const unsigned nS = static_cast<unsigned>(wk.nSb);
      for (unsigned b = (blockIdx.x + G - nS % G) % G; b < n_routed && !aborted(S); b += G) {
        const int e = S.active[1 + b / wk.nIb], i0 = 8 * static_cast<int>(b % wk.nIb);
        if (produce_gu(S, p, maps, j, e, i0, pol, budget, lane)) issued_at(j);
        ++j;
      }
    }
    const unsigned gu_claim = static_cast<unsigned>(kFClaim);
    // the first claim of CTA c is c itself (no round trip to the counter);
    // the counter numbers the claims after the first G.  Two claims are
    // requested ahead, so that the counter's round trip stays hidden even
    // when the ring has room and a claim's units issue at once.  A CTA uses
    // its claims in the order it requested them, which is increasing, so
    // every claim below the total is used by the CTA that took it.
    const unsigned gu_base = G * gu_claim;
    unsigned claim = static_gu ? n_routed : blockIdx.x * gu_claim;
    unsigned ahead0 = n_routed, ahead1 = n_routed;  // lane 0's requested claims
    if (lane == 0 && claim < n_routed) {
      ahead0 = gu_base + atomicAdd(p.unit_claims, gu_claim);
      ahead1 = gu_base + atomicAdd(p.unit_claims, gu_claim);
    }
    while (claim < n_routed && !aborted(S)) {
      const unsigned end = min(claim + gu_claim, n_routed);
      for (unsigned b = claim; b < end; ++b) {
        const int e = S.active[1 + b / wk.nIb], i0 = 8 * static_cast<int>(b % wk.nIb);
        if (produce_gu(S, p, maps, j, e, i0, pol, budget, lane)) issued_at(j);
        ++j;
      }
      claim = __shfl_sync(0xFFFFFFFFu, ahead0, 0);
      ahead0 = ahead1;
      if (lane == 0 && claim < n_routed) ahead1 = gu_base + atomicAdd(p.unit_claims, gu_claim);
    }
    // one end marker per quad (each quad takes every kFQuads-th stage, so
    // kFQuads consecutive markers reach every quad once)
    auto end_markers = [&]() {
      for (int k = 0; k < kFQuads && !aborted(S); ++k, ++j) {
        if (lane == 0) {
          fwait(&S.empty[j % kFStages], ((j / kFStages) & 1) ^ 1, S, budget, p.status);
          if (!aborted(S)) {
            S.stage_unit[j % kFStages] = make_int2(-1, 0);
            ptx::mbar_arrive(&S.full[j % kFStages]);
          }
        }
        __syncwarp();
      }
    };
    end_markers();
    if (wk.row_owner) {
      for (int k = 0; k < wk.n_down_stages && !aborted(S); ++k, ++j)
        if (produce_rows(S, p, wk, j, k, pol, budget, lane)) issued_at(j);
    }
    // Down items, claimed from their own counter the same way (their costs
    // differ with the expert's token count, so a static split would not
    // balance them); their weights need no h, so they stream while the
    // gate|up units are still computing.  A CTA claims at most cap items:
    // before the grid barrier no down stage is consumed, and without a cap
    // the CTAs that reach this point first would take several items per quad
    // when there are few (decode).
    const unsigned n_down = wk.row_owner ? 0u : static_cast<unsigned>(wk.n_exp * wk.nrb);
    const unsigned per_claim = n_down >= 8u * G ? 2u : 1u;
    const unsigned cap = max(static_cast<unsigned>(kFQuads), (4u * n_down / 3u + G - 1u) / G);
    const unsigned dn_base = G * per_claim;  // first claims static, as for gate|up
    claim = blockIdx.x * per_claim;
    // requested ahead as for gate|up, up to cap items per CTA
    unsigned taken = per_claim;
    ahead0 = n_down;
    ahead1 = n_down;
    if (lane == 0 && claim < n_down) {
      if (taken < cap) { ahead0 = dn_base + atomicAdd(p.down_claims, per_claim); taken += per_claim; }
      if (taken < cap) { ahead1 = dn_base + atomicAdd(p.down_claims, per_claim); taken += per_claim; }
    }
    while (claim < n_down && !aborted(S)) {
      const unsigned end = min(claim + per_claim, n_down);
      for (unsigned b = claim; b < end; ++b, ++j) {
        const int2 it = down_item(S, p, wk, b);
        if (produce_item(S, p, wk, j, it.x, it.y, pol, budget, lane)) issued_at(j);
      }
      claim = __shfl_sync(0xFFFFFFFFu, ahead0, 0);
      ahead0 = ahead1;
      ahead1 = n_down;
      if (lane == 0 && claim < n_down && taken < cap) {
        ahead1 = dn_base + atomicAdd(p.down_claims, per_claim);
        taken += per_claim;
      }
    }
    end_markers();
    // after an abort, let the copies already in flight land before exiting
    if (aborted(S) && lane == 0) {
      int never = 0;
#pragma unroll
      for (int i = 0; i < kFStages; ++i)
        if (last_use[i] >= 0)
          ptx::mbar_wait(&S.full[i], (last_use[i] / kFStages) & 1, &never, ptx::kDrainBudgetNs);
    }
  } else if ((warp & 3) != 0) {
    // ----------------------------------------------------------- consumers
    const int cw = consumer_warp(warp);
    const int q = cw >> 2, wq = cw & 3;
    // bit 31 of the grid-barrier counter (used by consumer thread 0 only)
    unsigned bar_phase = consumer_tid() == 0 ? ld_acquire_u32(p.grid_bar) & 0x80000000u : 0u;
    phase_router(S, p, cw, lane);
    grid_sync(p.grid_bar, bar_phase, S, budget, p.status);
    phase_select_lists(S, p, cw, lane, bar_phase, budget);
    if (consumer_tid() == 0) ptx::mbar_arrive(&S.routed);
    const Work wk = make_work(S, p);
    uint32_t npass = 0;
    // quad q takes ring stages q, q + kFQuads, ...: its gate|up units up to
    // its end marker, then its down stages, so that each stage it waits for
    // reuses the slot of a stage it consumed itself (a wait is never two
    // phases ahead of a slot's barrier)
    int j = q;
    while (consume_gu(S, p, j, q, wq, lane, budget, npass)) j += kFQuads;
    fwait(&S.red_done[q], 0, S, budget, p.status);
    grid_sync(p.grid_bar, bar_phase, S, budget, p.status);
    // every h is written: the down MMAs take the fp16 copies unless some h
    // is outside fp16's range
    const bool f16 = __ldcg(p.h_wide) == 0u;
    for (j += kFQuads; consume_down(S, p, wk, j, wq, f16, lane, budget); j += kFQuads) {
    }
    if (wk.row_owner) {
      ptx::named_barrier(1, kFConsumers);
      combine_rows(S, p, wk);
    } else {
      grid_sync(p.grid_bar, bar_phase, S, budget, p.status);
      phase_combine(S, p);
    }
  } else {
    // ------------------------------------------------------------ reducers
    reduce_gu(S, p, (warp >> 2) - 1, lane, budget);
  }
  __syncthreads();
  if (threadIdx.x == 0 && aborted(S)) set_status(p.status, MOE_DEV_TIMEOUT);
}

int device_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

unsigned long long fused_wait_budget_ns() {
  static unsigned long long v = 0;
  if (!v) {
    const char *e = getenv("MOE_WAIT_BUDGET_NS");
    v = e ? strtoull(e, nullptr, 10) : 2000000000ull;
    if (!v) v = 1;
  }
  return v;
}

}  // namespace

size_t fused_smem_bytes() { return sizeof(FusedSmem); }

bool fused_decode_supported(int T, int H, int I, int Is) {
  if (T < 1 || T > kFusedMaxT || H > kFusedMaxH || H % 512 != 0) return false;
  if (I > kFusedMaxI || Is > kFusedMaxI || I % 128 != 0 || Is % 128 != 0) return false;
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return false;
  if (!sms[dev]) {
    // one resident CTA per SM is required for the grid barriers
    int per_sm = 0;
    if (cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(FusedSmem))) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused_kernel, kFThreads,
                                                      sizeof(FusedSmem)) != cudaSuccess ||
        per_sm < 1) {
      sms[dev] = -1;
    } else {
      sms[dev] = device_sms();
    }
  }
  // the SMs must cover the Is / 8 shared gate|up units (one per CTA) and the
  // router's 257 rows in groups of at most 16 per K-slice
  return sms[dev] > 0 && sms[dev] * 8 >= Is && (sms[dev] / (H / 512)) * 16 >= kE + 1;
}

cudaError_t launch_decode_fused(const moe_bf16 *x, int T, int H, int I, int Is,
                                const moe_weights &w, uint16_t *x16, float *xscale,
                                float *rpart, int32_t *sel_ids, float *sel_w,
                                float *sel_sg, moe_bf16 *h_routed,
                                moe_bf16 *h_shared, moe_bf16 *out, int32_t *ids_out,
                                float *weights_out, float *logits_out, float *gate_logit_out,
                                uint32_t *status, unsigned *grid_bar, unsigned *unit_claims,
                                unsigned *down_claims, float *y, uint16_t *h16,
                                unsigned *h_wide, const moe_bf16 *resid, cudaStream_t s) {
  FusedParams p{};
  p.x = x; p.x16 = x16; p.xscale = xscale;
  p.T = T; p.H = H; p.I = I; p.Is = Is; p.KS = H / 512;
  p.w_router = w.w_router; p.w_gate = Is > 0 ? w.w_shared_gate : nullptr;
  p.w13_q = w.w13_q; p.w13_s = w.w13_s; p.w2_q = w.w2_q; p.w2_s = w.w2_s;
  p.ws13_q = w.ws13_q; p.ws13_s = w.ws13_s; p.ws2_q = w.ws2_q; p.ws2_s = w.ws2_s;
  p.rpart = rpart; p.sel_ids = sel_ids; p.sel_w = sel_w; p.sel_sg = sel_sg;
  p.unit_claims = unit_claims;
  p.down_claims = down_claims;
  p.y = y;
  p.h_routed = h_routed; p.h_shared = h_shared; p.out = out; p.resid = resid;
  p.h16_routed = h16;
  p.h16_shared = h16 + static_cast<size_t>(T) * kK * I;
  p.h_wide = h_wide;
  p.ids_out = ids_out; p.weights_out = weights_out; p.logits_out = logits_out;
  p.gate_logit_out = gate_logit_out; p.status = status; p.grid_bar = grid_bar;
  p.budget_ns = fused_wait_budget_ns();
  // tensor maps of the gate|up rows and scales, kept per thread for the last
  // weight set (encoding them takes host time on every call otherwise)
  struct MapKey {
    const void *w, *ws, *sc, *ssc;
    int H, I, Is, dev;
    bool operator==(const MapKey &o) const {
      return w == o.w && ws == o.ws && sc == o.sc && ssc == o.ssc && H == o.H && I == o.I &&
             Is == o.Is && dev == o.dev;
    }
  };
  static thread_local MapKey mkey{};
  static thread_local FusedMaps maps{};
  int dev = 0;
  cudaGetDevice(&dev);
  const MapKey key{w.w13_q, w.ws13_q, w.w13_s, w.ws13_s, H, I, Is, dev};
  if (!(key == mkey) || !maps.ok) {
    FusedMaps m{};
    const uint64_t ng = static_cast<uint64_t>(H) / kG;
    auto rows_map = [&](CUtensorMap *t, const void *base, uint64_t half, uint64_t ne) {
      const uint64_t dims[5] = {256, static_cast<uint64_t>(H) / 256, half, 2, ne};
      const uint64_t str[4] = {256, static_cast<uint64_t>(H), half * H, 2 * half * H};
      const uint32_t box[5] = {256, static_cast<uint32_t>(H / 256), 8, 2, 1};
      return tc_make_map_nd(t, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, dims, str, box);
    };
    auto scale_map = [&](CUtensorMap *t, const void *base, uint64_t half, uint64_t ne) {
      const uint64_t dims[4] = {8 * ng, half / 8, 2, ne};
      const uint64_t str[3] = {16 * ng, half * ng * 2, 2 * half * ng * 2};
      const uint32_t box[4] = {static_cast<uint32_t>(8 * ng), 1, 2, 1};
      return tc_make_map_nd(t, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, dims, str, box);
    };
    bool ok = rows_map(&m.w[0], w.w13_q, I, kE) && scale_map(&m.s[0], w.w13_s, I, kE);
    if (Is > 0) {
      ok = ok && rows_map(&m.w[1], w.ws13_q, Is, 1) && scale_map(&m.s[1], w.ws13_s, Is, 1);
    } else {
      m.w[1] = m.w[0];
      m.s[1] = m.s[0];
    }
    // a test-only build (MOE_FUSED_BULK_COPIES = 1) takes the bulk-copy path
    // that serves when the maps cannot be encoded, so that it stays tested
    m.ok = ok && !MOE_FUSED_BULK_COPIES ? 1 : 0;
    maps = m;
    mkey = key;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(device_sms());
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = sizeof(FusedSmem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel, maps, p);
}

}  // namespace moe
