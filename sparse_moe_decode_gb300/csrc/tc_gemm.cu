// tc_gemm.cu -- prefill-size T: the expert SwiGLU (A4/A6), the down
// projection with the weighted combine (A5/A6/A7) and the router (A1) as
// grouped GEMMs on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Orientation: D[row, token] = sum_k W[row, k] * X[token, k].  The weight
// tile is the M = 128 operand, the tokens of one expert are N (<= 128), so
// one pass streams each weight tile once for all of its expert's tokens, and
// the per-row group scale s[row][k / 128] is one scalar per TMEM lane.
//
// int8 weights: TMA brings a 128 x 128 int8 tile (128-byte swizzle) into
// shared memory; worker warps convert it exactly to bf16 (|q| <= 128 is exact
// in bf16) into the canonical K-major SWIZZLE_128B layout; one thread issues
// tcgen05.mma (bf16 x bf16 -> fp32) for the 128-wide K group into one of two
// TMEM partial buffers; the workers read the partial back (tcgen05.ld),
// multiply it by the row's group scale and add it to an fp32 accumulator in
// registers ("scale promotion"): W = q * s is never rounded.
//
// Warp roles (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues MMAs, warps 2..9 convert, promote and run the epilogue.  Every wait
// is bounded by a %globaltimer budget; on expiry the CTA drains what it has
// in flight, frees TMEM, sets MOE_DEV_TIMEOUT and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kTcThreads = 320;
constexpr int kWorkers = 8;                 // worker warps
constexpr int kQS = 3, kAS = 2, kBS = 2;    // pipeline depths
constexpr int kBRows = 32;                  // rows per B TMA box
constexpr uint32_t kQBytes = 128 * 128;     // int8 A tile
constexpr uint32_t kABytes = 2 * 128 * 128; // bf16 A tile, two K halves
constexpr uint32_t kBBytes = 2 * 128 * 128; // bf16 B tile (<= 128 rows), two K halves
constexpr uint32_t kXchBytes = 64 * 128 * 4;
constexpr uint32_t kTmemCols = 256;         // two partial buffers of 128 columns

constexpr size_t kOffQ = 0;
constexpr size_t kOffA = kOffQ + kQS * kQBytes;
constexpr size_t kOffB = kOffA + kAS * kABytes;
constexpr size_t kOffX = kOffB + kBS * kBBytes;
constexpr size_t kOffBar = kOffX + kXchBytes;
constexpr size_t kTcSmem = kOffBar + 256 + 1024;  // + barriers + alignment slack

enum Mode : int { kGateUp = 0, kDown = 1, kRouter = 2 };

struct Bars {
  uint64_t q_full[kQS], q_empty[kQS], a_full[kAS], a_empty[kAS], b_full[kBS], b_empty[kBS];
  uint64_t p_full[2], p_empty[2], done, xch_full, xch_empty;
  uint32_t tmem_holder;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct TcParams {
  const int4 *items;      // {expert (kE = shared), mtile, first row of B, n tokens}
  const int *n_items;
  int K_routed, K_shared;          // reduction lengths
  int rows_routed, rows_shared;    // gate/up: I and Is; down: H for both
  const moe_bf16 *s_routed, *s_shared;  // group scales [rows][K/G]
  moe_bf16 *h_routed, *h_shared;   // gate/up outputs
  float *out_acc;                  // down: fp32 [T][H]
  const int *perm;
  const float *weights, *sgate;
  int H;
  float *logits;                   // router: [T][E]
  int T_router;
  uint32_t *status;
  unsigned long long budget_ns;
};

__device__ __forceinline__ uint4 cvt16_i8_bf16_lo(uint4 q, uint4 &hi) {
  // 16 int8 -> 16 bf16: exact magic-number conversion to fp32, then the
  // upper halves (exact for integers of <= 8 significant bits) are packed.
  const f4 a = i8x4_to_f32(q.x), b = i8x4_to_f32(q.y), c = i8x4_to_f32(q.z),
           d = i8x4_to_f32(q.w);
  auto pk = [](float lo, float hi_) {
    return __byte_perm(__float_as_uint(lo), __float_as_uint(hi_), 0x7632);
  };
  uint4 lo;
  lo.x = pk(a.x, a.y); lo.y = pk(a.z, a.w); lo.z = pk(b.x, b.y); lo.w = pk(b.z, b.w);
  hi.x = pk(c.x, c.y); hi.y = pk(c.z, c.w); hi.z = pk(d.x, d.y); hi.w = pk(d.z, d.w);
  return lo;
}

template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAs,
               const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBs,
               const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars *bars = reinterpret_cast<Bars *>(smem + kOffBar);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // router mode: item it = (128-row tile it % 2, 128 tokens from 128 * (it / 2))
  const int n_items = MODE == kRouter ? 2 * ((p.T_router + 127) / 128) : *p.n_items;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQS; ++i) {
      ptx::mbar_init(&bars->q_full[i], 1);
      ptx::mbar_init(&bars->q_empty[i], kWorkers);
    }
    for (int i = 0; i < kAS; ++i) {
      ptx::mbar_init(&bars->a_full[i], MODE == kRouter ? 1 : kWorkers);
      ptx::mbar_init(&bars->a_empty[i], 1);
    }
    for (int i = 0; i < kBS; ++i) {
      ptx::mbar_init(&bars->b_full[i], 1);
      ptx::mbar_init(&bars->b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->p_full[i], 1);
      ptx::mbar_init(&bars->p_empty[i], kWorkers);
    }
    ptx::mbar_init(&bars->done, 1);
    ptx::mbar_init(&bars->xch_full, 4);   // the four warps holding up rows
    ptx::mbar_init(&bars->xch_empty, 4);  // the four warps holding gate rows
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_holder, kTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_holder;
  const uint64_t budget = p.budget_ns;

  auto item_at = [&](int it) {
    if (MODE == kRouter) {
      const int t0 = (it >> 1) * 128;
      return make_int4(0, it & 1, t0, min(128, p.T_router - t0));
    }
    return p.items[it];
  };
  auto groups_of = [&](const int4 &itm) {
    return (itm.x == kE ? p.K_shared : p.K_routed) / kG;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmA); ptx::tma_prefetch_desc(&tmAs);
      ptx::tma_prefetch_desc(&tmB); ptx::tma_prefetch_desc(&tmBs);
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      uint32_t na = 0, nb_issued = 0;  // A-side and B-side stages issued
      bool stop = false;
      for (int it = blockIdx.x; it < n_items && !stop; it += gridDim.x) {
        const int4 itm = item_at(it);
        const bool sh = itm.x == kE;
        const int ng = groups_of(itm);
        const void *ta = sh ? static_cast<const void *>(&tmAs) : static_cast<const void *>(&tmA);
        const void *tb = sh ? static_cast<const void *>(&tmBs) : static_cast<const void *>(&tmB);
        int rA0, rA1;
        if (MODE == kGateUp) {
          const int half = sh ? p.rows_shared : p.rows_routed;
          const int base = sh ? 0 : itm.x * 2 * half;
          rA0 = base + itm.y * 64;
          rA1 = base + half + itm.y * 64;
        } else {
          const int base = sh ? 0 : itm.x * p.rows_routed;
          rA0 = base + itm.y * 128;
          rA1 = rA0 + 64;
        }
        const int nb = (itm.w + kBRows - 1) / kBRows;
        for (int g = 0; g < ng; ++g) {
          if (MODE != kRouter) {
            const uint32_t s = na % kQS;
            if (!ptx::mbar_wait(&bars->q_empty[s], ((na / kQS) & 1) ^ 1, abort, budget)) { stop = true; break; }
            uint8_t *dst = smem + kOffQ + s * kQBytes;
            ptx::mbar_expect_tx(&bars->q_full[s], kQBytes);
            ptx::tma_load_2d(dst, ta, g * 128, rA0, &bars->q_full[s], pol_w);
            ptx::tma_load_2d(dst + kQBytes / 2, ta, g * 128, rA1, &bars->q_full[s], pol_w);
          } else {
            const uint32_t s = na % kAS;
            if (!ptx::mbar_wait(&bars->a_empty[s], ((na / kAS) & 1) ^ 1, abort, budget)) { stop = true; break; }
            uint8_t *dst = smem + kOffA + s * kABytes;
            ptx::mbar_expect_tx(&bars->a_full[s], kABytes);
            ptx::tma_load_2d(dst, ta, g * 128, itm.y * 128, &bars->a_full[s], pol_x);
            ptx::tma_load_2d(dst + kABytes / 2, ta, g * 128 + 64, itm.y * 128, &bars->a_full[s],
                             pol_x);
          }
          ++na;
          const uint32_t sb = nb_issued % kBS;
          if (!ptx::mbar_wait(&bars->b_empty[sb], ((nb_issued / kBS) & 1) ^ 1, abort, budget)) { stop = true; break; }
          uint8_t *dst = smem + kOffB + sb * kBBytes;
          ptx::mbar_expect_tx(&bars->b_full[sb], 2u * nb * kBRows * 128);
          for (int h = 0; h < 2; ++h)
            for (int bb = 0; bb < nb; ++bb)
              ptx::tma_load_2d(dst + h * (kBBytes / 2) + bb * kBRows * 128, tb, g * 128 + h * 64,
                               itm.z + bb * kBRows, &bars->b_full[sb], pol_x);
          ++nb_issued;
        }
      }
      // After an abort, the copies still in flight must land before the CTA
      // exits: wait (bounded) for the last stages issued on each ring.
      if (*abort) {
        int never = 0;
        const uint32_t ra = MODE != kRouter ? kQS : kAS;
        for (uint32_t k = 0; k < ra && k < na; ++k) {
          const uint32_t g2 = na - 1 - k;
          uint64_t *bar = MODE != kRouter ? &bars->q_full[g2 % kQS] : &bars->a_full[g2 % kAS];
          ptx::mbar_wait(bar, (g2 / ra) & 1, &never, budget);
        }
        for (uint32_t k = 0; k < kBS && k < nb_issued; ++k) {
          const uint32_t g2 = nb_issued - 1 - k;
          ptx::mbar_wait(&bars->b_full[g2 % kBS], (g2 / kBS) & 1, &never, budget);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t gs = 0;
      bool issued = false;
      for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x) {
        const int4 itm = item_at(it);
        const int ng = groups_of(itm);
        const int n16 = (itm.w + 15) & ~15;
        const uint32_t idesc = ptx::idesc_bf16_f32(128, n16);
        for (int g = 0; g < ng; ++g, ++gs) {
          const int sa = gs % kAS, sb = gs % kBS, pb = gs & 1;
          if (!ptx::mbar_wait(&bars->a_full[sa], (gs / kAS) & 1, abort, budget)) break;
          if (!ptx::mbar_wait(&bars->b_full[sb], (gs / kBS) & 1, abort, budget)) break;
          if (!ptx::mbar_wait(&bars->p_empty[pb], ((gs >> 1) & 1) ^ 1, abort, budget)) break;
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smem + kOffA + sa * kABytes);
          const uint32_t b0 = ptx::smem_u32(smem + kOffB + sb * kBBytes);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * (kABytes / 2) + (k & 3) * 32;
            ptx::mma_bf16(tmem + pb * 128, ptx::sw128_desc(a0 + off), ptx::sw128_desc(b0 + off),
                          idesc, k > 0);
          }
          ptx::mma_commit(&bars->a_empty[sa]);
          ptx::mma_commit(&bars->b_empty[sb]);
          ptx::mma_commit(&bars->p_full[pb]);
          issued = true;
        }
      }
      if (issued) {  // all MMAs complete before TMEM is released
        ptx::mma_commit(&bars->done);
        int never = 0;
        ptx::mbar_wait(&bars->done, 0, &never, budget);
      }
    }
  } else {
    // ---------------------------------------------------------- workers
    const int wk = warp - 2;             // 0..7
    const int quarter = warp & 3;        // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;   // tile row of this thread
    const int ch = wk >> 2;              // column half / K half
    float acc[64];
    uint32_t gs_conv = 0, gs = 0;
    // conversion of step gs_conv (MODE != kRouter); returns false on abort
    auto convert = [&](uint32_t step) -> bool {
      const int s = step % kQS, sa = step % kAS;
      if (!ptx::mbar_wait(&bars->q_full[s], (step / kQS) & 1, abort, budget)) return false;
      if (!ptx::mbar_wait(&bars->a_empty[sa], ((step / kAS) & 1) ^ 1, abort, budget)) return false;
      const uint8_t *src = smem + kOffQ + s * kQBytes + r * 128;
      uint8_t *dst = smem + kOffA + sa * kABytes + ch * (kABytes / 2) + r * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = ch * 4 + u;  // int8 16-byte chunk of the row
        const uint4 q = *reinterpret_cast<const uint4 *>(src + ((c ^ (r & 7)) << 4));
        uint4 hi;
        const uint4 lo = cvt16_i8_bf16_lo(q, hi);
        *reinterpret_cast<uint4 *>(dst + (((2 * u) ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(dst + (((2 * u + 1) ^ (r & 7)) << 4)) = hi;
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&bars->a_full[sa]);
        ptx::mbar_arrive(&bars->q_empty[s]);
      }
      return true;
    };
    // flatten (item, group) for the conversion look-ahead
    int conv_it = blockIdx.x, conv_g = 0;
    auto conv_next = [&]() -> bool {  // converts the next step, if any
      if (MODE == kRouter) return true;
      if (conv_it >= n_items) return true;
      if (!convert(gs_conv)) return false;
      ++gs_conv;
      if (++conv_g == groups_of(item_at(conv_it))) { conv_g = 0; conv_it += gridDim.x; }
      return true;
    };
    bool ok = conv_next();
    uint32_t n_done = 0;  // items finished by this CTA (exchange phase)
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++n_done) {
      const int4 itm = item_at(it);
      const bool sh = itm.x == kE;
      const int ng = groups_of(itm);
      // this thread's weight row within its expert, for the group scales
      const moe_bf16 *srow = nullptr;
      if (MODE == kGateUp) {
        const int half = sh ? p.rows_shared : p.rows_routed;
        const int rr = r < 64 ? itm.y * 64 + r : half + itm.y * 64 + (r - 64);
        srow = (sh ? p.s_shared : p.s_routed + static_cast<size_t>(itm.x) * 2 * half * ng) +
               static_cast<size_t>(rr) * ng;
      } else if (MODE == kDown) {
        const int rr = itm.y * 128 + r;
        srow = (sh ? p.s_shared : p.s_routed + static_cast<size_t>(itm.x) * p.rows_routed * ng) +
               static_cast<size_t>(rr) * ng;
      }
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
      for (int g = 0; g < ng; ++g, ++gs) {
        if (!conv_next()) { ok = false; break; }
        const float sc = MODE == kRouter ? 1.0f : bf16_to_f32(srow[g]);
        const int pb = gs & 1;
        if (!ptx::mbar_wait(&bars->p_full[pb], (gs >> 1) & 1, abort, budget)) { ok = false; break; }
        ptx::tc_fence_after();
        float v[32];
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + pb * 128 + ch * 64;
        ptx::tmem_ld32(taddr, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = fmaf(sc, v[j], acc[j]);
        ptx::tmem_ld32(taddr + 32, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[32 + j] = fmaf(sc, v[j], acc[32 + j]);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->p_empty[pb]);
      }
      if (!ok) break;
      // ------------------------------------------------------ epilogue
      const int n = itm.w;
      if (MODE == kGateUp) {
        // up rows (lanes 64..127) hand their accumulators to the gate rows
        // through shared memory; both sides wait with the bounded waits
        float *xch = reinterpret_cast<float *>(smem + kOffX);
        const uint32_t par = n_done & 1;
        if (r >= 64) {
          if (!ptx::mbar_wait(&bars->xch_empty, par ^ 1, abort, budget)) break;
#pragma unroll
          for (int j = 0; j < 64; ++j) xch[(ch * 64 + j) * 64 + (r - 64)] = acc[j];
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&bars->xch_full);
        } else {
          if (!ptx::mbar_wait(&bars->xch_full, par, abort, budget)) break;
          const int Irows = sh ? p.rows_shared : p.rows_routed;
          moe_bf16 *hout = sh ? p.h_shared : p.h_routed;
          const int i = itm.y * 64 + r;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int col = ch * 64 + j;
            if (col < n) {
              const float u = xch[col * 64 + r];
              hout[static_cast<size_t>(itm.z + col) * Irows + i] = f32_to_bf16(silu_mul(acc[j], u));
            }
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&bars->xch_empty);
        }
      } else if (MODE == kDown) {
        const int nrow = itm.y * 128 + r;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int col = ch * 64 + j;
          if (col < n) {
            const int pp = itm.z + col;
            int t;
            float w;
            if (sh) { t = pp; w = p.sgate[t]; }
            else { const int ent = p.perm[pp]; t = ent >> 3; w = p.weights[ent]; }
            if (w != 0.0f) ptx::red_add_f32(p.out_acc + static_cast<size_t>(t) * p.H + nrow, w * acc[j]);
          }
        }
      } else {
        const int e = itm.y * 128 + r;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int col = ch * 64 + j;
          if (col < n) p.logits[static_cast<size_t>(itm.z + col) * kE + e] = acc[j];
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_status(p.status, MOE_DEV_TIMEOUT);
}

// ----------------------------------------------------- work-item lists

// Items: gate/up -> (e, 64-row pair tile m, first list row, n); down ->
// (e, 128-row tile m, first, n); the shared expert is e == kE with B rows
// indexed by token.  One CTA; thread e lays out expert e's items.
__global__ void build_items_kernel(const int32_t *__restrict__ offsets, int T, int I, int Is,
                                   int H, int4 *__restrict__ gu, int *__restrict__ n_gu,
                                   int4 *__restrict__ dn, int *__restrict__ n_dn) {
  __shared__ int tiles[kE + 1];
  __shared__ int base[kE + 2];
  const int e = threadIdx.x;  // 256 threads
  const int cnt = offsets[e + 1] - offsets[e];
  tiles[e] = (cnt + 127) / 128;
  __syncthreads();
  if (e == 0) {
    base[0] = 0;
    for (int i = 0; i < kE; ++i) base[i + 1] = base[i] + tiles[i];
  }
  __syncthreads();
  const int mg = I / 64, md = H / 128;
  for (int nt = 0; nt < tiles[e]; ++nt) {
    const int first = offsets[e] + nt * 128;
    const int n = min(128, cnt - nt * 128);
    for (int m = 0; m < mg; ++m) gu[(base[e] + nt) * mg + m] = make_int4(e, m, first, n);
    for (int m = 0; m < md; ++m) dn[(base[e] + nt) * md + m] = make_int4(e, m, first, n);
  }
  const int nr = base[kE];
  const int ts = Is > 0 ? (T + 127) / 128 : 0;
  const int mgs = Is / 64;
  for (int k = e; k < ts * mgs; k += blockDim.x) {
    const int nt = k / mgs, m = k % mgs;
    gu[nr * mg + k] = make_int4(kE, m, nt * 128, min(128, T - nt * 128));
  }
  for (int k = e; k < ts * md; k += blockDim.x) {
    const int nt = k / md, m = k % md;
    dn[nr * md + k] = make_int4(kE, m, nt * 128, min(128, T - nt * 128));
  }
  if (e == 0) {
    *n_gu = nr * mg + ts * mgs;
    *n_dn = nr * md + ts * md;
  }
}

// X_sorted[p] = x[perm[p] / K]: the tokens of each expert as contiguous rows.
__global__ void gather_rows_kernel(const moe_bf16 *__restrict__ x, int H,
                                   const int32_t *__restrict__ perm,
                                   const int32_t *__restrict__ offsets, moe_bf16 *__restrict__ xs) {
  const int total = offsets[kE];
  const int per_row = H / 8;  // 16-byte chunks
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < static_cast<size_t>(total) * per_row; i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int prow = static_cast<int>(i / per_row), c = static_cast<int>(i % per_row);
    const int t = perm[prow] / kK;
    reinterpret_cast<uint4 *>(xs + static_cast<size_t>(prow) * H)[c] =
        reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * H)[c];
  }
}

__global__ void acc_to_bf16_kernel(const float *__restrict__ acc, size_t n4,
                                   moe_bf16 *__restrict__ out) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4 *>(acc)[i];
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    reinterpret_cast<uint2 *>(out)[i] = o;
  }
}

// ------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D row-major tensor [rows][cols] of `esize`-byte elements, box
// [box_rows][box_cols], 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t rows,
              uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn enc = encoder();
  if (!enc || !base) return false;
  const cuuint64_t gdim[2] = {cols, rows};
  const cuuint64_t gstride[1] = {cols * static_cast<uint64_t>(esize)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void *>(base), gdim, gstride, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev] > 0 ? n[dev] : 148;
}

template <int MODE>
cudaError_t launch_tc(const CUtensorMap &a, const CUtensorMap &as, const CUtensorMap &b,
                      const CUtensorMap &bs, const TcParams &p, cudaStream_t s) {
  static bool attr[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kTcSmem));
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  tc_gemm_kernel<MODE><<<sm_count(), kTcThreads, kTcSmem, s>>>(a, as, b, bs, p);
  return cudaGetLastError();
}

unsigned long long wait_budget_ns() {
  static unsigned long long v = 0;
  if (!v) {
    const char *e = getenv("MOE_WAIT_BUDGET_NS");
    v = e ? strtoull(e, nullptr, 10) : 2000000000ull;
    if (!v) v = 1;
  }
  return v;
}

}  // namespace

size_t tc_items_bytes(int T, int I, int Is, int H) {
  const size_t tiles = static_cast<size_t>(T) * kK / 128 + kE;
  const size_t ts = (static_cast<size_t>(T) + 127) / 128;
  const size_t gu = tiles * (I / 64) + ts * (Is / 64);
  const size_t dn = tiles * (H / 128) + ts * (H / 128);
  return (gu + dn + 16) * sizeof(int4);
}

cudaError_t launch_router_tc(const moe_bf16 *x, int T, int H, const moe_bf16 *w_router,
                             float *logits, uint32_t *status, cudaStream_t s) {
  CUtensorMap a, b;
  if (!make_map(&a, w_router, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kE, H, 128, 64) ||
      !make_map(&b, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, kBRows, 64))
    return cudaErrorInvalidValue;
  TcParams p{};
  p.K_routed = p.K_shared = H;
  p.logits = logits; p.T_router = T;
  p.status = status; p.budget_ns = wait_budget_ns();
  return launch_tc<kRouter>(a, a, b, b, p, s);
}

cudaError_t launch_experts_tc(const moe_bf16 *x, int T, int H, int I, int Is,
                              const moe_weights &w, const Lists &L, const int32_t *perm,
                              const float *weights, const float *sgate, moe_bf16 *xs,
                              moe_bf16 *h_routed, moe_bf16 *h_shared, float *out_acc,
                              moe_bf16 *out, int4 *items, int *counters, uint32_t *status,
                              cudaStream_t s, StageRecorder &rec) {
#define TC_STEP(expr)                          \
  do {                                         \
    cudaError_t e_ = (expr);                   \
    if (e_ == cudaSuccess) e_ = rec();         \
    if (e_ != cudaSuccess) return e_;          \
  } while (0)
  int4 *gu = items;
  const size_t tiles = static_cast<size_t>(T) * kK / 128 + kE;
  const size_t ts = (static_cast<size_t>(T) + 127) / 128;
  int4 *dn = items + tiles * (I / 64) + ts * (Is / 64);
  build_items_kernel<<<1, kE, 0, s>>>(L.offsets, T, I, Is, H, gu, counters, dn, counters + 1);
  TC_STEP(cudaGetLastError());
  gather_rows_kernel<<<sm_count() * 4, 256, 0, s>>>(x, H, L.perm, L.offsets, xs);
  TC_STEP(cudaGetLastError());
  TC_STEP(cudaMemsetAsync(out_acc, 0, sizeof(float) * static_cast<size_t>(T) * H, s));
  const size_t rows_r = static_cast<size_t>(T) * kK;
  CUtensorMap a13, a13s, bx, bxs, a2, a2s, bh, bhs;
  const bool shared = Is > 0;
  bool ok = make_map(&a13, w.w13_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                     static_cast<uint64_t>(kE) * 2 * I, H, 64, 128) &&
            make_map(&bx, xs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows_r, H, kBRows, 64) &&
            make_map(&a2, w.w2_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                     static_cast<uint64_t>(kE) * H, I, 64, 128) &&
            make_map(&bh, h_routed, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows_r, I, kBRows, 64);
  if (shared)
    ok = ok && make_map(&a13s, w.ws13_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 2 * Is, H, 64, 128) &&
         make_map(&bxs, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, kBRows, 64) &&
         make_map(&a2s, w.ws2_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, H, Is, 64, 128) &&
         make_map(&bhs, h_shared, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, Is, kBRows, 64);
  else {
    a13s = a13; bxs = bx; a2s = a2; bhs = bh;
  }
  if (!ok) return cudaErrorInvalidValue;
  TcParams p{};
  p.items = gu; p.n_items = counters;
  p.K_routed = H; p.K_shared = H;
  p.rows_routed = I; p.rows_shared = Is;
  p.s_routed = w.w13_s; p.s_shared = w.ws13_s;
  p.h_routed = h_routed; p.h_shared = h_shared;
  p.status = status; p.budget_ns = wait_budget_ns();
  TC_STEP(launch_tc<kGateUp>(a13, a13s, bx, bxs, p, s));
  TcParams q{};
  q.items = dn; q.n_items = counters + 1;
  q.K_routed = I; q.K_shared = Is;
  q.rows_routed = H; q.rows_shared = H;
  q.s_routed = w.w2_s; q.s_shared = w.ws2_s;
  q.out_acc = out_acc; q.perm = perm; q.weights = weights; q.sgate = sgate; q.H = H;
  q.status = status; q.budget_ns = wait_budget_ns();
  TC_STEP(launch_tc<kDown>(a2, a2s, bh, bhs, q, s));
  const size_t n4 = static_cast<size_t>(T) * H / 4;
  acc_to_bf16_kernel<<<sm_count() * 4, 256, 0, s>>>(out_acc, n4, out);
  TC_STEP(cudaGetLastError());
  return cudaSuccess;
#undef TC_STEP
}

}  // namespace moe
