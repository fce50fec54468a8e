// tc_expert.cu -- prefill-size T: the expert gate|up projections with the
// SwiGLU (A4/A6), the down projection with the weighted combine (A5/A6/A7),
// the token -> expert lists and work items (A3) and the tokens' fp16 copies,
// as grouped GEMMs on the 5th-generation tensor cores with the dequantised
// weight operand held in tensor memory.
//
// Orientation: D[row, token] = sum_k W[row, k] * X[token, k].  128 weight
// rows are the M operand (one TMEM lane each), the tokens of one expert tile
// are N (<= 96): each weight tile is streamed from HBM once for all of its
// expert's tokens (an expert with more than 96 tokens gets several tiles).
//
// gate|up (gateup_split_kernel) and down + combine (down_split_kernel): the
// int8 weights times their group scales become two exact fp16 operands (the
// scale split in two, below) held in TMEM, the activations are per-row
// power-of-two scaled fp16 copies (x by scale_gather_kernel, h in place by
// h_scale_kernel), and the MMAs sum each item's whole reduction in TMEM: no
// product is rounded and no per-group partial leaves the tensor memory.
//
// Every wait is bounded by a %globaltimer budget; on expiry the CTA drains
// what it has in flight, frees TMEM, sets MOE_DEV_TIMEOUT and returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kConv = 4;                   // converter warps (one per TMEM lane quarter)
constexpr int kXTile = 96;                 // tokens per work item at most (N)
constexpr int kXQS = 6, kXBS = 4;          // shared-memory ring depths
constexpr int kXBRows = 32;                // rows per activation TMA box
constexpr uint32_t kXQBytes = 128 * 128;   // int8 weight tile
constexpr uint32_t kXBBytes = 2 * kXTile * 128;  // 16-bit activation tile (<= 96 rows), two K halves
constexpr uint32_t kXXchBytes = kXTile * 64 * 4;  // gate|up exchange of the up rows
constexpr uint32_t kXTmemCols = 512;

constexpr size_t kXOffQ = 0;
constexpr size_t kXOffB = kXOffQ + kXQS * kXQBytes;
constexpr size_t kXOffX = kXOffB + kXBS * kXBBytes;
constexpr size_t kXOffBar = kXOffX + kXXchBytes;
constexpr size_t kXSmem = kXOffBar + 512 + 1024;  // + barriers + alignment slack
static_assert(kXSmem <= 232448, "shared memory per CTA");

// Tensor maps: weights (gate|up: 3-D, the 64 gate rows and the matching 64
// up rows of a group in one copy; down: 128 rows), and activations as 3-D
// (64 elements, rows, K chunks of 64) with boxes of 32, 64 or 96 rows and two
// K chunks, so that one copy brings a group's whole activation tile.
struct XMaps {
  CUtensorMap a[2];     // routed, shared
  CUtensorMap b[2][3];  // routed, shared x box rows 32, 64, 96
};

struct XParams {
  const int4 *items;                  // {expert (kE = shared), m tile, first B row, n}
  const int *n_items;
  int K_routed, K_shared;             // reduction lengths
  int rows_routed, rows_shared;       // gate|up: I and Is; down: H for both
  const moe_bf16 *s_routed, *s_shared;  // group scales [rows][K / 128]
  // gate|up
  const float *xscale;                // [T] 2^s of each token's fp16 copy
  moe_bf16 *h_routed, *h_shared;      // [slots][I], [T][Is]
  // down
  float *out_acc;                     // [T][H] fp32 (combine mode)
  float *y_slots;                     // [T][K + 1][H] fp32, unweighted (per-slot mode), or NULL
  const float *weights, *sgate;
  int H;
  const int *perm;                    // list position -> entry t * K + j
  // h rows: routed list positions [0, T*K), shared tokens at T*K + t
  const float *hscale;                // down: 2^s of each row's fp16 copy of h
  int T8;                             // T * K
  uint32_t *status;
  unsigned long long budget_ns;
};

// ------------------------------ gate|up with the scales split (no promotion)
//
// Every bf16 group scale s = m * 2^E (m an 8-bit integer significand) is
// split as s = s_a + s_b, s_a = (m & 0xF0) * 2^E, s_b = (m & 0x0F) * 2^E.
// Then q * s_a and q * s_b (|q| <= 127) have at most 11 significant bits each
// and, scaled by a per-row power of two 2^-e (e from the row's largest group
// exponent), are exact fp16 values for every group whose scale is within
// 2^21 of the row's largest.  The weight row becomes two fp16 rows A1 = q *
// s_a * 2^-e and A2 = q * s_b * 2^-e, and the MMAs accumulate A1 x B and
// A2 x B over the whole reduction in TMEM: the products are exact and the
// scales need no promotion.  2^e (per row) and 2^s (per token) are applied to
// the fp32 sums in the epilogue.  The conversion is one fp16 FMA per pair of
// weights: with u = q + 128 placed in the mantissa of 1024 (1024 + u exact),
// (1024 + u) * s' - 1152 * s' = q * s' is rounded once, and is exact.
//
// Warp roles (480 threads): warp 0 issues the TMA copies, warp 1 the MMAs of
// A1 and warp 2 those of A2 of every K group, each into its own accumulator
// (the epilogue adds the two), warps 3..6 convert (one per TMEM lane
// quarter), warps 7..14 run the epilogue (two per lane quarter, splitting the
// token columns).
constexpr int kGThreads = 480;
constexpr int kGConv0 = 3;  // converter warps 3..6; epilogue warps 7..14
constexpr int kGAS = 2;     // TMEM A stages (one per issuer)
constexpr int kGEpi = 8;

// TMEM: A stage sa at [128 sa, 128 sa + 128): A1 in its first 64 columns, A2
// in the next 64; accumulator of issuer i at 256 + 128 i (96 wide).
__host__ __device__ constexpr uint32_t g_acol(int sa, int part) { return 128u * sa + 64u * part; }
__host__ __device__ constexpr uint32_t g_dcol(int i) { return 256u + 128u * i; }
static_assert(g_dcol(1) + kXTile <= kXTmemCols, "tensor memory columns");

struct GBars {
  uint64_t q_full[kXQS], q_empty[kXQS], a_full[kGAS], a_empty[kGAS], b_full[kXBS],
      b_empty[kXBS];
  uint64_t d_full[2], d_empty[2], done[2], xch_full, xch_empty;
  uint32_t tmem_holder;
  int abort;
};
static_assert(sizeof(GBars) <= 512, "barrier block");

// Exponent field of the largest nonzero |scale| among the row's ng groups,
// clamped so that 2^-e and 2^e below are normal floats.
__device__ __forceinline__ int row_scale_exp(const moe_bf16 *srow, int ng) {
  int ef = 0;
  for (int g = 0; g < ng; ++g) ef = max(ef, static_cast<int>((srow[g] >> 7) & 0xFF));
  return max(8, min(254, ef));
}

__global__ void __launch_bounds__(kGThreads, 1)
gateup_split_kernel(const __grid_constant__ XMaps maps, const XParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  GBars *bars = reinterpret_cast<GBars *>(smem + kXOffBar);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = *p.n_items;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kXQS; ++i) {
      ptx::mbar_init(&bars->q_full[i], 1);
      ptx::mbar_init(&bars->q_empty[i], kConv);
    }
    for (int i = 0; i < kGAS; ++i) {
      ptx::mbar_init(&bars->a_full[i], kConv);
      ptx::mbar_init(&bars->a_empty[i], 2);  // both issuers
    }
    for (int i = 0; i < kXBS; ++i) {
      ptx::mbar_init(&bars->b_full[i], 1);
      ptx::mbar_init(&bars->b_empty[i], 2);  // both issuers
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->d_full[i], 1);
      ptx::mbar_init(&bars->d_empty[i], kGEpi);
      ptx::mbar_init(&bars->done[i], 1);
    }
    ptx::mbar_init(&bars->xch_full, kGEpi / 2);   // the warps holding up rows
    ptx::mbar_init(&bars->xch_empty, kGEpi / 2);  // the warps holding gate rows
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_holder, kXTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_holder;
  const uint64_t budget = p.budget_ns;
  auto groups_of = [&](const int4 &itm) {
    return (itm.x == kE ? p.K_shared : p.K_routed) / kG;
  };
  // the scales of weight row r (0..63 gate, 64..127 up) of item itm
  auto scale_row = [&](const int4 &itm, int r, int ng) {
    const bool sh = itm.x == kE;
    const int half = sh ? p.rows_shared : p.rows_routed;
    const int rr = r < 64 ? itm.y * 64 + r : half + itm.y * 64 + (r - 64);
    return (sh ? p.s_shared : p.s_routed + static_cast<size_t>(itm.x) * 2 * half * ng) +
           static_cast<size_t>(rr) * ng;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&maps.a[0]); ptx::tma_prefetch_desc(&maps.a[1]);
      for (int i = 0; i < 3; ++i) {
        ptx::tma_prefetch_desc(&maps.b[0][i]); ptx::tma_prefetch_desc(&maps.b[1][i]);
      }
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      uint32_t nq = 0, nb = 0;
      bool stop = false;
      int4 nxt = blockIdx.x < n_items ? p.items[blockIdx.x] : make_int4(0, 0, 0, 0);
      for (int it = blockIdx.x; it < n_items && !stop; it += gridDim.x) {
        const int4 itm = nxt;  // descriptors are read one item ahead
        if (it + static_cast<int>(gridDim.x) < n_items) nxt = p.items[it + gridDim.x];
        const bool sh = itm.x == kE;
        const int ng = groups_of(itm);
        const int rA = (sh ? 0 : itm.x * 2 * p.rows_routed) + itm.y * 64;
        const int nbx = (itm.w + kXBRows - 1) / kXBRows;
        for (int g = 0; g < ng; ++g) {
          const uint32_t sq = nq % kXQS;
          if (!ptx::mbar_wait(&bars->q_empty[sq], ((nq / kXQS) & 1) ^ 1, abort, budget)) { stop = true; break; }
          ptx::mbar_expect_tx(&bars->q_full[sq], kXQBytes);
          ptx::tma_load_3d(smem + kXOffQ + sq * kXQBytes, &maps.a[sh ? 1 : 0], g * 128, rA, 0,
                           &bars->q_full[sq], pol_w);
          ++nq;
          const uint32_t sb = nb % kXBS;
          if (!ptx::mbar_wait(&bars->b_empty[sb], ((nb / kXBS) & 1) ^ 1, abort, budget)) { stop = true; break; }
          ptx::mbar_expect_tx(&bars->b_full[sb], 2u * nbx * kXBRows * 128);
          ptx::tma_load_3d(smem + kXOffB + sb * kXBBytes, &maps.b[sh ? 1 : 0][nbx - 1], 0, itm.z,
                           2 * g, &bars->b_full[sb], pol_x);
          ++nb;
        }
      }
      if (*abort) {  // let the copies in flight land before exiting
        int never = 0;
        for (uint32_t k = 0; k < kXQS && k < nq; ++k) {
          const uint32_t j = nq - 1 - k;
          ptx::mbar_wait(&bars->q_full[j % kXQS], (j / kXQS) & 1, &never, ptx::kDrainBudgetNs);
        }
        for (uint32_t k = 0; k < kXBS && k < nb; ++k) {
          const uint32_t j = nb - 1 - k;
          ptx::mbar_wait(&bars->b_full[j % kXBS], (j / kXBS) & 1, &never, ptx::kDrainBudgetNs);
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // --------------------------------- MMA issuers (A1 part, A2 part)
    if (lane == 0) {
      const int me = warp - 1;
      uint32_t gs = 0, nit = 0;
      bool issued = false;
      int4 nxt = blockIdx.x < n_items ? p.items[blockIdx.x] : make_int4(0, 0, 0, 0);
      for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x, ++nit) {
        const int4 itm = nxt;  // descriptors are read one item ahead
        if (it + static_cast<int>(gridDim.x) < n_items) nxt = p.items[it + gridDim.x];
        const int ng = groups_of(itm);
        const int n16 = (itm.w + 15) & ~15;
        const uint32_t bhalf = static_cast<uint32_t>((itm.w + kXBRows - 1) / kXBRows) * kXBRows * 128;
        const uint32_t idesc = ptx::idesc_f16_f32(128, n16);
        // the accumulator must have been read by the previous item's epilogue
        if (!ptx::mbar_wait(&bars->d_empty[me], (nit & 1) ^ 1, abort, budget)) break;
        ptx::tc_fence_after();
        bool first = true;
        for (int g = 0; g < ng; ++g, ++gs) {
          const int sa = gs % kGAS, sb = gs % kXBS;
          if (!ptx::mbar_wait(&bars->a_full[sa], (gs / kGAS) & 1, abort, budget)) break;
          if (!ptx::mbar_wait(&bars->b_full[sb], (gs / kXBS) & 1, abort, budget)) break;
          ptx::tc_fence_after();
          const uint32_t b0 = ptx::smem_u32(smem + kXOffB + sb * kXBBytes);
#pragma unroll
          for (int k = 0; k < 8; ++k) {  // K = 16 per instruction: 8 TMEM columns of A
            const uint64_t bd = ptx::sw128_desc(b0 + (k >> 2) * bhalf + (k & 3) * 32);
            ptx::mma_tmem_a(tmem + g_dcol(me), tmem + g_acol(sa, me) + k * 8, bd, idesc,
                            !(first && k == 0));
          }
          first = false;
          ptx::mma_commit(&bars->a_empty[sa]);
          ptx::mma_commit(&bars->b_empty[sb]);
          issued = true;
        }
        if (*abort) break;
        ptx::mma_commit(&bars->d_full[me]);  // this item's sums are complete
      }
      if (issued) {  // all MMAs complete before TMEM is released
        ptx::mma_commit(&bars->done[me]);
        int never = 0;
        ptx::mbar_wait(&bars->done[me], 0, &never, ptx::kDrainBudgetNs);
      }
    }
  } else if (warp < kGConv0 + kConv) {
    // ------------------------------------------------------- converters
    const int quarter = warp & 3;  // TMEM lanes 32 * quarter .. + 31
    const int r = quarter * 32 + lane;
    const uint32_t tl = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t gs = 0;
    bool ok = true;
    int4 nxt = blockIdx.x < n_items ? p.items[blockIdx.x] : make_int4(0, 0, 0, 0);
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int4 itm = nxt;  // descriptors are read one item ahead
      const int ng = groups_of(itm);
      const moe_bf16 *srow = scale_row(itm, r, ng);
      if (it + static_cast<int>(gridDim.x) < n_items) {  // the next item's scales into L1
        nxt = p.items[it + gridDim.x];
        const moe_bf16 *ns = scale_row(nxt, r, groups_of(nxt));
        asm volatile("prefetch.L1 [%0];" ::"l"(ns));
      }
      const int ef = row_scale_exp(srow, ng);
      const float down = __uint_as_float(static_cast<uint32_t>(258 - ef) << 23);  // 2^-e
      for (int g = 0; g < ng; ++g, ++gs) {
        const int sq = gs % kXQS, sa = gs % kGAS;
        // s = s_a + s_b: s_a keeps the top four significand bits of s
        const uint16_t sbits = srow[gateup_scale_group(g, ng)];
        const float s_a = bf16_to_f32(static_cast<uint16_t>(sbits & 0xFFF0u));
        const float s_b = bf16_to_f32(sbits) - s_a;
        // multipliers s' and the constants -1152 s' (all exact in fp16)
        const __half2 ha = __float2half2_rn(s_a * down), hb = __float2half2_rn(s_b * down);
        const __half2 ca = __float2half2_rn(-1152.0f * s_a * down);
        const __half2 cb = __float2half2_rn(-1152.0f * s_b * down);
        const uint32_t ha2 = *reinterpret_cast<const uint32_t *>(&ha);
        const uint32_t hb2 = *reinterpret_cast<const uint32_t *>(&hb);
        const uint32_t ca2 = *reinterpret_cast<const uint32_t *>(&ca);
        const uint32_t cb2 = *reinterpret_cast<const uint32_t *>(&cb);
        if (!ptx::mbar_wait(&bars->q_full[sq], (gs / kXQS) & 1, abort, budget)) { ok = false; break; }
        if (!ptx::mbar_wait(&bars->a_empty[sa], ((gs / kGAS) & 1) ^ 1, abort, budget)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint8_t *src = smem + kXOffQ + sq * kXQBytes + r * 128;
        uint4 q[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) q[c] = *reinterpret_cast<const uint4 *>(src + ((c ^ (r & 7)) << 4));
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t v1[32], v2[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 qc = q[4 * hf + c];
            const uint32_t w[4] = {qc.x, qc.y, qc.z, qc.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t u = w[i] ^ 0x80808080u;  // q + 128 per byte
              const uint32_t m[2] = {__byte_perm(u, 0x64646464u, 0x4140),   // 1024 + u
                                     __byte_perm(u, 0x64646464u, 0x4342)};
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(v1[8 * c + 2 * i + h])
                    : "r"(m[h]), "r"(ha2), "r"(ca2));
                asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(v2[8 * c + 2 * i + h])
                    : "r"(m[h]), "r"(hb2), "r"(cb2));
              }
            }
          }
          if (hf == 1) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars->q_empty[sq]);
          }
          ptx::tmem_st32(tmem + tl + g_acol(sa, 0) + 32 * hf, v1);
          ptx::tmem_st32(tmem + tl + g_acol(sa, 1) + 32 * hf, v2);
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->a_full[sa]);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int ch = (warp - kGConv0 - kConv) >> 2;  // column blocks ch, ch + 2, ch + 4
    const int r = quarter * 32 + lane;
    const uint32_t tl = static_cast<uint32_t>(quarter * 32) << 16;
    float acc[48];
    uint32_t nit = 0;
    int4 nxt = blockIdx.x < n_items ? p.items[blockIdx.x] : make_int4(0, 0, 0, 0);
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++nit) {
      const int4 itm = nxt;  // descriptors are read one item ahead
      if (it + static_cast<int>(gridDim.x) < n_items) nxt = p.items[it + gridDim.x];
      const bool sh = itm.x == kE;
      const int ng = groups_of(itm);
      const int n = itm.w, nblk = (n + 15) >> 4;
      const float up = __uint_as_float(
          static_cast<uint32_t>(row_scale_exp(scale_row(itm, r, ng), ng) - 4) << 23);  // 2^e
      float cs[3];  // gate rows: 2^s of the columns' tokens (lane j: column j of each block)
#pragma unroll
      for (int jb = 0; jb < 3; ++jb) {
        cs[jb] = 0.0f;
        const int cl = (ch + 2 * jb) * 16 + (lane & 15);
        if (r < 64 && cl < n) cs[jb] = p.xscale[sh ? itm.z + cl : p.perm[itm.z + cl] / kK];
      }
      if (!ptx::mbar_wait(&bars->d_full[0], nit & 1, abort, budget)) break;
      if (!ptx::mbar_wait(&bars->d_full[1], nit & 1, abort, budget)) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int jb = 0; jb < 3; ++jb) {
        const int b = ch + 2 * jb;
        if (b < nblk) {
          float v[16], w[16];
          ptx::tmem_ld16(tmem + tl + g_dcol(0) + b * 16, v);
          ptx::tmem_ld16(tmem + tl + g_dcol(1) + b * 16, w);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[jb * 16 + j] = (v[j] + w[j]) * up;
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&bars->d_empty[0]);
        ptx::mbar_arrive(&bars->d_empty[1]);
      }
      // SwiGLU: the up rows hand their sums to the gate rows through shared
      // memory; acc[jb * 16 + j] is column (ch + 2 * jb) * 16 + j of this row
      float *xch = reinterpret_cast<float *>(smem + kXOffX);
      const uint32_t par = nit & 1;
      if (r >= 64) {
        if (!ptx::mbar_wait(&bars->xch_empty, par ^ 1, abort, budget)) break;
#pragma unroll
        for (int jb = 0; jb < 3; ++jb) {
          const int b = ch + 2 * jb;
          if (b < nblk) {
#pragma unroll
            for (int j = 0; j < 16; ++j) xch[(b * 16 + j) * 64 + (r - 64)] = acc[jb * 16 + j];
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->xch_full);
      } else {
        if (!ptx::mbar_wait(&bars->xch_full, par, abort, budget)) break;
        const int Irows = sh ? p.rows_shared : p.rows_routed;
        moe_bf16 *hout = sh ? p.h_shared : p.h_routed;
        const int i = itm.y * 64 + r;
#pragma unroll
        for (int jb = 0; jb < 3; ++jb) {
          const int b = ch + 2 * jb;
          if (b < nblk) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = b * 16 + j;
              const float sj = __shfl_sync(0xFFFFFFFFu, cs[jb], j);  // lane j holds column j's
              if (col < n) {
                const float u = xch[col * 64 + r] * sj;
                hout[static_cast<size_t>(itm.z + col) * Irows + i] =
                    f32_to_bf16(silu_mul(acc[jb * 16 + j] * sj, u));
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->xch_empty);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kXTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_status(p.status, MOE_DEV_TIMEOUT);
}

// ----------------------------- down + combine with the scales split (no promotion)
//
// The same scheme as gateup_split_kernel for the down projection: the weight
// tile is 128 consecutive output rows, the activations are the h rows
// converted in place to fp16 with a power of two per row (h_scale_kernel),
// and the epilogue adds w * 2^s_h * 2^e * (A1 x h + A2 x h) to the fp32 output
// rows with vector reductions.
__global__ void __launch_bounds__(kGThreads, 1)
down_split_kernel(const __grid_constant__ XMaps maps, const XParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  GBars *bars = reinterpret_cast<GBars *>(smem + kXOffBar);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = *p.n_items;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kXQS; ++i) {
      ptx::mbar_init(&bars->q_full[i], 1);
      ptx::mbar_init(&bars->q_empty[i], kConv);
    }
    for (int i = 0; i < kGAS; ++i) {
      ptx::mbar_init(&bars->a_full[i], kConv);
      ptx::mbar_init(&bars->a_empty[i], 2);  // both issuers
    }
    for (int i = 0; i < kXBS; ++i) {
      ptx::mbar_init(&bars->b_full[i], 1);
      ptx::mbar_init(&bars->b_empty[i], 2);  // both issuers
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->d_full[i], 1);
      ptx::mbar_init(&bars->d_empty[i], kGEpi);
      ptx::mbar_init(&bars->done[i], 1);
    }
    ptx::mbar_init(&bars->xch_full, kGEpi / 2);   // the warps holding up rows
    ptx::mbar_init(&bars->xch_empty, kGEpi / 2);  // the warps holding gate rows
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_holder, kXTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_holder;
  const uint64_t budget = p.budget_ns;
  auto groups_of = [&](const int4 &itm) {
    return (itm.x == kE ? p.K_shared : p.K_routed) / kG;
  };
  // the scales of output row r of item itm's 128-row tile
  auto scale_row = [&](const int4 &itm, int r, int ng) {
    const bool sh = itm.x == kE;
    return (sh ? p.s_shared : p.s_routed + static_cast<size_t>(itm.x) * p.rows_routed * ng) +
           static_cast<size_t>(itm.y * 128 + r) * ng;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&maps.a[0]); ptx::tma_prefetch_desc(&maps.a[1]);
      for (int i = 0; i < 3; ++i) {
        ptx::tma_prefetch_desc(&maps.b[0][i]); ptx::tma_prefetch_desc(&maps.b[1][i]);
      }
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      uint32_t nq = 0, nb = 0;
      bool stop = false;
      int4 nxt = blockIdx.x < n_items ? p.items[blockIdx.x] : make_int4(0, 0, 0, 0);
      for (int it = blockIdx.x; it < n_items && !stop; it += gridDim.x) {
        const int4 itm = nxt;  // descriptors are read one item ahead
        if (it + static_cast<int>(gridDim.x) < n_items) nxt = p.items[it + gridDim.x];
        const bool sh = itm.x == kE;
        const int ng = groups_of(itm);
        const int rA = (sh ? 0 : itm.x * p.rows_routed) + itm.y * 128;
        const int nbx = (itm.w + kXBRows - 1) / kXBRows;
        for (int g = 0; g < ng; ++g) {
          const uint32_t sq = nq % kXQS;
          if (!ptx::mbar_wait(&bars->q_empty[sq], ((nq / kXQS) & 1) ^ 1, abort, budget)) { stop = true; break; }
          ptx::mbar_expect_tx(&bars->q_full[sq], kXQBytes);
          ptx::tma_load_2d(smem + kXOffQ + sq * kXQBytes, &maps.a[sh ? 1 : 0], g * 128, rA,
                           &bars->q_full[sq], pol_w);
          ++nq;
          const uint32_t sb = nb % kXBS;
          if (!ptx::mbar_wait(&bars->b_empty[sb], ((nb / kXBS) & 1) ^ 1, abort, budget)) { stop = true; break; }
          ptx::mbar_expect_tx(&bars->b_full[sb], 2u * nbx * kXBRows * 128);
          ptx::tma_load_3d(smem + kXOffB + sb * kXBBytes, &maps.b[sh ? 1 : 0][nbx - 1], 0, itm.z,
                           2 * g, &bars->b_full[sb], pol_x);
          ++nb;
        }
      }
      if (*abort) {  // let the copies in flight land before exiting
        int never = 0;
        for (uint32_t k = 0; k < kXQS && k < nq; ++k) {
          const uint32_t j = nq - 1 - k;
          ptx::mbar_wait(&bars->q_full[j % kXQS], (j / kXQS) & 1, &never, ptx::kDrainBudgetNs);
        }
        for (uint32_t k = 0; k < kXBS && k < nb; ++k) {
          const uint32_t j = nb - 1 - k;
          ptx::mbar_wait(&bars->b_full[j % kXBS], (j / kXBS) & 1, &never, ptx::kDrainBudgetNs);
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // --------------------------------- MMA issuers (A1 part, A2 part)
    if (lane == 0) {
      const int me = warp - 1;
      uint32_t gs = 0, nit = 0;
      bool issued = false;
      int4 nxt = blockIdx.x < n_items ? p.items[blockIdx.x] : make_int4(0, 0, 0, 0);
      for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x, ++nit) {
        const int4 itm = nxt;  // descriptors are read one item ahead
        if (it + static_cast<int>(gridDim.x) < n_items) nxt = p.items[it + gridDim.x];
        const int ng = groups_of(itm);
        const int n16 = (itm.w + 15) & ~15;
        const uint32_t bhalf = static_cast<uint32_t>((itm.w + kXBRows - 1) / kXBRows) * kXBRows * 128;
        const uint32_t idesc = ptx::idesc_f16_f32(128, n16);
        // the accumulator must have been read by the previous item's epilogue
        if (!ptx::mbar_wait(&bars->d_empty[me], (nit & 1) ^ 1, abort, budget)) break;
        ptx::tc_fence_after();
        bool first = true;
        for (int g = 0; g < ng; ++g, ++gs) {
          const int sa = gs % kGAS, sb = gs % kXBS;
          if (!ptx::mbar_wait(&bars->a_full[sa], (gs / kGAS) & 1, abort, budget)) break;
          if (!ptx::mbar_wait(&bars->b_full[sb], (gs / kXBS) & 1, abort, budget)) break;
          ptx::tc_fence_after();
          const uint32_t b0 = ptx::smem_u32(smem + kXOffB + sb * kXBBytes);
#pragma unroll
          for (int k = 0; k < 8; ++k) {  // K = 16 per instruction: 8 TMEM columns of A
            const uint64_t bd = ptx::sw128_desc(b0 + (k >> 2) * bhalf + (k & 3) * 32);
            ptx::mma_tmem_a(tmem + g_dcol(me), tmem + g_acol(sa, me) + k * 8, bd, idesc,
                            !(first && k == 0));
          }
          first = false;
          ptx::mma_commit(&bars->a_empty[sa]);
          ptx::mma_commit(&bars->b_empty[sb]);
          issued = true;
        }
        if (*abort) break;
        ptx::mma_commit(&bars->d_full[me]);  // this item's sums are complete
      }
      if (issued) {  // all MMAs complete before TMEM is released
        ptx::mma_commit(&bars->done[me]);
        int never = 0;
        ptx::mbar_wait(&bars->done[me], 0, &never, ptx::kDrainBudgetNs);
      }
    }
  } else if (warp < kGConv0 + kConv) {
    // ------------------------------------------------------- converters
    const int quarter = warp & 3;  // TMEM lanes 32 * quarter .. + 31
    const int r = quarter * 32 + lane;
    const uint32_t tl = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t gs = 0;
    bool ok = true;
    int4 nxt = blockIdx.x < n_items ? p.items[blockIdx.x] : make_int4(0, 0, 0, 0);
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int4 itm = nxt;  // descriptors are read one item ahead
      const int ng = groups_of(itm);
      const moe_bf16 *srow = scale_row(itm, r, ng);
      if (it + static_cast<int>(gridDim.x) < n_items) {  // the next item's scales into L1
        nxt = p.items[it + gridDim.x];
        const moe_bf16 *ns = scale_row(nxt, r, groups_of(nxt));
        asm volatile("prefetch.L1 [%0];" ::"l"(ns));
      }
      const int ef = row_scale_exp(srow, ng);
      const float down = __uint_as_float(static_cast<uint32_t>(258 - ef) << 23);  // 2^-e
      for (int g = 0; g < ng; ++g, ++gs) {
        const int sq = gs % kXQS, sa = gs % kGAS;
        // s = s_a + s_b: s_a keeps the top four significand bits of s
        const uint16_t sbits = srow[g];
        const float s_a = bf16_to_f32(static_cast<uint16_t>(sbits & 0xFFF0u));
        const float s_b = bf16_to_f32(sbits) - s_a;
        // multipliers s' and the constants -1152 s' (all exact in fp16)
        const __half2 ha = __float2half2_rn(s_a * down), hb = __float2half2_rn(s_b * down);
        const __half2 ca = __float2half2_rn(-1152.0f * s_a * down);
        const __half2 cb = __float2half2_rn(-1152.0f * s_b * down);
        const uint32_t ha2 = *reinterpret_cast<const uint32_t *>(&ha);
        const uint32_t hb2 = *reinterpret_cast<const uint32_t *>(&hb);
        const uint32_t ca2 = *reinterpret_cast<const uint32_t *>(&ca);
        const uint32_t cb2 = *reinterpret_cast<const uint32_t *>(&cb);
        if (!ptx::mbar_wait(&bars->q_full[sq], (gs / kXQS) & 1, abort, budget)) { ok = false; break; }
        if (!ptx::mbar_wait(&bars->a_empty[sa], ((gs / kGAS) & 1) ^ 1, abort, budget)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint8_t *src = smem + kXOffQ + sq * kXQBytes + r * 128;
        uint4 q[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) q[c] = *reinterpret_cast<const uint4 *>(src + ((c ^ (r & 7)) << 4));
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t v1[32], v2[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 qc = q[4 * hf + c];
            const uint32_t w[4] = {qc.x, qc.y, qc.z, qc.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t u = w[i] ^ 0x80808080u;  // q + 128 per byte
              const uint32_t m[2] = {__byte_perm(u, 0x64646464u, 0x4140),   // 1024 + u
                                     __byte_perm(u, 0x64646464u, 0x4342)};
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(v1[8 * c + 2 * i + h])
                    : "r"(m[h]), "r"(ha2), "r"(ca2));
                asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(v2[8 * c + 2 * i + h])
                    : "r"(m[h]), "r"(hb2), "r"(cb2));
              }
            }
          }
          if (hf == 1) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars->q_empty[sq]);
          }
          ptx::tmem_st32(tmem + tl + g_acol(sa, 0) + 32 * hf, v1);
          ptx::tmem_st32(tmem + tl + g_acol(sa, 1) + 32 * hf, v2);
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->a_full[sa]);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int ch = (warp - kGConv0 - kConv) >> 2;  // column blocks ch, ch + 2, ch + 4
    const int r = quarter * 32 + lane;
    const uint32_t tl = static_cast<uint32_t>(quarter * 32) << 16;
    float acc[48];
    uint32_t nit = 0;
    int4 nxt = blockIdx.x < n_items ? p.items[blockIdx.x] : make_int4(0, 0, 0, 0);
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++nit) {
      const int4 itm = nxt;  // descriptors are read one item ahead
      if (it + static_cast<int>(gridDim.x) < n_items) nxt = p.items[it + gridDim.x];
      const bool sh = itm.x == kE;
      const int ng = groups_of(itm);
      const int n = itm.w, nblk = (n + 15) >> 4;
      const float up = __uint_as_float(
          static_cast<uint32_t>(row_scale_exp(scale_row(itm, r, ng), ng) - 4) << 23);  // 2^e
      // the columns' token and combine weight (the h row's 2^s included;
      // lane j: column j of each block)
      float cs[3];
      int ct[3];
#pragma unroll
      for (int jb = 0; jb < 3; ++jb) {
        cs[jb] = 0.0f;
        ct[jb] = 0;
        const int cl = (ch + 2 * jb) * 16 + (lane & 15);
        if (cl < n) {
          // combine mode: the token's output row and w * 2^s; per-slot mode:
          // the slot's y row (t * (K + 1) + j, the shared expert at j = K)
          // and 2^s alone
          if (sh) {
            const int t = itm.z + cl;
            ct[jb] = p.y_slots ? t * (kK + 1) + kK : t;
            cs[jb] = (p.y_slots ? 1.0f : (p.sgate ? p.sgate[t] : 0.0f)) * p.hscale[p.T8 + t];
          } else {
            const int ent = p.perm[itm.z + cl];
            ct[jb] = p.y_slots ? ent + ent / kK : ent / kK;
            cs[jb] = (p.y_slots ? 1.0f : p.weights[ent]) * p.hscale[itm.z + cl];
          }
        }
      }
      if (!ptx::mbar_wait(&bars->d_full[0], nit & 1, abort, budget)) break;
      if (!ptx::mbar_wait(&bars->d_full[1], nit & 1, abort, budget)) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int jb = 0; jb < 3; ++jb) {
        const int b = ch + 2 * jb;
        if (b < nblk) {
          float v[16], w[16];
          ptx::tmem_ld16(tmem + tl + g_dcol(0) + b * 16, v);
          ptx::tmem_ld16(tmem + tl + g_dcol(1) + b * 16, w);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[jb * 16 + j] = (v[j] + w[j]) * up;
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&bars->d_empty[0]);
        ptx::mbar_arrive(&bars->d_empty[1]);
      }
      // Weighted combine, out_acc[t][row] += w * acc: a 4 x 4 transpose
      // among each four lanes leaves every lane four consecutive rows of one
      // column, added with one 16-byte reduction.
      {
        const int q4 = lane & 3;
        const bool lo2 = (q4 & 2) == 0, odd = (q4 & 1) != 0;
        const int nrow4 = itm.y * 128 + quarter * 32 + (lane & ~3);
#pragma unroll
        for (int jb = 0; jb < 3; ++jb) {
          const int b = ch + 2 * jb;
          if (b < nblk) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const float *v = &acc[jb * 16 + c4 * 4];  // this row, columns c4*4 .. +3
              const float r0 = __shfl_xor_sync(0xFFFFFFFFu, lo2 ? v[2] : v[0], 2);
              const float r1 = __shfl_xor_sync(0xFFFFFFFFu, lo2 ? v[3] : v[1], 2);
              const float x0 = lo2 ? v[0] : r0, x1 = lo2 ? v[1] : r1;
              const float x2 = lo2 ? r0 : v[2], x3 = lo2 ? r1 : v[3];
              const float p0 = __shfl_xor_sync(0xFFFFFFFFu, odd ? x0 : x1, 1);
              const float p1 = __shfl_xor_sync(0xFFFFFFFFu, odd ? x2 : x3, 1);
              const float y0 = odd ? p0 : x0, y1 = odd ? x1 : p0;
              const float y2 = odd ? p1 : x2, y3 = odd ? x3 : p1;
              const int j = c4 * 4 + q4;  // this lane's column now, rows nrow4 .. +3
              const int tj = __shfl_sync(0xFFFFFFFFu, ct[jb], j);
              const float wj = __shfl_sync(0xFFFFFFFFu, cs[jb], j);
              if (b * 16 + j < n && wj != 0.0f) {
                if (p.y_slots)  // each (slot, row) is written by exactly one item
                  *reinterpret_cast<float4 *>(p.y_slots + static_cast<size_t>(tj) * p.H + nrow4) =
                      make_float4(wj * y0, wj * y1, wj * y2, wj * y3);
                else
                  ptx::red_add_v4_f32(p.out_acc + static_cast<size_t>(tj) * p.H + nrow4, wj * y0,
                                      wj * y1, wj * y2, wj * y3);
              }
            }
          }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kXTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_status(p.status, MOE_DEV_TIMEOUT);
}

// ------------------------------------ token -> expert lists, work items

// One CTA per expert e (grid kE, kLiThreads threads).  Every CTA reads the
// per-expert counts of the selection (so it knows the offsets of the experts
// before it), then compacts the entries with ids == e in entry order, which
// yields the list sorted by (e, t, j) as the one-CTA counting sort does, and
// lays out e's work items: gate|up -> (e, 64-row pair tile m, first list row, n), down ->
// (e, 128-row tile m, first, n).  CTA 0 also writes the shared expert's items
// (e == kE, B rows indexed by token), the item totals and slot_of = -1 for
// entries that name no expert.
constexpr int kLiThreads = 1024;
constexpr int kLiPer = 8;  // entries per thread and pass (two CTAs of 1024 threads per SM)

__global__ void __launch_bounds__(kLiThreads, 2)
lists_items_kernel(const int32_t *__restrict__ ids, int T, Lists L, int I, int Is, int H,
                   int4 *__restrict__ gu, int *__restrict__ n_gu, int4 *__restrict__ dn,
                   int *__restrict__ n_dn) {
  __shared__ int hist[kE];
  __shared__ int pre[kE], tpre[kE];
  __shared__ int scan_tmp[32];
  __shared__ int run;
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = T * kK;
  if (tid < kE) hist[tid] = L.counts[tid];  // from the selection kernel
  if (tid == 0) run = 0;
  __syncthreads();
  const int c = tid < kE ? hist[tid] : 0;
  const int off = block_exclusive_scan_256(c, scan_tmp);
  const int tl = block_exclusive_scan_256((c + kXTile - 1) / kXTile, scan_tmp);
  if (tid < kE) { pre[tid] = off; tpre[tid] = tl; }
  __syncthreads();
  const int cnt = hist[e], base = pre[e];
  if (tid == 0) {
    L.offsets[e] = base;
    if (e == kE - 1) L.offsets[kE] = base + cnt;
  }
  // ordered compaction: thread tid takes entries i0 + tid * kLiPer + u
  for (int i0 = 0; i0 < n && cnt > 0; i0 += kLiThreads * kLiPer) {
    int v[kLiPer];
    int m = 0;
#pragma unroll
    for (int u = 0; u < kLiPer; ++u) {
      const int i = i0 + tid * kLiPer + u;
      v[u] = i < n ? ids[i] : -1;
      m += v[u] == e;
    }
    // exclusive scan of m over the block, in thread order
    int incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) scan_tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = scan_tmp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += y;
      }
      scan_tmp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int pos = base + run + (warp > 0 ? scan_tmp[warp - 1] : 0) + incl - m;
#pragma unroll
    for (int u = 0; u < kLiPer; ++u) {
      if (v[u] == e) {
        const int i = i0 + tid * kLiPer + u;
        L.perm[pos] = i;
        if (L.slot_of) L.slot_of[i] = pos;
        ++pos;
      }
    }
    __syncthreads();
    if (tid == 0) run += scan_tmp[31];
    __syncthreads();
  }
  if (e == 0 && L.slot_of) {  // entries that name no expert get no slot
    for (int i = tid; i < n; i += kLiThreads) {
      const int x = ids[i];
      if (x < 0 || x >= kE) L.slot_of[i] = -1;
    }
  }
  // work items of expert e
  const int mg = I / 64, md = H / 128;
  const int tiles = (cnt + kXTile - 1) / kXTile, tb = tpre[e];
  for (int k = tid; k < tiles * (mg + md); k += kLiThreads) {
    const int nt = k / (mg + md), m = k % (mg + md);
    const int first = base + nt * kXTile, nn = min(kXTile, cnt - nt * kXTile);
    if (m < mg) gu[(tb + nt) * mg + m] = make_int4(e, m, first, nn);
    else dn[(tb + nt) * md + (m - mg)] = make_int4(e, m - mg, first, nn);
  }
  if (e == 0) {
    const int nr = tpre[kE - 1] + (hist[kE - 1] + kXTile - 1) / kXTile;  // all routed tiles
    const int ts = Is > 0 ? (T + kXTile - 1) / kXTile : 0;
    const int mgs = Is / 64;
    for (int k = tid; k < ts * mgs; k += kLiThreads) {
      const int nt = k / mgs, m = k % mgs;
      gu[nr * mg + k] = make_int4(kE, m, nt * kXTile, min(kXTile, T - nt * kXTile));
    }
    for (int k = tid; k < ts * md; k += kLiThreads) {
      const int nt = k / md, m = k % md;
      dn[nr * md + k] = make_int4(kE, m, nt * kXTile, min(kXTile, T - nt * kXTile));
    }
    if (tid == 0) {
      *n_gu = nr * mg + ts * mgs;
      *n_dn = nr * md + ts * md;
    }
  }
}

// The gate|up activation operand in fp16, one warp per token t: the token
// times 2^-s, with 2^s chosen per token so that its largest magnitude lands
// in [2^14, 2^15) (every element within 2^29 of that largest is then exact
// in fp16), written to x16[t] (the shared expert's operand) and to row p of
// xs16 for each list position p = slot_of[t * K + j] of the token (the routed
// experts' operand).  2^s is kept in xscale[t]; the token's fp32 output row
// is zeroed for the combine's reductions (when out_acc is given).
constexpr int kGatherMaxChunks = 8;  // 16-byte chunks per lane held in registers (H <= 2048)

__global__ void scale_gather_kernel(const moe_bf16 *__restrict__ x, int T, int H,
                                    const int32_t *__restrict__ slot_of, uint16_t *__restrict__ xs16,
                                    uint16_t *__restrict__ x16, float *__restrict__ xscale,
                                    float *__restrict__ out_acc) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const moe_bf16 *xr = x + static_cast<size_t>(t) * H;
  // 16-byte chunk c of this lane holds elements c * 256 + lane * 8 .. + 7; H
  // is a multiple of 128, so the last chunk may cover only half the lanes
  const int nc = (H + 255) / 256;
  const bool in_regs = nc <= kGatherMaxChunks;
  auto valid = [&](int c) { return c * 256 + lane * 8 < H; };
  uint4 v[kGatherMaxChunks];
  float m = 0.0f;
  auto absmax = [&](const uint4 &q) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  };
  if (in_regs) {
#pragma unroll
    for (int c = 0; c < kGatherMaxChunks; ++c)
      if (valid(c)) v[c] = ld_nc(xr + c * 256 + lane * 8);
#pragma unroll
    for (int c = 0; c < kGatherMaxChunks; ++c)
      if (valid(c)) absmax(v[c]);
  } else {
    for (int c = 0; c < nc; ++c)
      if (valid(c)) absmax(ld_nc(xr + c * 256 + lane * 8));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  int sexp = 0;
  if (m > 0.0f && isfinite(m)) {
    sexp = static_cast<int>((__float_as_uint(m) >> 23) & 0xFF) - 127 - 14;
    sexp = max(-110, min(110, sexp));
  }
  const float down = __uint_as_float(static_cast<uint32_t>(127 - sexp) << 23);  // 2^-s
  int pos[kK];
#pragma unroll
  for (int j = 0; j < kK; ++j) pos[j] = slot_of[static_cast<size_t>(t) * kK + j];
  auto emit = [&](int c, const uint4 &q) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(bf16_lo(w[i]) * down, bf16_hi(w[i]) * down);
      o[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
    const int k = c * 256 + lane * 8;
    *reinterpret_cast<uint4 *>(x16 + static_cast<size_t>(t) * H + k) = ov;
#pragma unroll
    for (int j = 0; j < kK; ++j)
      if (pos[j] >= 0) *reinterpret_cast<uint4 *>(xs16 + static_cast<size_t>(pos[j]) * H + k) = ov;
  };
  if (in_regs) {
#pragma unroll
    for (int c = 0; c < kGatherMaxChunks; ++c)
      if (valid(c)) emit(c, v[c]);
  } else {
    for (int c = 0; c < nc; ++c)
      if (valid(c)) emit(c, ld_nc(xr + c * 256 + lane * 8));
  }
  if (out_acc) {
    float4 *orow = reinterpret_cast<float4 *>(out_acc + static_cast<size_t>(t) * H);
    for (int k = lane; k < H / 4; k += 32) orow[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  if (lane == 0) xscale[t] = __uint_as_float(static_cast<uint32_t>(127 + sexp) << 23);
}

// h in place from bf16 to fp16 for the down projection: row p (a routed list
// position p < S, or the shared expert's token t at S + t) is multiplied by
// 2^-s with 2^s chosen from the row's largest |h| as for the tokens, so every
// element within 2^29 of that largest is exact; 2^s is kept in hscale
// (routed at p, shared at T*K + t).  One warp per row, held in registers.
constexpr int kHMaxChunks = 8;  // 16-byte chunks per lane (rows of up to 2048)

__global__ void h_scale_kernel(moe_bf16 *__restrict__ h_routed, int I, moe_bf16 *__restrict__ h_shared,
                               int Is, const int32_t *__restrict__ offsets, int T,
                               float *__restrict__ hscale) {
  const int S = offsets[kE];
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= S + (Is > 0 ? T : 0)) return;
  const bool sh = row >= S;
  const size_t idx = sh ? static_cast<size_t>(T) * kK + (row - S) : static_cast<size_t>(row);
  const int len = sh ? Is : I;
  moe_bf16 *hr = sh ? h_shared + static_cast<size_t>(row - S) * Is : h_routed + static_cast<size_t>(row) * I;
  // 16-byte chunk c of this lane holds elements c * 256 + lane * 8 .. + 7;
  // len is a multiple of 128, so the last chunk may cover only half the lanes
  auto valid = [&](int c) { return c * 256 + lane * 8 < len; };
  uint4 v[kHMaxChunks];
  float m = 0.0f;
#pragma unroll
  for (int c = 0; c < kHMaxChunks; ++c)
    if (valid(c)) v[c] = *reinterpret_cast<const uint4 *>(hr + c * 256 + lane * 8);
#pragma unroll
  for (int c = 0; c < kHMaxChunks; ++c)
    if (valid(c)) {
      const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  int sexp = 0;
  if (m > 0.0f && isfinite(m)) {
    sexp = static_cast<int>((__float_as_uint(m) >> 23) & 0xFF) - 127 - 14;
    sexp = max(-110, min(110, sexp));
  }
  const float down = __uint_as_float(static_cast<uint32_t>(127 - sexp) << 23);
#pragma unroll
  for (int c = 0; c < kHMaxChunks; ++c)
    if (valid(c)) {
      const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 hh = __floats2half2_rn(bf16_lo(w[i]) * down, bf16_hi(w[i]) * down);
        o[i] = *reinterpret_cast<const uint32_t *>(&hh);
      }
      *reinterpret_cast<uint4 *>(hr + c * 256 + lane * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  if (lane == 0) hscale[idx] = __uint_as_float(static_cast<uint32_t>(127 + sexp) << 23);
}

// Per-expert entry counts of ids [n] (the lists' input when no selection
// kernel counted them): a shared-memory histogram per CTA, added into
// counts (zeroed before the launch).  Ids >= kE are skipped and set
// MOE_DEV_BAD_EXPERT; negative ids are skipped.
__global__ void expert_counts_kernel(const int32_t *__restrict__ ids, int n,
                                     int32_t *__restrict__ counts, uint32_t *status) {
  __shared__ int hist[kE];
  for (int i = threadIdx.x; i < kE; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int e = ids[i];
    if (e >= kE) bad = true;
    else if (e >= 0) atomicAdd(&hist[e], 1);
  }
  if (bad) set_status(status, MOE_DEV_BAD_EXPERT);
  __syncthreads();
  for (int i = threadIdx.x; i < kE; i += blockDim.x)
    if (hist[i]) atomicAdd(counts + i, hist[i]);
}

// out = bf16(acc (+ resid)), four elements per thread and step; resid (the
// residual, bf16, may be the same buffer as out) is added before the one
// rounding.
__global__ void acc_to_bf16_kernel(const float *__restrict__ acc, size_t n4,
                                   const moe_bf16 *resid, moe_bf16 *out) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n4;
       i0 += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u * stride < n4) v[u] = __ldcg(reinterpret_cast<const float4 *>(acc) + i0 + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u * stride < n4) {
        if (resid) {
          const uint2 r = reinterpret_cast<const uint2 *>(resid)[i0 + u * stride];
          v[u].x += bf16_lo(r.x); v[u].y += bf16_hi(r.x);
          v[u].z += bf16_lo(r.y); v[u].w += bf16_hi(r.y);
        }
        uint2 o;
        o.x = pack_bf16x2(v[u].x, v[u].y);
        o.y = pack_bf16x2(v[u].z, v[u].w);
        reinterpret_cast<uint2 *>(out)[i0 + u * stride] = o;
      }
  }
}

cudaError_t launch_gateup_split(const XMaps &maps, const XParams &p, cudaStream_t s) {
  static bool attr[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gateup_split_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kXSmem));
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  gateup_split_kernel<<<tc_sm_count(), kGThreads, kXSmem, s>>>(maps, p);
  return cudaGetLastError();
}

cudaError_t launch_down_split(const XMaps &maps, const XParams &p, cudaStream_t s) {
  static bool attr[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(down_split_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kXSmem));
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  down_split_kernel<<<tc_sm_count(), kGThreads, kXSmem, s>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_counts(const int32_t *ids, int T, int32_t *counts, uint32_t *status,
                                 cudaStream_t s) {
  const int n = T * kK;
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * kE, s);
  if (e != cudaSuccess) return e;
  const int grid = min(tc_sm_count(), (n + 4095) / 4096);
  expert_counts_kernel<<<grid, 1024, 0, s>>>(ids, n, counts, status);
  return cudaGetLastError();
}

size_t tc_items_bytes(int T, int I, int Is, int H) {
  const size_t tiles = static_cast<size_t>(T) * kK / kXTile + kE;
  const size_t ts = (static_cast<size_t>(T) + kXTile - 1) / kXTile;
  const size_t gu = tiles * (I / 64) + ts * (Is / 64);
  const size_t dn = tiles * (H / 128) + ts * (H / 128);
  return (gu + dn + 16) * sizeof(int4);
}

cudaError_t launch_experts_tc(const moe_bf16 *x, int T, int H, int I, int Is,
                              const moe_weights &w, const int32_t *ids, const Lists &L,
                              const float *weights,
                              const float *sgate, uint16_t *xs16, uint16_t *x16, float *xscale,
                              float *hscale,
                              moe_bf16 *h_routed, moe_bf16 *h_shared, float *out_acc,
                              moe_bf16 *out, int4 *items, int *counters, uint32_t *status,
                              cudaStream_t s, StageRecorder &rec, float *y_slots,
                              const moe_bf16 *resid) {
#define TC_STEP(expr)                          \
  do {                                         \
    cudaError_t e_ = (expr);                   \
    if (e_ == cudaSuccess) e_ = rec();         \
    if (e_ != cudaSuccess) return e_;          \
  } while (0)
  int4 *gu = items;
  const size_t tiles = static_cast<size_t>(T) * kK / kXTile + kE;
  const size_t ts = (static_cast<size_t>(T) + kXTile - 1) / kXTile;
  int4 *dn = items + tiles * (I / 64) + ts * (Is / 64);
  lists_items_kernel<<<kE, kLiThreads, 0, s>>>(ids, T, L, I, Is, H, gu, counters, dn,
                                              counters + 1);
  TC_STEP(cudaGetLastError());
  scale_gather_kernel<<<(T + 7) / 8, 256, 0, s>>>(x, T, H, L.slot_of, xs16, x16, xscale,
                                                   y_slots ? nullptr : out_acc);
  TC_STEP(cudaGetLastError());
  const size_t rows_r = static_cast<size_t>(T) * kK;
  // Activation maps: (64 elements, rows, K / 64 chunks), chunk stride 128 B,
  // boxes (64, 32 * i, 2).
  auto act_maps = [&](CUtensorMap (&m)[3], const void *base, CUtensorMapDataType dt,
                      uint64_t rows, uint64_t K) {
    const uint64_t dims[3] = {64, rows, K / 64};
    const uint64_t strides[2] = {K * 2, 128};
    bool ok = true;
    for (int i = 0; i < 3; ++i) {
      const uint32_t box[3] = {64, static_cast<uint32_t>(kXBRows * (i + 1)), 2};
      ok = ok && tc_make_map3(&m[i], base, dt, 2, dims, strides, box);
    }
    return ok;
  };
  XMaps gm{}, dm{};
  const bool shared = Is > 0;
  bool ok;
  {  // gate|up weights: (H, rows, gate|up) with the up rows I rows after the gate rows
    const uint64_t dims[3] = {static_cast<uint64_t>(H), static_cast<uint64_t>(kE) * 2 * I, 2};
    const uint64_t strides[2] = {static_cast<uint64_t>(H), static_cast<uint64_t>(I) * H};
    const uint32_t box[3] = {128, 64, 2};
    ok = tc_make_map3(&gm.a[0], w.w13_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dims, strides, box);
  }
  ok = ok && act_maps(gm.b[0], xs16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rows_r, H) &&
       tc_make_map(&dm.a[0], w.w2_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                   static_cast<uint64_t>(kE) * H, I, 128, 128) &&
       act_maps(dm.b[0], h_routed, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rows_r, I);
  if (shared) {
    const uint64_t dims[3] = {static_cast<uint64_t>(H), 2 * static_cast<uint64_t>(Is), 2};
    const uint64_t strides[2] = {static_cast<uint64_t>(H), static_cast<uint64_t>(Is) * H};
    const uint32_t box[3] = {128, 64, 2};
    ok = ok && tc_make_map3(&gm.a[1], w.ws13_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dims, strides,
                            box) &&
         act_maps(gm.b[1], x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, T, H) &&
         tc_make_map(&dm.a[1], w.ws2_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, H, Is, 128, 128) &&
         act_maps(dm.b[1], h_shared, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, T, Is);
  } else {
    gm.a[1] = gm.a[0]; dm.a[1] = dm.a[0];
    for (int i = 0; i < 3; ++i) { gm.b[1][i] = gm.b[0][i]; dm.b[1][i] = dm.b[0][i]; }
  }
  if (!ok) return cudaErrorInvalidValue;
  XParams p{};
  p.items = gu; p.n_items = counters;
  p.K_routed = H; p.K_shared = H;
  p.rows_routed = I; p.rows_shared = Is;
  p.s_routed = w.w13_s; p.s_shared = w.ws13_s;
  p.xscale = xscale; p.perm = L.perm;
  p.h_routed = h_routed; p.h_shared = h_shared;
  p.T8 = T * kK;
  p.status = status; p.budget_ns = tc_wait_budget_ns();
  TC_STEP(launch_gateup_split(gm, p, s));
  {
    const int rows = T * kK + (Is > 0 ? T : 0);  // at most; the kernel reads the count
    h_scale_kernel<<<(rows + 7) / 8, 256, 0, s>>>(h_routed, I, h_shared, Is, L.offsets, T,
                                                  hscale);
    TC_STEP(cudaGetLastError());
  }
  XParams q{};
  q.items = dn; q.n_items = counters + 1;
  q.K_routed = I; q.K_shared = Is;
  q.rows_routed = H; q.rows_shared = H;
  q.s_routed = w.w2_s; q.s_shared = w.ws2_s;
  q.out_acc = out_acc; q.y_slots = y_slots;
  q.perm = L.perm; q.weights = weights; q.sgate = sgate; q.H = H;
  q.hscale = hscale; q.T8 = T * kK;
  q.status = status; q.budget_ns = tc_wait_budget_ns();
  TC_STEP(launch_down_split(dm, q, s));
  if (y_slots) return cudaSuccess;
  const size_t n4 = static_cast<size_t>(T) * H / 4;
  acc_to_bf16_kernel<<<tc_sm_count() * 4, 256, 0, s>>>(out_acc, n4, resid, out);
  TC_STEP(cudaGetLastError());
  return cudaSuccess;
#undef TC_STEP
}

}  // namespace moe
