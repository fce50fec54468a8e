// select.cuh -- warp-per-token top-8 selection (A2).
//
// Method (ninfer-windows PR #8, the commit that swaps eight dependent
// selection rounds for a warp merge network):
// each lane holds 8 candidates sorted under the selector's total order; five
// xor exchanges merge runs pairwise, each exchange being 8 independent
// shuffles followed by three compare-exchange stages over static indices.
// The tail is a softmax over the 8 selected logits and a sigmoid of the
// shared-expert gate logit.
//
// GB300 form: the (value, id) pair is one 64-bit key whose unsigned order is
// the selector's total order (value first, then lower id), so each
// compare-exchange is a 64-bit max/min.  -0.0 is mapped to +0.0 before the
// key is built, so the two zeros tie and the lower id wins, as IEEE ==
// prescribes.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint64_t rank_key(float v, int id) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0u) u = 0u;                          // -0 -> +0
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);      // order-preserving
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(0xFFFF - id);
}

__device__ __forceinline__ int key_id(uint64_t k) {
  return 0xFFFF - static_cast<int>(k & 0xFFFFu);
}

__device__ __forceinline__ float key_value(uint64_t k) {
  uint32_t u = static_cast<uint32_t>(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

// compare-exchange so that a keeps the better (larger) key
__device__ __forceinline__ void cx(uint64_t &a, uint64_t &b) {
  const uint64_t hi = a > b ? a : b;
  const uint64_t lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// 19-comparator sorting network, descending.
__device__ __forceinline__ void sort8(uint64_t (&k)[8]) {
  cx(k[0], k[2]); cx(k[1], k[3]); cx(k[4], k[6]); cx(k[5], k[7]);
  cx(k[0], k[4]); cx(k[1], k[5]); cx(k[2], k[6]); cx(k[3], k[7]);
  cx(k[0], k[1]); cx(k[2], k[3]); cx(k[4], k[5]); cx(k[6], k[7]);
  cx(k[2], k[4]); cx(k[3], k[5]);
  cx(k[1], k[4]); cx(k[3], k[6]);
  cx(k[1], k[2]); cx(k[3], k[4]); cx(k[5], k[6]);
}

// Keep the best 8 of the union of this lane's sorted run and its partner's
// (lane ^ mask): elementwise best of A[i] and B[7-i] is bitonic and holds
// the 8 best; three half-cleaner stages sort it.
__device__ __forceinline__ void merge_level(uint64_t (&k)[8], int mask) {
  uint64_t p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = __shfl_xor_sync(0xFFFFFFFFu, k[i], mask);
#pragma unroll
  for (int i = 0; i < 8; ++i) k[i] = k[i] > p[7 - i] ? k[i] : p[7 - i];
  cx(k[0], k[4]); cx(k[1], k[5]); cx(k[2], k[6]); cx(k[3], k[7]);
  cx(k[0], k[2]); cx(k[1], k[3]); cx(k[4], k[6]); cx(k[5], k[7]);
  cx(k[0], k[1]); cx(k[2], k[3]); cx(k[4], k[5]); cx(k[6], k[7]);
}

// Select for N tokens with the whole warp, lane l holding the logits of
// experts 8l .. 8l+7 of token n in v[n].  The N merge networks are
// independent, so their shuffles and compare-exchanges interleave.  On
// return every lane holds each token's ids (rank order) and softmax weights;
// ok[n] is false for a non-finite row (ids -1, weights 0).
template <int N>
__device__ __forceinline__ void select_top8_multi(const float (&v)[N][8], int lane,
                                                  int (&ids)[N][8], float (&w)[N][8],
                                                  bool (&ok)[N]) {
  uint64_t k[N][8];
#pragma unroll
  for (int n = 0; n < N; ++n) {
    bool finite = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      finite &= isfinite(v[n][i]);
      k[n][i] = rank_key(v[n][i], 8 * lane + i);
    }
    ok[n] = __all_sync(0xFFFFFFFFu, finite);
  }
#pragma unroll
  for (int n = 0; n < N; ++n) sort8(k[n]);
  // the five levels run as a loop: the selection runs once per token and
  // launch, so a compact body (fetched once) beats straight-line code
#pragma unroll 1
  for (int m = 1; m < 32; m <<= 1)
#pragma unroll
    for (int n = 0; n < N; ++n) merge_level(k[n], m);
#pragma unroll
  for (int n = 0; n < N; ++n) {
    // softmax over the 8 selected logits, max-subtracted (rank 0 is the max)
    const float z0 = key_value(k[n][0]);
    float e[8], s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      e[i] = expf(key_value(k[n][i]) - z0);
      s += e[i];
    }
    const float inv = 1.0f / s;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ids[n][i] = ok[n] ? key_id(k[n][i]) : -1;
      w[n][i] = ok[n] ? e[i] * inv : 0.0f;
    }
    if (MOE_SABOTAGE == 1 && ok[n]) {  // test-only build (see common.cuh)
      int e8 = ids[n][7];
      bool taken = true;
      while (taken) {
        e8 = (e8 + 1) & 255;
        taken = false;
#pragma unroll
        for (int i = 0; i < 7; ++i) taken |= ids[n][i] == e8;
      }
      ids[n][7] = e8;
    }
    if (MOE_SABOTAGE == 2) {  // test-only build (see common.cuh)
      const float t = w[n][6];
      w[n][6] = w[n][7];
      w[n][7] = t;
    }
  }
}

// One token, fewest dependent steps (the fused decode kernel selects each
// token once per launch, on the critical path of the whole block): each
// lane sorts its 8 keys once; then 8 rounds each take the warp's best head.
// A round reduces the heads' value halves with one warp max; among the lanes
// holding that value the lowest holds the lowest expert ids (lane l owns
// experts 8l .. 8l+7), and its head is its own best under the total order,
// so it is the round's winner; it broadcasts its key and drops it.  The
// selected (value, id) pairs and their rank order are those of the merge
// network above (both are the selector's total order), and the softmax below
// is the same arithmetic in the same order, so the results are identical.
// Same contract as select_top8_regs.
__device__ __forceinline__ bool select_top8_rounds(const float (&v)[8], int lane, int (&ids)[8],
                                                   float (&w)[8]) {
  uint64_t k[8];
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    finite &= isfinite(v[i]);
    k[i] = rank_key(v[i], 8 * lane + i);
  }
  const bool ok = __all_sync(0xFFFFFFFFu, finite);
  sort8(k);
  uint64_t best[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    // every finite key's value half is at least 0x00800000, so a drained
    // lane's zero head never ties a real one
    const uint32_t hi = static_cast<uint32_t>(k[0] >> 32);
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, hi);
    const int win = __ffs(__ballot_sync(0xFFFFFFFFu, hi == m)) - 1;
    best[r] = __shfl_sync(0xFFFFFFFFu, k[0], win);
    if (lane == win) {
#pragma unroll
      for (int i = 0; i < 7; ++i) k[i] = k[i + 1];
      k[7] = 0;
    }
  }
  const float z0 = key_value(best[0]);
  float e[8], s = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    e[i] = expf(key_value(best[i]) - z0);
    s += e[i];
  }
  const float inv = 1.0f / s;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    ids[i] = ok ? key_id(best[i]) : -1;
    w[i] = ok ? e[i] * inv : 0.0f;
  }
  if (MOE_SABOTAGE == 1 && ok) {  // test-only build (see common.cuh)
    int e8 = ids[7];
    bool taken = true;
    while (taken) {
      e8 = (e8 + 1) & 255;
      taken = false;
#pragma unroll
      for (int i = 0; i < 7; ++i) taken |= ids[i] == e8;
    }
    ids[7] = e8;
  }
  if (MOE_SABOTAGE == 2) {  // test-only build (see common.cuh)
    const float t = w[6];
    w[6] = w[7];
    w[7] = t;
  }
  return ok;
}

// One token (see select_top8_multi); returns false for a non-finite row.
__device__ __forceinline__ bool select_top8_regs(const float (&v)[8], int lane, int (&ids)[8],
                                                 float (&w)[8]) {
  const float(&vv)[1][8] = reinterpret_cast<const float(&)[1][8]>(v);
  int(&ii)[1][8] = reinterpret_cast<int(&)[1][8]>(ids);
  float(&ww)[1][8] = reinterpret_cast<float(&)[1][8]>(w);
  bool ok[1];
  select_top8_multi<1>(vv, lane, ii, ww, ok);
  return ok[0];
}

// As select_top8_regs, reading the 256 fp32 logits of `row` (16-byte aligned).
__device__ __forceinline__ bool select_top8_warp(const float *row, int lane, int (&ids)[8],
                                                 float (&w)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(row)[2 * lane];
  const float4 b = reinterpret_cast<const float4 *>(row)[2 * lane + 1];
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  return select_top8_regs(v, lane, ids, w);
}

__device__ __forceinline__ float sigmoidf_(float g) {
  if (MOE_SABOTAGE == 3) return 0.0f;  // test-only build (see common.cuh)
  return 1.0f / (1.0f + expf(-g));
}

}  // namespace moe
