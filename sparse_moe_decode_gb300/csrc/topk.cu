// topk.cu -- exact top-k candidates over wide rows, and the exact merge of
// candidate lists (k <= 16).
//
// What it computes: the candidate selector of the DFlash2 drafter takes the
// top-k lm_head entries of each block position on the GPU, with k raised
// from 8 to 16 (lucebox commit list, "candidate selector head"); the
// two-GPU drafter splits the vocabulary and joins the halves with an exact
// top-16 merge (ninfer-tp2 v0.4.0 notes).  The order is the MoE selector's:
// greater value wins, the lower index breaks a tie, -0 ties +0
// (sparse_moe_ranked_better in ninfer-windows PR #8; the split proposal head
// of ninfer-tp2 v0.4.x sends ties to the lower row the same way).  Every k
// from 1 to 16 is served by the same code; there are no per-k instances to
// leave holes (the lucebox fix for K = 9..11 and 13..15 returning scratch).
//
// GB300 form.  A (value, index) pair is one 64-bit key whose unsigned order
// is the selector's order: the high word is the value's bits made
// order-preserving (-0 first mapped to +0), the low word the complement of
// the index, so a lower index gives a larger key.  Key 0 is below every real
// key and pads short runs.
//   phase 1 (topk_chunk_kernel): one warp per 1024 columns of a row; each
//     lane streams 32 values (eight coalesced 16-byte loads, all in flight at
//     once) and keeps their order-preserving 32-bit images.  The lane maxima
//     give a floor (the 16th best of them), the keys at or above it are
//     appended to the warp's candidate list in shared memory, and each
//     candidate's rank is the number of larger candidates; ranks 0..15 are
//     the chunk's best 16, written as one sorted run.  No barrier spans
//     warps; each logit is read once (HBM-bound).
//   phase 2 (topk_merge_kernel): one CTA per row; the best k-th key of any
//     run is a floor for the row, warps append the keys at or above it (32
//     runs per pass) and rank them, and the CTA ranks the warps' best 16 to
//     give the first k.  The same kernel merges caller lists of (id, value)
//     pairs.
// A row holding NaN or +-inf is a precondition violation, as for the MoE
// selector: its ids are -1, its values 0, and MOE_DEV_NONFINITE is set.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRun = 16;                              // run length: the largest k served
constexpr int kTkThreads = 256;                       // 8 warps
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkVec = 8;                             // 16-byte loads per lane
constexpr int kTkWarpCols = 32 * 4 * kTkVec;          // 1024 columns per warp
// The run written for a chunk that held a non-finite value (or folded in for
// a caller list with a negative id): every real key has a low word >= 2^31
// (indices < 2^31), so key 1 is never a real entry.
constexpr uint64_t kInvalidKey = 1ull;

__device__ __forceinline__ uint64_t cand_key(float v, uint32_t id) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0u) u = 0u;                          // -0 ties +0
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);      // order-preserving
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(~id);
}

__device__ __forceinline__ int32_t cand_id(uint64_t k) {
  return static_cast<int32_t>(~static_cast<uint32_t>(k));
}

__device__ __forceinline__ uint64_t kmax(uint64_t a, uint64_t b) { return a > b ? a : b; }

// Candidate space of one warp: 512 keys (in phase 1 at most 16 lanes reach
// the floor, with 32 keys each; in phase 2 a pass takes 32 lists of at most
// 16 keys), after the warp's running best 16.
constexpr int kTkCand = kRun + 16 * 32;

struct TopkSmem {
  uint64_t cand[kTkWarps][kTkCand];
  uint64_t top[kTkWarps][kRun];       // each warp's best 16 by rank (0 = none)
  uint64_t lane_max[kTkWarps][32];
  uint64_t out[kRun];                 // the CTA's best 16 by rank
  uint64_t floor_key[kTkWarps];
};

// rank of x among the n keys at c (keys distinct except 0): the number of
// larger keys.  Broadcast reads of shared memory, four compares in flight.
__device__ __forceinline__ int rank_in(const uint64_t *c, int n, uint64_t x) {
  int r = 0, f = 0;
  for (; f + 4 <= n; f += 4)
    r += (c[f] > x) + (c[f + 1] > x) + (c[f + 2] > x) + (c[f + 3] > x);
  for (; f < n; ++f) r += c[f] > x;
  return r;
}

// The warp's best 16 of its n candidates in S.cand[warp] into S.top[warp]
// (slot = rank; a slot no key reaches keeps 0).  Keys are distinct, so the
// ranks are.  Ends with the warp synchronised.
__device__ __forceinline__ void warp_rank_top(TopkSmem &S, int warp, int lane, int n) {
  __syncwarp();
  if (lane < kRun) S.top[warp][lane] = 0ull;
  __syncwarp();
  for (int e = lane; e < n; e += 32) {
    const uint64_t x = S.cand[warp][e];
    const int r = rank_in(S.cand[warp], n, x);
    if (r < kRun) S.top[warp][r] = x;
  }
  __syncwarp();
}

// Appends the keys of this lane selected by mask (bit i: keys[i]) to
// S.cand[warp] after `start` entries; returns the new total.
template <int M>
__device__ __forceinline__ int warp_append(TopkSmem &S, int warp, int lane, int start,
                                           const uint64_t (&keys)[M], uint32_t mask) {
  const int c = __popc(mask);
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += y;
  }
  const int total = start + __shfl_sync(0xFFFFFFFFu, incl, 31);
  int off = start + incl - c;
#pragma unroll
  for (int i = 0; i < M; ++i)
    if ((mask >> i) & 1u) S.cand[warp][off++] = keys[i];
  return total;
}

// The CTA's best 16 of the warps' S.top entries into S.out, by all threads
// (entry tid < 128 ranks itself against the 128).  Ends synchronised.
__device__ __forceinline__ void cta_rank_top(TopkSmem &S) {
  if (threadIdx.x < kRun) S.out[threadIdx.x] = 0ull;
  __syncthreads();
  const uint64_t *all = &S.top[0][0];
  if (threadIdx.x < kTkWarps * kRun) {
    const uint64_t x = all[threadIdx.x];
    if (x != 0ull) {
      const int r = rank_in(all, kTkWarps * kRun, x);
      if (r < kRun) S.out[r] = x;
    }
  }
  __syncthreads();
}

// Phase 1: the sorted best 16 keys of each 1024-column chunk of each row,
// one warp per chunk and no barrier across warps.  Warp g of the grid takes
// row g / n_wc, columns (g % n_wc) * 1024 ...; lane l the float4 at l + 32 i
// of them.  The 16th best of the warp's 32 lane maxima bounds the chunk's
// 16th best from below (16 lanes each hold a key at least that large), so
// only keys at or above it are candidates, and only the 16 lanes whose
// maxima reach it hold any (at most 512 candidates).
__global__ void __launch_bounds__(kTkThreads, 4) topk_chunk_kernel(
    const float *__restrict__ logits, int ld, int N, int n_wc, int n_warps,
    uint64_t *__restrict__ runs) {
  __shared__ TopkSmem S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * kTkWarps + warp;
  if (g >= n_warps) return;  // whole warps only: nothing below syncs the CTA
  const int t = g / n_wc, c = g - t * n_wc;
  const float *row = logits + static_cast<size_t>(t) * ld;
  const int base = c * kTkWarpCols + 4 * lane;
  float4 q[kTkVec];
  if ((c + 1) * kTkWarpCols <= N) {
#pragma unroll
    for (int i = 0; i < kTkVec; ++i)  // all loads in flight at once
      q[i] = __ldcs(reinterpret_cast<const float4 *>(row + base + 128 * i));
  } else {
#pragma unroll
    for (int i = 0; i < kTkVec; ++i) {
      const int col = base + 128 * i;
      q[i].x = col < N ? __ldcs(row + col) : 0.0f;
      q[i].y = col + 1 < N ? __ldcs(row + col + 1) : 0.0f;
      q[i].z = col + 2 < N ? __ldcs(row + col + 2) : 0.0f;
      q[i].w = col + 3 < N ? __ldcs(row + col + 3) : 0.0f;
    }
  }
  // order-preserving 32-bit images of the values; adding +0 first turns -0
  // into +0 (the two tie), and leaves every other value as it is
  uint32_t o[4 * kTkVec];
  uint32_t mo = 0u, mn = ~0u;
  int first = -1;
#pragma unroll
  for (int i = 0; i < kTkVec; ++i) {
    const float v[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t u = __float_as_uint(v[e] + 0.0f);
      const uint32_t w = u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
      o[4 * i + e] = w;
      mn = min(mn, w);  // columns past N were loaded as +0: finite
    }
  }
  if ((c + 1) * kTkWarpCols > N) {
#pragma unroll
    for (int i = 0; i < 4 * kTkVec; ++i)  // 0: below the image of any value (-inf's is 0x007FFFFF)
      if (base + 128 * (i / 4) + (i % 4) >= N) o[i] = 0u;
  }
#pragma unroll
  for (int i = 0; i < 4 * kTkVec; ++i) mo = max(mo, o[i]);
  // NaN and +-inf are the images at or above +inf's and at or below -inf's
  bool bad = mo >= 0xFF800000u || mn <= 0x007FFFFFu;
  // the lane's best key: its largest image at its lowest column holding it
#pragma unroll
  for (int i = 4 * kTkVec - 1; i >= 0; --i)
    if (o[i] == mo) first = i;
  const uint64_t mk = mo == 0u ? 0ull
      : (static_cast<uint64_t>(mo) << 32) |
            static_cast<uint32_t>(~static_cast<uint32_t>(base + 128 * (first / 4) + (first % 4)));
  // the floor: the lane maximum ranked 15th (0 when fewer than 16 lanes
  // hold columns; zero maxima all rank after the real ones)
  S.lane_max[warp][lane] = mk;
  if (lane == 0) S.floor_key[warp] = 0ull;
  __syncwarp();
  if (mk != 0ull && rank_in(S.lane_max[warp], 32, mk) == kRun - 1) S.floor_key[warp] = mk;
  __syncwarp();
  const uint64_t fl = S.floor_key[warp];
  const uint32_t fo = static_cast<uint32_t>(fl >> 32);
  const int fcol = static_cast<int>(~static_cast<uint32_t>(fl));  // -1 when fl == 0
  // candidates: key >= floor, i.e. a larger image, or the same image at a
  // column no higher than the floor's
  // (with no floor, fo = 0 and fcol = -1: every image above 0, i.e. every
  // column below N, passes)
  const int dcol = fcol - base;
  uint32_t mask = 0u;
#pragma unroll
  for (int i = 0; i < 4 * kTkVec; ++i)
    if (o[i] > fo || (o[i] == fo && 128 * (i / 4) + (i % 4) <= dcol)) mask |= 1u << i;
  // append the candidates' keys to the warp's list
  const int cnt = __popc(mask);
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += y;
  }
  const int n = __shfl_sync(0xFFFFFFFFu, incl, 31);
  int off = incl - cnt;
#pragma unroll
  for (int i = 0; i < 4 * kTkVec; ++i)
    if ((mask >> i) & 1u)
      S.cand[warp][off++] = (static_cast<uint64_t>(o[i]) << 32) |
                            static_cast<uint32_t>(~static_cast<uint32_t>(base + 128 * (i / 4) + (i % 4)));
  warp_rank_top(S, warp, lane, n);
  bad = __any_sync(0xFFFFFFFFu, bad);
  if (lane < kRun)
    runs[(static_cast<size_t>(t) * n_wc + c) * kRun + lane] = bad ? kInvalidKey : S.top[warp][lane];
}

// Phase 2: one CTA per row folds the row's n_lists lists into the best k.
// PAIRS = false: runs of 16 sorted keys from phase 1; the values are read
// back from the row (so a selected -0.0 comes back as -0.0).  PAIRS = true:
// caller lists of k (id, value) pairs in any order; the values are copied
// from the entry whose id was selected.  The best k-th key of any list
// bounds the row's k-th best from below, and so do the k-th best head of
// any 32 lists and any k-th best found so far; only keys at or above the
// largest are candidates.  Each warp takes 32 lists per pass and keeps its
// best 16; one pass over the lists.
template <bool PAIRS>
__global__ void __launch_bounds__(kTkThreads) topk_merge_kernel(
    const uint64_t *__restrict__ runs, const int32_t *__restrict__ in_ids,
    const float *__restrict__ in_vals, int n_lists, int k, const float *__restrict__ logits,
    int ld, int N, int32_t *__restrict__ ids_out, float *__restrict__ vals_out,
    uint32_t *status) {
  __shared__ TopkSmem S;
  __shared__ int32_t s_ids[kRun];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x;
  const size_t row0 = static_cast<size_t>(t) * n_lists;
  // a list's keys (0 past its end), its k-th best, and whether it is valid
  auto load_list = [&](int j, uint64_t (&b)[kRun], bool &bad_list) -> uint64_t {
#pragma unroll
    for (int i = 0; i < kRun; ++i) b[i] = 0ull;
    bad_list = false;
    if (j >= n_lists) return 0ull;
    if (!PAIRS) {
      const ulonglong2 *src = reinterpret_cast<const ulonglong2 *>(runs + (row0 + j) * kRun);
#pragma unroll
      for (int i = 0; i < kRun; i += 2) {
        const ulonglong2 u = __ldcg(src + i / 2);
        b[i] = u.x;
        b[i + 1] = u.y;
      }
      bad_list = b[0] == kInvalidKey;
      uint64_t kth = 0ull;
#pragma unroll
      for (int i = 0; i < kRun; ++i)
        if (i == k - 1) kth = b[i];
      return kth;
    }
    const size_t o = (row0 + j) * k;
    uint64_t lo = ~0ull;
#pragma unroll
    for (int i = 0; i < kRun; ++i)
      if (i < k) {
        const int32_t id = in_ids[o + i];
        bad_list |= id < 0;
        b[i] = cand_key(in_vals[o + i], static_cast<uint32_t>(id));
        lo = b[i] < lo ? b[i] : lo;
      }
    return lo;  // k entries: the smallest is the list's k-th best
  };
  // One pass: each warp takes 32 lists at a time.  Three floors, each at
  // most the row's k-th best: a list's k-th best key, the k-th best of the
  // 32 lists' heads (k lists each hold a key at least that large), and the
  // warp's running k-th best.  Keys at or above the largest are candidates.
  bool bad = false;
  if (lane < kRun) S.top[warp][lane] = 0ull;
  for (int j0 = warp * 32; j0 < n_lists; j0 += kTkThreads) {
    uint64_t b[kRun];
    bool bl;
    uint64_t fl = load_list(j0 + lane, b, bl);
    bad |= bl;
    uint64_t head = 0ull;
#pragma unroll
    for (int i = 0; i < kRun; ++i) head = kmax(head, b[i]);
    __syncwarp();
    S.lane_max[warp][lane] = head;
    __syncwarp();
    if (head != 0ull && rank_in(S.lane_max[warp], 32, head) == k - 1) fl = kmax(fl, head);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) fl = kmax(fl, __shfl_xor_sync(0xFFFFFFFFu, fl, m));
    fl = kmax(fl, S.top[warp][k - 1]);
    uint32_t mask = 0u;
#pragma unroll
    for (int i = 0; i < kRun; ++i)
      if (b[i] != 0ull && b[i] >= fl) mask |= 1u << i;
    // the running best 16 first, then this pass's candidates
    __syncwarp();
    if (lane < kRun) S.cand[warp][lane] = S.top[warp][lane];
    const int n = warp_append(S, warp, lane, kRun, b, mask);
    warp_rank_top(S, warp, lane, n);
  }
  bad = __syncthreads_or(bad);
  cta_rank_top(S);
  if (warp == 0) {
    const uint64_t r = lane < kRun ? S.out[lane] : 0ull;
    if (lane < k) {
      const int32_t id = bad ? -1 : cand_id(r);
      ids_out[static_cast<size_t>(t) * k + lane] = id;
      // The value is the key's image inverted; the image is one-to-one but
      // for -0, which shares +0's, so a selected zero is read back from the
      // row for its sign.  (N >= k real keys reach every row's best k, so
      // the id is a column of the row; the bound is checked all the same.)
      if (!PAIRS) {
        const uint32_t img = static_cast<uint32_t>(r >> 32);
        float v = __uint_as_float((img & 0x80000000u) ? (img & 0x7FFFFFFFu) : ~img);
        if (img == 0x80000000u)
          v = (id >= 0 && id < N) ? __ldcs(logits + static_cast<size_t>(t) * ld + id) : 0.0f;
        vals_out[static_cast<size_t>(t) * k + lane] = bad ? 0.0f : v;
      }
      else if (bad)
        vals_out[static_cast<size_t>(t) * k + lane] = 0.0f;
      s_ids[lane] = id;
    }
    if (bad && lane == 0) set_status(status, MOE_DEV_NONFINITE);
  }
  if (PAIRS && !bad) {
    __syncthreads();
    // ids within a row are distinct, so exactly one entry matches each slot
    const size_t o = row0 * k;
    for (int e = threadIdx.x; e < n_lists * k; e += kTkThreads) {
      const int32_t id = in_ids[o + e];
      for (int j = 0; j < k; ++j)
        if (s_ids[j] == id) vals_out[static_cast<size_t>(t) * k + j] = in_vals[o + e];
    }
  }
}

}  // namespace

int topk_chunks(int N) { return (N + kTkWarpCols - 1) / kTkWarpCols; }

cudaError_t launch_topk(const float *logits, int T, int ld, int N, int k, int32_t *ids,
                        float *values, uint64_t *runs, uint32_t *status, cudaStream_t s) {
  const int n_wc = topk_chunks(N);
  const int n_warps = T * n_wc;
  topk_chunk_kernel<<<(n_warps + kTkWarps - 1) / kTkWarps, kTkThreads, 0, s>>>(
      logits, ld, N, n_wc, n_warps, runs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  topk_merge_kernel<false><<<T, kTkThreads, 0, s>>>(runs, nullptr, nullptr, n_wc, k, logits,
                                                    ld, N, ids, values, status);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const int32_t *ids, const float *values, int T, int n_lists,
                              int k, int32_t *ids_out, float *values_out, uint32_t *status,
                              cudaStream_t s) {
  topk_merge_kernel<true><<<T, kTkThreads, 0, s>>>(nullptr, ids, values, n_lists, k, nullptr, 0,
                                                   0, ids_out, values_out, status);
  return cudaGetLastError();
}

}  // namespace moe
