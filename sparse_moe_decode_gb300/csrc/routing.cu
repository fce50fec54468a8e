// routing.cu -- A1 router GEMV, A2 top-8 selection, A3 token -> expert lists.
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace moe {

// ----------------------------------------------------------- A1 router
//
// One warp per router row (256 expert rows + the shared-gate row), eight
// tokens per CTA row.  A lane owns 8 consecutive bf16 of each 256-wide slice
// of the row; bf16 x bf16 products are exact in fp32, partial sums are fp32.
constexpr int kRouterWarps = 8;
constexpr int kRouterTok = 8;

__global__ void __launch_bounds__(kRouterWarps * 32)
router_gemv_kernel(const moe_bf16 *__restrict__ x, int T, int H,
                   const moe_bf16 *__restrict__ w_router, const moe_bf16 *__restrict__ w_gate,
                   float *__restrict__ logits, float *__restrict__ gate_logit, int row_begin) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = row_begin + blockIdx.x * kRouterWarps + warp;
  const int rows = kE + (w_gate != nullptr ? 1 : 0);
  if (r >= rows) return;
  const moe_bf16 *wrow = r < kE ? w_router + static_cast<size_t>(r) * H : w_gate;
  const int t0 = blockIdx.y * kRouterTok;
  const int nt = min(kRouterTok, T - t0);
  float acc[kRouterTok];
#pragma unroll
  for (int i = 0; i < kRouterTok; ++i) acc[i] = 0.0f;
  for (int k = lane * 8; k < H; k += 256) {
    const uint4 wv = ld_nc(wrow + k);
    const float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                         bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
    for (int i = 0; i < kRouterTok; ++i) {
      if (i < nt) {
        const uint4 xv = ld_nc(x + static_cast<size_t>(t0 + i) * H + k);
        float a = acc[i];
        a = fmaf(wf[0], bf16_lo(xv.x), a); a = fmaf(wf[1], bf16_hi(xv.x), a);
        a = fmaf(wf[2], bf16_lo(xv.y), a); a = fmaf(wf[3], bf16_hi(xv.y), a);
        a = fmaf(wf[4], bf16_lo(xv.z), a); a = fmaf(wf[5], bf16_hi(xv.z), a);
        a = fmaf(wf[6], bf16_lo(xv.w), a); a = fmaf(wf[7], bf16_hi(xv.w), a);
        acc[i] = a;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kRouterTok; ++i) {
    const float v = warp_sum(acc[i]);
    if (lane == 0 && i < nt) {
      if (r < kE) logits[static_cast<size_t>(t0 + i) * kE + r] = v;
      else if (gate_logit) gate_logit[t0 + i] = v;
    }
  }
}

// The shared-expert gate row alone: one warp per token, the same lane
// order and fp32 summation as the router kernel above.
__global__ void __launch_bounds__(kRouterWarps * 32)
gate_gemv_kernel(const moe_bf16 *__restrict__ x, int T, int H,
                 const moe_bf16 *__restrict__ w_gate, float *__restrict__ gate_logit) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const moe_bf16 *xr = x + static_cast<size_t>(t) * H;
  float a = 0.0f;
  for (int k = lane * 8; k < H; k += 256) {
    const uint4 wv = ld_nc(w_gate + k), xv = ld_nc(xr + k);
    a = fmaf(bf16_lo(wv.x), bf16_lo(xv.x), a); a = fmaf(bf16_hi(wv.x), bf16_hi(xv.x), a);
    a = fmaf(bf16_lo(wv.y), bf16_lo(xv.y), a); a = fmaf(bf16_hi(wv.y), bf16_hi(xv.y), a);
    a = fmaf(bf16_lo(wv.z), bf16_lo(xv.z), a); a = fmaf(bf16_hi(wv.z), bf16_hi(xv.z), a);
    a = fmaf(bf16_lo(wv.w), bf16_lo(xv.w), a); a = fmaf(bf16_hi(wv.w), bf16_hi(xv.w), a);
  }
  a = warp_sum(a);
  if (lane == 0) gate_logit[t] = a;
}

cudaError_t launch_router_gemv(const moe_bf16 *x, int T, int H, const moe_bf16 *w_router,
                               const moe_bf16 *w_gate, float *logits, float *gate_logit,
                               cudaStream_t s, bool gate_only) {
  if (gate_only) {
    if (!w_gate || !gate_logit) return cudaSuccess;
    gate_gemv_kernel<<<(T + kRouterWarps - 1) / kRouterWarps, kRouterWarps * 32, 0, s>>>(
        x, T, H, w_gate, gate_logit);
    return cudaGetLastError();
  }
  const int row_begin = 0;
  const int rows = kE + (w_gate && gate_logit ? 1 : 0) - row_begin;
  if (rows <= 0) return cudaSuccess;
  dim3 grid((rows + kRouterWarps - 1) / kRouterWarps, (T + kRouterTok - 1) / kRouterTok);
  router_gemv_kernel<<<grid, kRouterWarps * 32, 0, s>>>(
      x, T, H, w_router, (w_gate && gate_logit) ? w_gate : nullptr, logits, gate_logit,
      row_begin);
  return cudaGetLastError();
}

// ---------------------------------------------------------- A2 selection

constexpr int kSelWarps = 4;

// One warp per token.  The shared gate's logit comes from gate_logit, or,
// when x and w_gate are given, from the token's own dot product with the gate
// row (the same lane order and fp32 summation as the router kernels; written
// to gate_out if that is given).  counts (optional, zeroed before the launch)
// receives the number of tokens that select each expert.
__global__ void __launch_bounds__(kSelWarps * 32)
select_kernel(const float *__restrict__ logits, int T, int ld,
              const float *__restrict__ gate_logit, const moe_bf16 *__restrict__ x,
              const moe_bf16 *__restrict__ w_gate, int H, float *__restrict__ gate_out,
              int32_t *__restrict__ ids, float *__restrict__ weights, float *__restrict__ sgate,
              int32_t *__restrict__ counts, uint32_t *status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  // the token's logits first, so that their load overlaps the gate's
  const float4 *lrow = reinterpret_cast<const float4 *>(logits + static_cast<size_t>(t) * ld);
  const float4 la = lrow[2 * lane], lb = lrow[2 * lane + 1];
  float g = 0.0f;
  if (w_gate) {
    // batches of 8 chunks (2048 elements), every load of a batch in flight
    // at once; the same lane order and fp32 summation as the router kernels
    const moe_bf16 *xr = x + static_cast<size_t>(t) * H;
    for (int k0 = 0; k0 < H; k0 += 2048) {
      uint4 wv[8], xv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int k = k0 + c * 256 + lane * 8;
        if (k < H) {
          wv[c] = ld_nc(w_gate + k);
          xv[c] = ld_nc(xr + k);
        }
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        if (k0 + c * 256 + lane * 8 >= H) break;
        g = fmaf(bf16_lo(wv[c].x), bf16_lo(xv[c].x), g); g = fmaf(bf16_hi(wv[c].x), bf16_hi(xv[c].x), g);
        g = fmaf(bf16_lo(wv[c].y), bf16_lo(xv[c].y), g); g = fmaf(bf16_hi(wv[c].y), bf16_hi(xv[c].y), g);
        g = fmaf(bf16_lo(wv[c].z), bf16_lo(xv[c].z), g); g = fmaf(bf16_hi(wv[c].z), bf16_hi(xv[c].z), g);
        g = fmaf(bf16_lo(wv[c].w), bf16_lo(xv[c].w), g); g = fmaf(bf16_hi(wv[c].w), bf16_hi(xv[c].w), g);
      }
    }
    g = warp_sum(g);
  } else if (gate_logit) {
    g = gate_logit[t];
  }
  int id[8];
  float w[8];
  const float lv[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
  const bool ok = select_top8_regs(lv, lane, id, w);
  if (!ok && lane == 0) set_status(status, MOE_DEV_NONFINITE);
  if (lane < 8) {
    int myid = id[0];
    float myw = w[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
      if (lane == i) { myid = id[i]; myw = w[i]; }
    ids[static_cast<size_t>(t) * kK + lane] = myid;
    weights[static_cast<size_t>(t) * kK + lane] = myw;
    if (counts && myid >= 0) atomicAdd(counts + myid, 1);
  }
  if (lane == 0) {
    if (sgate && (gate_logit || w_gate)) sgate[t] = sigmoidf_(g);
    if (gate_out && w_gate) gate_out[t] = g;
  }
}

cudaError_t launch_select(const float *logits, int T, int ld, const float *gate_logit,
                          int32_t *ids, float *weights, float *sgate, uint32_t *status,
                          cudaStream_t s, const moe_bf16 *x, const moe_bf16 *w_gate, int H,
                          float *gate_out, int32_t *counts) {
  select_kernel<<<(T + kSelWarps - 1) / kSelWarps, kSelWarps * 32, 0, s>>>(
      logits, T, ld, gate_logit, x, w_gate, H, gate_out, ids, weights, sgate, counts, status);
  return cudaGetLastError();
}

// -------------------------------------------------------------- A3 lists
//
// Deterministic counting sort of the T*K entries by (expert, t, j) in one
// CTA.  Pass 1 counts per expert; an exclusive scan gives offsets.  Pass 2
// walks tokens in chunks of 256: a per-expert bitmap over the chunk's
// entries (bit t * K + j) gives each entry its rank among earlier entries of
// the same expert, so that a token naming one expert in two slots still
// gets two distinct places, and a running per-expert base carries the count
// across chunks.
constexpr int kListThreads = 1024;
constexpr int kListChunk = 256;                     // tokens per chunk
constexpr int kListWords = kListChunk * kK / 32;    // bitmap words per expert
constexpr size_t kListSmem = sizeof(uint32_t) * kE * kListWords +   // bitmap
                             sizeof(uint16_t) * kE * kListWords +   // word prefixes
                             sizeof(int16_t) * kListChunk * kK;     // the chunk's ids
constexpr int kListBatch = 8;  // independent loads in flight per thread

__global__ void __launch_bounds__(kListThreads)
lists_kernel(const int32_t *__restrict__ ids, int T, Lists L, uint32_t *status) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem);
  uint16_t *wpre = reinterpret_cast<uint16_t *>(smem + sizeof(uint32_t) * kE * kListWords);
  __shared__ int cnt[kE], base[kE], run[kE], scan_tmp[8];
  int16_t *cids = reinterpret_cast<int16_t *>(smem + (sizeof(uint32_t) + sizeof(uint16_t)) *
                                                          kE * kListWords);
  const int tid = threadIdx.x;
  const int n = T * kK;
  if (tid < kE) { cnt[tid] = 0; run[tid] = 0; }
  __syncthreads();
  // Loads are batched (kListBatch per thread in flight) so that one CTA
  // streams the ids at bandwidth rather than at one latency per entry.
  bool bad = false;
  for (int i0 = 0; i0 < n; i0 += kListThreads * kListBatch) {
    int e[kListBatch];
#pragma unroll
    for (int u = 0; u < kListBatch; ++u) {
      const int i = i0 + u * kListThreads + tid;
      e[u] = i < n ? ids[i] : -1;
    }
#pragma unroll
    for (int u = 0; u < kListBatch; ++u) {
      if (e[u] >= kE) bad = true;
      else if (e[u] >= 0) atomicAdd(&cnt[e[u]], 1);
    }
  }
  if (bad) set_status(status, MOE_DEV_BAD_EXPERT);
  __syncthreads();
  const int c = tid < kE ? cnt[tid] : 0;
  const int off = block_exclusive_scan_256(c, scan_tmp);
  const int act = block_exclusive_scan_256(c > 0 ? 1 : 0, scan_tmp);
  if (tid < kE) {
    base[tid] = off;
    L.counts[tid] = c;
    L.offsets[tid] = off;
    if (tid == kE - 1) L.offsets[kE] = off + c;
    if (c > 0) L.active[1 + act] = tid;
    if (tid == kE - 1) L.active[0] = act + (c > 0 ? 1 : 0);
  }
  __syncthreads();
  for (int t0 = 0; t0 < T; t0 += kListChunk) {
    const int tn = min(kListChunk, T - t0);
    const int words = (tn * kK + 31) / 32;
    for (int i = tid; i < kE * kListWords; i += kListThreads) bitmap[i] = 0u;
    __syncthreads();
    for (int i0 = 0; i0 < tn * kK; i0 += kListThreads * kListBatch) {
      int e[kListBatch];
#pragma unroll
      for (int u = 0; u < kListBatch; ++u) {
        const int i = i0 + u * kListThreads + tid;
        e[u] = i < tn * kK ? ids[static_cast<size_t>(t0) * kK + i] : -1;
      }
#pragma unroll
      for (int u = 0; u < kListBatch; ++u) {
        const int i = i0 + u * kListThreads + tid;
        if (i < tn * kK) {
          const int ev = (e[u] >= 0 && e[u] < kE) ? e[u] : -1;  // out of range -> no slot
          cids[i] = static_cast<int16_t>(ev);
          if (ev >= 0) atomicOr(&bitmap[ev * kListWords + i / 32], 1u << (i & 31));
        }
      }
    }
    __syncthreads();
    // per-expert exclusive prefix of popcounts over the chunk's words
    const int lane = tid & 31, warp = tid >> 5;
    for (int e = warp; e < kE; e += kListThreads / 32) {
      const int w0 = 2 * lane, w1 = 2 * lane + 1;
      const int p0 = w0 < words ? __popc(bitmap[e * kListWords + w0]) : 0;
      const int p1 = w1 < words ? __popc(bitmap[e * kListWords + w1]) : 0;
      int incl = p0 + p1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = incl - p0 - p1;
      wpre[e * kListWords + w0] = static_cast<uint16_t>(excl);
      wpre[e * kListWords + w1] = static_cast<uint16_t>(excl + p0);
    }
    __syncthreads();
    for (int i = tid; i < tn * kK; i += kListThreads) {
      const size_t gi = static_cast<size_t>(t0) * kK + i;
      const int e = cids[i];
      if (e < 0) {
        if (L.slot_of) L.slot_of[gi] = -1;
        continue;
      }
      const int wd = i / 32;
      const uint32_t below = bitmap[e * kListWords + wd] & ((1u << (i & 31)) - 1u);
      const int pos = base[e] + run[e] + wpre[e * kListWords + wd] + __popc(below);
      L.perm[pos] = static_cast<int32_t>(gi);
      if (L.slot_of) L.slot_of[gi] = pos;
    }
    __syncthreads();
    if (tid < kE) {
      int tot = 0;
      for (int w = 0; w < words; ++w) tot += __popc(bitmap[tid * kListWords + w]);
      run[tid] += tot;
    }
    __syncthreads();
  }
}

cudaError_t launch_lists(const int32_t *ids, int T, Lists L, uint32_t *status, cudaStream_t s) {
  static bool attr_set = false;  // the attribute is per-function, set once per process
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(lists_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kListSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  lists_kernel<<<1, kListThreads, kListSmem, s>>>(ids, T, L, status);
  return cudaGetLastError();
}

}  // namespace moe
