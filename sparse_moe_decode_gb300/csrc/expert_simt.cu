// expert_simt.cu -- weight-streaming int8 group-128 expert kernels for
// decode-size T (A4 gate|up + SwiGLU, A5 down, A6 shared expert) and the A7
// combine.
//
// Layout of the work: blockIdx.y = 0 is the shared expert (every token),
// blockIdx.y = 1 + a is the a-th active routed expert (its tokens are the
// list entries offsets[e] .. offsets[e+1]).  A CTA streams a slice of that
// expert's rows exactly once and applies them to all of the expert's tokens,
// TT tokens at a time, so weight bytes are read once per distinct expert.
//
// Inner product: a lane owns 16 consecutive int8 weights (one 16-byte load)
// per 512-wide slice of a row; those 16 lie inside one 128-group, so the
// group scale multiplies the 16-term fp32 partial once.  int8 -> fp32 is the
// exact magic-number conversion of common.cuh; products with bf16
// activations are exact in fp32, sums are fp32.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kGUWarps = 8;
constexpr int kGUPairs = 2;              // gate/up row pairs per warp
constexpr int kGUSegChunks = 4;          // 16-byte chunks per lane per segment (2048 K)
constexpr int kTT = 8;                   // tokens per pass

struct ExpertJob {
  const int8_t *q;       // [rows][K] int8 for this expert
  const moe_bf16 *s;     // [rows][K/G]
  int rows_half;         // I (gate rows; up rows follow)
  int count;             // tokens of this expert
  int first;             // list position of the first token (routed) or 0
  bool shared;
};

__device__ __forceinline__ bool expert_job(int item, int I, int Is, int T, const int8_t *q,
                                           const moe_bf16 *s, const int8_t *qs,
                                           const moe_bf16 *ss, size_t q_stride,
                                           size_t s_stride, const Lists &L, ExpertJob &j) {
  if (item == 0) {
    if (Is == 0) return false;
    j.q = qs; j.s = ss; j.rows_half = Is; j.count = T; j.first = 0; j.shared = true;
    return true;
  }
  const int a = item - 1;
  if (a >= L.active[0]) return false;
  const int e = L.active[1 + a];
  j.q = q + static_cast<size_t>(e) * q_stride;
  j.s = s + static_cast<size_t>(e) * s_stride;
  j.rows_half = I;
  j.first = L.offsets[e];
  j.count = L.offsets[e + 1] - j.first;
  j.shared = false;
  return true;
}

// token index of the c-th token of a job
__device__ __forceinline__ int job_token(const ExpertJob &j, const Lists &L, int c) {
  return j.shared ? c : L.perm[j.first + c] / kK;
}

__device__ __forceinline__ float dot16(const uint4 w, const uint4 xa, const uint4 xb) {
  const f4 w0 = i8x4_to_f32(w.x), w1 = i8x4_to_f32(w.y), w2 = i8x4_to_f32(w.z),
           w3 = i8x4_to_f32(w.w);
  float a = w0.x * bf16_lo(xa.x);
  a = fmaf(w0.y, bf16_hi(xa.x), a); a = fmaf(w0.z, bf16_lo(xa.y), a);
  a = fmaf(w0.w, bf16_hi(xa.y), a); a = fmaf(w1.x, bf16_lo(xa.z), a);
  a = fmaf(w1.y, bf16_hi(xa.z), a); a = fmaf(w1.z, bf16_lo(xa.w), a);
  a = fmaf(w1.w, bf16_hi(xa.w), a); a = fmaf(w2.x, bf16_lo(xb.x), a);
  a = fmaf(w2.y, bf16_hi(xb.x), a); a = fmaf(w2.z, bf16_lo(xb.y), a);
  a = fmaf(w2.w, bf16_hi(xb.y), a); a = fmaf(w3.x, bf16_lo(xb.z), a);
  a = fmaf(w3.y, bf16_hi(xb.z), a); a = fmaf(w3.z, bf16_lo(xb.w), a);
  a = fmaf(w3.w, bf16_hi(xb.w), a);
  return a;
}

// ------------------------------------------------------- A4 gate|up + SwiGLU

__global__ void __launch_bounds__(kGUWarps * 32)
gateup_simt_kernel(const moe_bf16 *__restrict__ x, int T, int H, int I, int Is,
                   const int8_t *__restrict__ w13_q, const moe_bf16 *__restrict__ w13_s,
                   const int8_t *__restrict__ ws13_q, const moe_bf16 *__restrict__ ws13_s,
                   Lists L, moe_bf16 *__restrict__ h_routed, moe_bf16 *__restrict__ h_shared) {
  ExpertJob job;
  if (!expert_job(blockIdx.y, I, Is, T, w13_q, w13_s, ws13_q, ws13_s,
                  static_cast<size_t>(2) * I * H, static_cast<size_t>(2) * I * (H / kG), L, job))
    return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = H / kG;
  const int nchunks = H / 16;  // 16-byte chunks per row
  for (int pr = 0; pr < kGUPairs; ++pr) {
    const int i = (blockIdx.x * kGUWarps + warp) * kGUPairs + pr;
    if (i >= job.rows_half) return;
    const int8_t *qg = job.q + static_cast<size_t>(i) * H;
    const int8_t *qu = job.q + static_cast<size_t>(job.rows_half + i) * H;
    const moe_bf16 *sg = job.s + static_cast<size_t>(i) * ng;
    const moe_bf16 *su = job.s + static_cast<size_t>(job.rows_half + i) * ng;
    for (int tb = 0; tb < job.count; tb += kTT) {
      const int nt = min(kTT, job.count - tb);
      int tok[kTT];
#pragma unroll
      for (int u = 0; u < kTT; ++u) tok[u] = u < nt ? job_token(job, L, tb + u) : 0;
      float ag[kTT], au[kTT];
#pragma unroll
      for (int u = 0; u < kTT; ++u) { ag[u] = 0.0f; au[u] = 0.0f; }
      for (int c0 = 0; c0 < nchunks; c0 += 32 * kGUSegChunks) {
        uint4 wg[kGUSegChunks], wu[kGUSegChunks];
        float scg[kGUSegChunks], scu[kGUSegChunks];
#pragma unroll
        for (int c = 0; c < kGUSegChunks; ++c) {
          const int ch = c0 + c * 32 + lane;
          if (ch < nchunks) {
            wg[c] = ld_stream(qg + ch * 16);
            wu[c] = ld_stream(qu + ch * 16);
            scg[c] = bf16_to_f32(sg[ch / 8]);
            scu[c] = bf16_to_f32(su[ch / 8]);
          } else {
            wg[c] = make_uint4(0, 0, 0, 0); wu[c] = wg[c];
            scg[c] = 0.0f; scu[c] = 0.0f;
          }
        }
#pragma unroll
        for (int c = 0; c < kGUSegChunks; ++c) {
          const int ch = c0 + c * 32 + lane;
          if (ch >= nchunks) continue;
#pragma unroll
          for (int u = 0; u < kTT; ++u) {
            if (u < nt) {
              const uint4 *xp = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(tok[u]) * H + ch * 16);
              const uint4 xa = ld_nc(xp), xb = ld_nc(xp + 1);
              ag[u] = fmaf(scg[c], dot16(wg[c], xa, xb), ag[u]);
              au[u] = fmaf(scu[c], dot16(wu[c], xa, xb), au[u]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kTT; ++u) {
        const float g = warp_sum(ag[u]);
        const float up = warp_sum(au[u]);
        if (lane == 0 && u < nt) {
          const uint16_t hv = f32_to_bf16(silu_mul(g, up));
          if (job.shared) h_shared[static_cast<size_t>(tb + u) * job.rows_half + i] = hv;
          else h_routed[static_cast<size_t>(job.first + tb + u) * job.rows_half + i] = hv;
        }
      }
    }
  }
}

cudaError_t launch_gateup_simt(const moe_bf16 *x, int T, int H, int I, int Is,
                               const moe_weights &w, Lists L, moe_bf16 *h_routed,
                               moe_bf16 *h_shared, cudaStream_t s) {
  const int rows = I > Is ? I : Is;
  const int per_cta = kGUWarps * kGUPairs;
  const int items = 1 + (T * kK < kE ? T * kK : kE);
  dim3 grid((rows + per_cta - 1) / per_cta, items);
  gateup_simt_kernel<<<grid, kGUWarps * 32, 0, s>>>(x, T, H, I, Is, w.w13_q, w.w13_s, w.ws13_q,
                                                    w.ws13_s, L, h_routed, h_shared);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- A5 down

constexpr int kDWarps = 8;

template <int CPR>  // 16-byte chunks per lane per row: ceil(I / 512)
__global__ void __launch_bounds__(kDWarps * 32)
down_simt_kernel(int T, int H, int I, int Is, const int8_t *__restrict__ w2_q,
                 const moe_bf16 *__restrict__ w2_s, const int8_t *__restrict__ ws2_q,
                 const moe_bf16 *__restrict__ ws2_s, Lists L,
                 const moe_bf16 *__restrict__ h_routed, const moe_bf16 *__restrict__ h_shared,
                 float *__restrict__ y) {
  constexpr int RPW = CPR == 1 ? 8 : (CPR == 2 ? 4 : 2);  // rows per warp
  ExpertJob job;
  if (!expert_job(blockIdx.y, I, Is, T, w2_q, w2_s, ws2_q, ws2_s, static_cast<size_t>(H) * I,
                  static_cast<size_t>(H) * (I / kG), L, job))
    return;
  const int Ii = job.rows_half;  // reduction length of this expert
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n0 = (blockIdx.x * kDWarps + warp) * RPW;
  if (n0 >= H) return;
  const int nchunks = Ii / 16;
  const int ng = Ii / kG;
  uint4 wr[RPW][CPR];
  float sc[RPW][CPR];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
#pragma unroll
    for (int c = 0; c < CPR; ++c) {
      const int ch = c * 32 + lane;
      const int n = n0 + r;
      if (ch < nchunks && n < H) {
        wr[r][c] = ld_stream(job.q + static_cast<size_t>(n) * Ii + ch * 16);
        sc[r][c] = bf16_to_f32(job.s[static_cast<size_t>(n) * ng + ch / 8]);
      } else {
        wr[r][c] = make_uint4(0, 0, 0, 0);
        sc[r][c] = 0.0f;
      }
    }
  }
  for (int c0 = 0; c0 < job.count; ++c0) {
    const moe_bf16 *hrow = job.shared ? h_shared + static_cast<size_t>(c0) * Ii
                                      : h_routed + static_cast<size_t>(job.first + c0) * Ii;
    float acc[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) acc[r] = 0.0f;
#pragma unroll
    for (int c = 0; c < CPR; ++c) {
      const int ch = c * 32 + lane;
      if (ch < nchunks) {
        const uint4 *hp = reinterpret_cast<const uint4 *>(hrow + ch * 16);
        const uint4 ha = hp[0], hb = hp[1];
#pragma unroll
        for (int r = 0; r < RPW; ++r) acc[r] = fmaf(sc[r][c], dot16(wr[r][c], ha, hb), acc[r]);
      }
    }
    size_t ybase;
    if (job.shared) {
      ybase = (static_cast<size_t>(c0) * (kK + 1) + kK) * H;
    } else {
      const int ent = L.perm[job.first + c0];  // t*K + j
      ybase = (static_cast<size_t>(ent / kK) * (kK + 1) + ent % kK) * H;
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const float v = warp_sum(acc[r]);
      if (lane == 0 && n0 + r < H) y[ybase + n0 + r] = v;
    }
  }
}

cudaError_t launch_down_simt(int T, int H, int I, int Is, const moe_weights &w, Lists L,
                             const moe_bf16 *h_routed, const moe_bf16 *h_shared, float *y,
                             cudaStream_t s) {
  const int Imax = I > Is ? I : Is;
  const int cpr = (Imax + 511) / 512;
  const int items = 1 + (T * kK < kE ? T * kK : kE);
  const int rpw = cpr == 1 ? 8 : (cpr == 2 ? 4 : 2);
  dim3 grid((H + kDWarps * rpw - 1) / (kDWarps * rpw), items);
  switch (cpr) {
    case 1:
      down_simt_kernel<1><<<grid, kDWarps * 32, 0, s>>>(T, H, I, Is, w.w2_q, w.w2_s, w.ws2_q,
                                                        w.ws2_s, L, h_routed, h_shared, y);
      break;
    case 2:
      down_simt_kernel<2><<<grid, kDWarps * 32, 0, s>>>(T, H, I, Is, w.w2_q, w.w2_s, w.ws2_q,
                                                        w.ws2_s, L, h_routed, h_shared, y);
      break;
    case 3:
      down_simt_kernel<3><<<grid, kDWarps * 32, 0, s>>>(T, H, I, Is, w.w2_q, w.w2_s, w.ws2_q,
                                                        w.ws2_s, L, h_routed, h_shared, y);
      break;
    case 4:
      down_simt_kernel<4><<<grid, kDWarps * 32, 0, s>>>(T, H, I, Is, w.w2_q, w.w2_s, w.ws2_q,
                                                        w.ws2_s, L, h_routed, h_shared, y);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// -------------------------------------------------------------- A7 combine

__global__ void combine_kernel(int T, int H, const float *__restrict__ y,
                               const float *__restrict__ weights,
                               const float *__restrict__ sgate, const moe_bf16 *resid,
                               moe_bf16 *out) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int H4 = H / 4;
  if (idx >= static_cast<size_t>(T) * H4) return;
  const int t = static_cast<int>(idx / H4);
  const int n = static_cast<int>(idx % H4) * 4;
  const float *yt = y + static_cast<size_t>(t) * (kK + 1) * H + n;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kK; ++j) {
    const float wj = weights[static_cast<size_t>(t) * kK + j];
    if (wj == 0.0f) continue;
    const float4 v = *reinterpret_cast<const float4 *>(yt + static_cast<size_t>(j) * H);
    acc.x = fmaf(wj, v.x, acc.x); acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z); acc.w = fmaf(wj, v.w, acc.w);
  }
  if (sgate) {
    const float g = sgate[t];
    if (g != 0.0f) {
      const float4 v = *reinterpret_cast<const float4 *>(yt + static_cast<size_t>(kK) * H);
      acc.x = fmaf(g, v.x, acc.x); acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z); acc.w = fmaf(g, v.w, acc.w);
    }
  }
  if (resid) {  // the residual, added before the one rounding (in place allowed)
    const uint2 r = *reinterpret_cast<const uint2 *>(resid + static_cast<size_t>(t) * H + n);
    acc.x += bf16_lo(r.x); acc.y += bf16_hi(r.x);
    acc.z += bf16_lo(r.y); acc.w += bf16_hi(r.y);
  }
  uint2 o;
  o.x = pack_bf16x2(acc.x, acc.y);
  o.y = pack_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2 *>(out + static_cast<size_t>(t) * H + n) = o;
}

cudaError_t launch_combine(int T, int H, const float *y, const float *weights,
                           const float *sgate, moe_bf16 *out, cudaStream_t s,
                           const moe_bf16 *resid) {
  const size_t n = static_cast<size_t>(T) * (H / 4);
  const int threads = 256;
  combine_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, s>>>(
      T, H, y, weights, sgate, resid, out);
  return cudaGetLastError();
}

}  // namespace moe
