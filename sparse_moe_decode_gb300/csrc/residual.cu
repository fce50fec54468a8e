// residual.cu -- the step after the block in a decoder layer: the next
// layer's input, the RMS norm of the residual sum times its weight vector
// (lucebox commit list, the fused residual add + RMS norm + weight multiply
// that keeps the residual sum beside the normalised output).  The residual
// add itself happens in the block's combine epilogue, before its one
// rounding; this kernel reads the rounded residual sum.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kNormWarps = 8;  // tokens per CTA

// One warp per token: lane l takes the 16-byte chunks l, l + 32, ... of the
// row (eight bf16 each; H is a multiple of 128, so the last chunk may cover
// only half the lanes), sums the squares in that order, then a fixed xor
// tree adds the lanes; x = bf16((r * inv) * gamma).
__global__ void __launch_bounds__(32 * kNormWarps)
rmsnorm_kernel(const moe_bf16 *__restrict__ r, int T, int H, const moe_bf16 *__restrict__ gamma,
               float eps, moe_bf16 *__restrict__ x) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kNormWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const moe_bf16 *row = r + static_cast<size_t>(t) * H;
  float ss = 0.0f;
  for (int k = lane * 8; k < H; k += 256) {
    const uint4 v = ld_nc(row + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = bf16_lo(w[i]), b = bf16_hi(w[i]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  for (int k = lane * 8; k < H; k += 256) {
    const uint4 v = ld_nc(row + k), gv = ld_nc(gamma + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = pack_bf16x2((bf16_lo(w[i]) * inv) * bf16_lo(gw[i]),
                         (bf16_hi(w[i]) * inv) * bf16_hi(gw[i]));
    *reinterpret_cast<uint4 *>(x + static_cast<size_t>(t) * H + k) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const moe_bf16 *r, int T, int H, const moe_bf16 *gamma, float eps,
                           moe_bf16 *x_next, cudaStream_t s) {
  rmsnorm_kernel<<<(T + kNormWarps - 1) / kNormWarps, 32 * kNormWarps, 0, s>>>(r, T, H, gamma,
                                                                              eps, x_next);
  return cudaGetLastError();
}

}  // namespace moe
