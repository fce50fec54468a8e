// common.cuh -- device helpers shared by the sm_103a kernels of the MoE block.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

constexpr int kE = 256;   // routed experts
constexpr int kK = 8;     // top-k
constexpr int kG = 128;   // quantisation group along the reduction dim
constexpr int kMaxH = 8192;
constexpr int kMaxI = 2048;
constexpr int kMaxT = 65536;

// ------------------------------------------------------------- bf16 bits

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

// fp32 -> bf16, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16(lo)) | (static_cast<uint32_t>(f32_to_bf16(hi)) << 16);
}

// ------------------------------------------------------ int8 -> fp32 exact
//
// Four signed bytes of w become four fp32 values without an I2F: the byte is
// moved to offset binary (q + 128 in [0, 255]), placed in the low mantissa
// byte of 2^23 (bit pattern 0x4B0000uu == 2^23 + u), and 2^23 + 128 is
// subtracted, which is exact.
struct f4 { float x, y, z, w; };

__device__ __forceinline__ f4 i8x4_to_f32(uint32_t w) {
  const uint32_t u = w ^ 0x80808080u;
  const float bias = 8388736.0f;  // 2^23 + 128
  f4 r;
  r.x = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - bias;
  r.y = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - bias;
  r.z = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - bias;
  r.w = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - bias;
  return r;
}

// 4 int8 -> two f16x2, exact: each byte in offset binary (q + 128) becomes
// the low mantissa byte of 1024.0 (f16 0x6400 | u), and 1152 = 1024 + 128 is
// subtracted from both halves.  lo = bytes 0,1; hi = bytes 2,3.
__device__ __forceinline__ void i8x4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

// ----------------------------------------------------------- warp helpers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Exclusive prefix sum over threads 0..255 of the block (all threads of the
// block call it; tmp holds >= 8 ints of shared memory).
__device__ __forceinline__ int block_exclusive_scan_256(int v, int *tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (threadIdx.x < 256 && lane == 31) tmp[warp] = incl;
  __syncthreads();
  int base = 0;
  if (threadIdx.x < 256)
    for (int w = 0; w < warp; ++w) base += tmp[w];
  __syncthreads();
  return base + incl - v;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + expf(-g)) * u;
}

// Streamed-once weight loads: keep them out of L1 and give them the L2
// evict-first policy so that activations and lists stay resident.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(evict_first_policy()));
  return r;
}

__device__ __forceinline__ uint4 ld_nc(const void *p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Test-only builds.  A library compiled with MOE_SABOTAGE = n (never the
// product library, which defines nothing) plants one known mistake, so that
// the parity tests can show that they catch it: 1 moves the 8th selected id
// to the next expert not already chosen, 2 swaps the softmax weights of
// ranks 7 and 8 (0-based 6 and 7) without their ids, 3 drops the shared
// expert's gate, 4 reads the next quantisation group's scale in gate|up.
#ifndef MOE_SABOTAGE
#define MOE_SABOTAGE 0
#endif

// The scale group a gate|up weight in group g (of ng) is dequantised with.
__device__ __forceinline__ int gateup_scale_group(int g, int ng) {
  return MOE_SABOTAGE == 4 ? (g + 1) % ng : g;
}

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace moe
