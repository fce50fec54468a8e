// tc_gemm.cu -- prefill-size T: the router logits (A1) as a GEMM on the
// 5th-generation tensor cores (tcgen05, TMEM, TMA), and the TMA helpers the
// expert GEMMs share.
//
// Orientation: D[expert, token] = sum_k Wr[expert, k] * x[token, k].  128
// router rows are the M = 128 operand, a tile of 32 tokens is N, so that a
// prefill chunk spreads over the SMs.  TMA brings
// both bf16 operands into shared memory in the canonical K-major
// SWIZZLE_128B layout; one thread issues tcgen05.mma (bf16 x bf16 -> fp32)
// over the reduction; the epilogue warps read it back (tcgen05.ld) and store
// the logits.  At N = 32 a tile costs more MMA issue than data, so two
// issuing threads share it: one takes the ring stages (64-wide K steps) of
// even index, the other those of odd index (so each ring slot always serves
// the same issuer), each into its own TMEM accumulator, and the epilogue
// adds the two (in that fixed order); the accumulator pairs are
// double-buffered across a CTA's tiles.
//
// Warp roles (224 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the even-step MMAs, warp 6 the odd-step ones, warps 2..5 (one per
// TMEM lane quarter) write the logits.  Every wait is
// bounded by a %globaltimer budget; on expiry the CTA drains what it has in
// flight, frees TMEM, sets MOE_DEV_TIMEOUT and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kRThreads = 224;
constexpr int kRStages = 8;                 // shared-memory ring depth
constexpr int kRTok = 32;                   // tokens per item (N)
constexpr uint32_t kRABytes = 128 * 128;    // 128 rows x 64 bf16 of K
constexpr uint32_t kRBBytes = kRTok * 128;  // 32 rows x 64 bf16 of K
constexpr uint32_t kRStageBytes = kRABytes + kRBBytes;
constexpr uint32_t kRTmemCols = 128;        // two buffers x two issuers x 32 columns
constexpr size_t kROffBar = kRStages * kRStageBytes;
constexpr size_t kRSmem = kROffBar + 256 + 1024;  // + barriers + alignment slack

struct RBars {
  uint64_t full[kRStages], empty[kRStages], acc_full[2], acc_empty[2], done[2];
  uint32_t tmem_holder;
  int abort;
};
static_assert(sizeof(RBars) <= 256, "barrier block");

// Items it = 2 * token tile + row tile; logits [T][kE].
__global__ void __launch_bounds__(kRThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 int T, int H, float *__restrict__ logits, uint32_t *status,
                 unsigned long long budget, int32_t *__restrict__ zero_counts) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  RBars *bars = reinterpret_cast<RBars *>(smem + kROffBar);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = 2 * ((T + kRTok - 1) / kRTok);
  const int nk = H / 64;
  if (zero_counts && blockIdx.x == 0)  // per-expert counts of the selection that follows
    for (int i = threadIdx.x; i < kE; i += blockDim.x) zero_counts[i] = 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRStages; ++i) {
      ptx::mbar_init(&bars->full[i], 1);
      ptx::mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->acc_full[i], 2);  // both issuers
      ptx::mbar_init(&bars->acc_empty[i], 4);
      ptx::mbar_init(&bars->done[i], 1);
    }
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_holder, kRTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_holder;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------ TMA producer
      ptx::tma_prefetch_desc(&tmW);
      ptx::tma_prefetch_desc(&tmX);
      const uint64_t pol = ptx::policy_evict_last();
      uint32_t n = 0;
      bool stop = false;
      for (int it = blockIdx.x; it < n_items && !stop; it += gridDim.x) {
        const int m = it & 1, t0 = (it >> 1) * kRTok;
        for (int k = 0; k < nk; ++k, ++n) {
          const uint32_t s = n % kRStages;
          if (!ptx::mbar_wait(&bars->empty[s], ((n / kRStages) & 1) ^ 1, abort, budget)) { stop = true; break; }
          uint8_t *dst = smem + s * kRStageBytes;
          ptx::mbar_expect_tx(&bars->full[s], kRStageBytes);
          ptx::tma_load_2d(dst, &tmW, k * 64, m * 128, &bars->full[s], pol);
          ptx::tma_load_2d(dst + kRABytes, &tmX, k * 64, t0, &bars->full[s], pol);
        }
      }
      if (*abort) {  // let the copies in flight land before exiting
        int never = 0;
        for (uint32_t k = 0; k < kRStages && k < n; ++k) {
          const uint32_t j = n - 1 - k;
          ptx::mbar_wait(&bars->full[j % kRStages], (j / kRStages) & 1, &never, ptx::kDrainBudgetNs);
        }
      }
    }
  } else if (warp == 1 || warp == 6) {
    if (lane == 0) {  // ------------------------------------ MMA issuers
      const int half = warp == 1 ? 0 : 1;  // ring stages n with n mod 2 = half
      const uint32_t idesc = ptx::idesc_bf16_f32(128, kRTok);
      uint32_t ni = 0;
      bool issued = false;
      for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x, ++ni) {
        const uint32_t ab = ni & 1;
        if (!ptx::mbar_wait(&bars->acc_empty[ab], ((ni >> 1) & 1) ^ 1, abort, budget)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + ab * 2 * kRTok + half * kRTok;
        const int k0 = (half - static_cast<int>(ni * nk)) & 1;  // first K step of this issuer
        for (int k = k0; k < nk; k += 2) {
          const uint32_t n = ni * nk + k;  // ring stage of this K step
          const uint32_t s = n % kRStages;
          if (!ptx::mbar_wait(&bars->full[s], (n / kRStages) & 1, abort, budget)) break;
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smem + s * kRStageBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_bf16(d, ptx::sw128_desc(a0 + kk * 32),
                          ptx::sw128_desc(a0 + kRABytes + kk * 32), idesc, k > k0 || kk > 0);
          ptx::mma_commit(&bars->empty[s]);
          issued = true;
        }
        if (*abort) break;
        ptx::mma_commit(&bars->acc_full[ab]);  // with no MMAs (nk = 1): at once
      }
      if (issued) {  // all MMAs complete before TMEM is released
        ptx::mma_commit(&bars->done[half]);
        int never = 0;
        ptx::mbar_wait(&bars->done[half], 0, &never, ptx::kDrainBudgetNs);
      }
    }
  } else {
    // -------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const uint32_t tl = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t ni = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++ni) {
      const uint32_t ab = ni & 1;
      if (!ptx::mbar_wait(&bars->acc_full[ab], (ni >> 1) & 1, abort, budget)) break;
      ptx::tc_fence_after();
      float v[32], v2[32];
      // nk = 1: the tile's one K step went to the issuer of its stage's parity
      const uint32_t only = (ni * nk) & 1;
      ptx::tmem_ld32(tmem + tl + ab * 2 * kRTok + (nk > 1 ? 0 : only * kRTok), v);
      if (nk > 1) ptx::tmem_ld32(tmem + tl + ab * 2 * kRTok + kRTok, v2);
      ptx::tmem_wait_ld();
      if (nk > 1) {
#pragma unroll
        for (int j = 0; j < kRTok; ++j) v[j] += v2[j];  // issuer 0's sum, then issuer 1's
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->acc_empty[ab]);
      const int e = (it & 1) * 128 + quarter * 32 + lane, t0 = (it >> 1) * kRTok;
#pragma unroll
      for (int j = 0; j < kRTok; ++j)
        if (t0 + j < T) logits[static_cast<size_t>(t0 + j) * kE + e] = v[j];
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kRTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_status(status, MOE_DEV_TIMEOUT);
}

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

}  // namespace

bool tc_make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
                 uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
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

bool tc_make_map3(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
                  const uint64_t dims[3], const uint64_t strides[2], const uint32_t box[3]) {
  EncodeTiledFn enc = encoder();
  if (!enc || !base) return false;
  const cuuint64_t gdim[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t gstride[2] = {strides[0], strides[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  (void)esize;
  return enc(m, dt, 3, const_cast<void *>(base), gdim, gstride, bx, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_make_map_nd(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int rank,
                    const uint64_t *dims, const uint64_t *strides, const uint32_t *box) {
  EncodeTiledFn enc = encoder();
  if (!enc || !base || rank < 1 || rank > 5) return false;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bx[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bx[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) gstride[i] = strides[i];
  }
  return enc(m, dt, static_cast<cuuint32_t>(rank), const_cast<void *>(base), gdim, gstride, bx,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_sm_count() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev] > 0 ? n[dev] : 148;
}

unsigned long long tc_wait_budget_ns() {
  static unsigned long long v = 0;
  if (!v) {
    const char *e = getenv("MOE_WAIT_BUDGET_NS");
    v = e ? strtoull(e, nullptr, 10) : 2000000000ull;
    if (!v) v = 1;
  }
  return v;
}

cudaError_t launch_router_tc(const moe_bf16 *x, int T, int H, const moe_bf16 *w_router,
                             float *logits, uint32_t *status, cudaStream_t s,
                             int32_t *zero_counts) {
  CUtensorMap a, b;
  if (!tc_make_map(&a, w_router, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kE, H, 128, 64) ||
      !tc_make_map(&b, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, kRTok, 64))
    return cudaErrorInvalidValue;
  static bool attr[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(router_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kRSmem));
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  const int n_items = 2 * ((T + kRTok - 1) / kRTok);
  const int grid = n_items < tc_sm_count() ? n_items : tc_sm_count();
  router_tc_kernel<<<grid, kRThreads, kRSmem, s>>>(a, b, T, H, logits, status,
                                                   tc_wait_budget_ns(), zero_counts);
  return cudaGetLastError();
}

}  // namespace moe
