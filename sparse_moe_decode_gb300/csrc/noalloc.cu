// noalloc.cu -- moe_block_forward_noalloc: the block forward with its
// scratch in a fixed device array, for callers that cannot allocate.
//
// Some hosts of this library cannot call cudaMalloc where they run the
// block: a plugin inside an inference runtime that owns all device memory
// through its own pool, a process with a fixed device-memory budget in which
// any allocation at run time may fail, or a latency-critical path that cannot
// afford the implicit device synchronisation of cudaMalloc.  This entry point
// takes only inputs and outputs; its scratch is the array below, which every
// GPU that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "moe_gb300.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {nullptr};

// Device address of g_scratch on the current device, looked up once per
// device (with that device current) and cached.
moe_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_block_forward_noalloc(const moe_dims *dims, const moe_weights *w,
                                                const moe_bf16 *x, int T, moe_bf16 *out,
                                                void *stream) {
  // every host-side check comes before anything is enqueued: a rejected
  // call has no side effect
  moe_status st = moe::block_forward_check(dims, w, x, T, out);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  const size_t need = moe_workspace_bytes(dims, T);
  if (need == 0) return MOE_ERR_UNSUPPORTED;
  if (need > kScratchBytes) return MOE_ERR_WORKSPACE;
  void *scratch = nullptr;
  if ((st = scratch_address(&scratch)) != MOE_OK) return st;
  // The array keeps the previous call's contents; only the device status
  // word (first 256 bytes) must start at zero.  Everything else the block
  // reads is written earlier in the same call.
  if (cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return moe_block_forward(dims, w, x, T, out, nullptr, nullptr, nullptr, nullptr, scratch,
                           kScratchBytes, stream);
}
