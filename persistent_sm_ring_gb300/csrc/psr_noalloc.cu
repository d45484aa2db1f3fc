// Allocation-free entry point: the ring-attention launch with its workspace
// taken from a fixed, file-scope device array instead of caller memory.
//
// Who needs it: callers that must not call cudaMalloc -- for example code
// running inside a host framework whose memory pool already owns the device
// memory, plug-ins that are not allowed to allocate, or latency-critical
// paths where cudaMalloc's implicit synchronisation is not acceptable.  They
// still pass their own inputs and outputs; only the scratch (ring slots,
// readiness flags, counters, queue) comes from here.
//
// Costs and limits:
//  * the array is PSR_NOALLOC_SCRATCH_BYTES (64 MiB) on every GPU that loads
//    this library, held until the process exits;
//  * shapes whose psr_workspace_bytes() exceed it are rejected;
//  * every call on a device shares the one array: two calls whose launches
//    overlap on the GPU (different streams, no ordering) race on it.
//    The control words and flags are cleared by each call before its launch;
//    the ring slots need no clearing (readiness flags guard every read).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/psr.h"

namespace {

constexpr size_t kScratchBytes = PSR_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, not a device address: the address is looked up per device below.
static __device__ __align__(256) unsigned char g_psr_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};  // per device ordinal, filled on first use

// Device address of g_psr_scratch on the current device (looked up once per
// device, with that device current).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PSR_ERR_CUDA;
  if (dev < 0 || dev >= 64) return PSR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_psr_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return PSR_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PSR_OK;
}

}  // namespace

extern "C" int psr_ring_attn_fwd_noalloc(const psr_shape* shape, const void* q, const void* k, const void* v, void* o,
                                         float* lse, const psr_partition* part, void* stream) {
  if (!shape) return PSR_ERR_ARG;
  const size_t need = psr_workspace_bytes(shape);
  if (need == 0) return PSR_ERR_UNSUPPORTED;              // not a supported shape at all
  if (need > kScratchBytes) return PSR_ERR_UNSUPPORTED;   // beyond the fixed scratch
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != PSR_OK) return rc;
  return psr_ring_attn_fwd(shape, q, k, v, o, lse, ws, kScratchBytes, part, stream);
}
