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
//  * a device-side timeout is read with psr_noalloc_get_stats, which reads
//    the array's control block the way psr_get_stats reads a workspace.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/psr.h"
#include "psr_internal.h"

namespace {

constexpr size_t kScratchBytes = PSR_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, not a device address: the address is looked up per device below.
static __device__ __align__(256) unsigned char g_psr_scratch[kScratchBytes];

// Driver calls that identify the current context, so that a device whose primary context was
// reset (cudaDeviceReset) gets its address looked up again: the module is loaded anew there and
// the array may have moved.
struct CtxApi {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxApi& ctx_api() {
  static CtxApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      api.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      api.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  return api;
}

struct ScratchEntry {
  unsigned long long ctx_id = 0;  // context the address belongs to (0 = none yet)
  void* addr = nullptr;
};
std::mutex g_mu;
ScratchEntry g_scratch[64];  // per device ordinal

// Id of the context current on this thread, or 0 if there is none yet (the runtime creates the
// device's primary context on its first call that needs one).
unsigned long long current_ctx_id() {
  const CtxApi& api = ctx_api();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!api.get_current || !api.get_id || api.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      api.get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_psr_scratch on the current device.  It is looked up once per device and
// context, with that device current: on the first call, and again after the device's context
// was reset.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PSR_ERR_CUDA;
  if (dev < 0 || dev >= 64) return PSR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchEntry& e = g_scratch[dev];
  const unsigned long long id = current_ctx_id();
  if (e.addr == nullptr || id == 0 || e.ctx_id != id) {
    void* p = nullptr;
    const cudaError_t rc = cudaGetSymbolAddress(&p, g_psr_scratch);  // creates the context if needed
    if (rc != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return PSR_ERR_CUDA;
    }
    e.addr = p;
    e.ctx_id = current_ctx_id();  // 0 if it cannot be read: then every call looks the address up
  }
  *out = e.addr;
  return PSR_OK;
}

}  // namespace

extern "C" int psr_ring_attn_fwd_noalloc(const psr_shape* shape, const void* q, const void* k, const void* v, void* o,
                                         float* lse, const psr_partition* part, void* stream) {
  // the same checks, in the same order, as psr_ring_attn_fwd; then the fixed scratch's limit
  size_t need = 0;
  const int rc = psr_internal_fwd_check(shape, q, k, v, o, lse, &need);
  if (rc != PSR_OK) return rc;
  if (need > kScratchBytes) return PSR_ERR_UNSUPPORTED;
  void* ws = nullptr;
  const int ra = scratch_address(&ws);
  if (ra != PSR_OK) return ra;
  return psr_ring_attn_fwd(shape, q, k, v, o, lse, ws, kScratchBytes, part, stream);
}

extern "C" int psr_noalloc_get_stats(psr_stats* out, void* stream) {
  if (!out) return PSR_ERR_ARG;
  void* ws = nullptr;
  const int ra = scratch_address(&ws);
  if (ra != PSR_OK) return ra;
  return psr_get_stats(ws, out, stream);
}
