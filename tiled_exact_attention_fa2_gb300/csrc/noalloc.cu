// fa2_bwd_noalloc: the backward pass with its scratch in a fixed, statically
// allocated device array, for callers that cannot allocate device memory.
//
// Who needs this: code that runs where it may not call cudaMalloc /
// cudaMallocAsync itself, for example inside a host framework whose caching
// allocator owns all device memory and forbids side allocations, in plugins
// or embedded runtimes that are handed pre-sized buffers only, or in
// latency-critical loops where an allocation could block or fail at run time.
// Such callers still pass every input and output buffer; only the backward
// pass's internal scratch (D = rowsum(dO * O) and the fp32 dQ accumulator)
// comes from the array below.
//
// Cost and limits: the array (kNoAllocScratchBytes = 64 MiB) exists on every
// GPU that loads this library, for the life of the process.  A problem whose
// scratch, fa2_bwd_workspace_bytes(B, H, N, d), exceeds it is rejected with
// FA2_ERR_SCRATCH_CAPACITY before anything is enqueued.  All calls share the
// one array: calls whose GPU work overlaps in time (different streams, or
// different host threads, on the same device) race on it and give wrong
// results.  The dQ accumulator part is zeroed by the first kernel of every
// call, and D is fully rewritten, so no state leaks from one call to the next.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fa2.h"
#include "launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 256;

}  // namespace

// The scratch.  In host code this name is only a host-side handle for the
// symbol, not a device address; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_fa2_noalloc_scratch[kNoAllocScratchBytes];

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

}  // namespace

namespace fa2 {

// Unique id of the calling thread's current CUDA context (cuCtxGetId, reached
// through the runtime so the library needs no link-time libcuda), or 0 when
// there is none or it cannot be read.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

}  // namespace fa2

namespace {

using fa2::current_context_id;

struct ScratchSlot {
  void* ptr;                 // device address of the array in context ctx_id
  unsigned long long ctx_id;  // 0: not looked up yet
};
std::mutex g_setup_mu;
ScratchSlot g_slots[kMaxDevices] = {};

// Set-up, with the device current: look up the device address of the
// scratch array once per device and CUDA context (again after a device reset
// or a context switch, which change the context id; on every call if the id
// cannot be read).  Returns nullptr on failure.
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  ScratchSlot& slot = g_slots[dev];
  const unsigned long long id = current_context_id();
  if (slot.ptr && id != 0 && id == slot.ctx_id) return slot.ptr;
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_fa2_noalloc_scratch);
  if (e != cudaSuccess || !ptr) {
    cudaGetLastError();
    slot = ScratchSlot{};
    fa2::record_cuda_failure(static_cast<int>(e != cudaSuccess ? e : cudaErrorInvalidSymbol),
                             "cudaGetSymbolAddress (noalloc scratch)");
    return nullptr;
  }
  // The lookup makes the device's primary context current if no context was.
  slot = ScratchSlot{ptr, current_context_id()};
  return ptr;
}

}  // namespace

extern "C" {

size_t fa2_noalloc_scratch_capacity(void) { return kNoAllocScratchBytes; }

int fa2_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                    void* stream) {
  // The checks fa2_bwd makes, in its order, before the capacity check and
  // before any CUDA call.
  if (int rc = fa2::validate_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d, scale)) return rc;
  if (fa2_bwd_workspace_bytes(B, H, N, d) > kNoAllocScratchBytes) return FA2_ERR_SCRATCH_CAPACITY;
  void* scratch = scratch_for_current_device();
  if (!scratch) return FA2_ERR_CUDA;
  return fa2_bwd_ws(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, scratch, kNoAllocScratchBytes,
                    stream);
}

}  // extern "C"
