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
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fa2.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 256;

}  // namespace

// The scratch.  In host code this name is only a host-side handle for the
// symbol, not a device address; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_fa2_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: look up the device address of
// the scratch array.  Returns nullptr on failure.
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fa2_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

size_t fa2_noalloc_scratch_capacity(void) { return kNoAllocScratchBytes; }

int fa2_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                    void* stream) {
  const size_t need = fa2_bwd_workspace_bytes(B, H, N, d);
  if (need > kNoAllocScratchBytes) return FA2_ERR_SCRATCH_CAPACITY;
  void* scratch = scratch_for_current_device();
  if (!scratch) return FA2_ERR_CUDA;
  // need == 0 means the sizes are invalid; fa2_bwd_ws reports which check failed.
  return fa2_bwd_ws(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, scratch, kNoAllocScratchBytes,
                    stream);
}

}  // extern "C"
