// dflash_ctx_fuse_noalloc: the context fuse for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they need the fuse: code running while another framework owns the device
// memory pool or has reserved all of it, code that must not grow the process
// footprint after start-up, or host code that only holds pointers it was
// handed.  This entry point takes only the inputs and the output; its scratch
// (the status word, the split counters and the fp32 pre-norm rows) lives in a
// fixed array in this file, which every GPU that loads the library keeps
// until the process exits.
#include <cstdint>
#include <mutex>

#include "dflash.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB per device
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device; the host-side symbol itself is not a device address).  The
// cached address belongs to the device's primary context: it is not looked
// up again after that context is destroyed (cudaDeviceReset).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return DFLASH_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return DFLASH_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" int dflash_ctx_fuse_noalloc(dflash_model m, const void* taps, int32_t T, void* ctx,
                                       void* stream) {
  if (m == nullptr || taps == nullptr || ctx == nullptr || T < 1) return DFLASH_ERR_INVALID_ARG;
  void* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  // Reject bad arguments and T beyond what fits in the fixed scratch
  // (DFLASH_ERR_CAPACITY) before touching the shared array, so that a call
  // that launches nothing does not clear the header under a call in flight.
  rc = dflash::ctx_fuse_check(m, taps, T, ctx, scratch, kNoAllocScratchBytes);
  if (rc) return rc;
  // the header (status word, split counters) must start at zero every call
  rc = dflash_workspace_init(scratch, kNoAllocScratchBytes, stream);
  if (rc) return rc;
  return dflash_ctx_fuse(m, taps, T, ctx, scratch, kNoAllocScratchBytes, stream);
}
