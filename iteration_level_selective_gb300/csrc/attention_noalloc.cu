// orca_attention_noalloc: ragged attention for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any routine that allocates device
// memory) at the point where they run attention: for example a host
// runtime that hands out all device memory itself and forbids other
// allocations, or code running under a memory budget with no spare
// allocation.  They still own and pass the inputs (q, the K/V slots) and
// the output.  This entry point runs the same kernel as orca_attention, with
// its scratch (the request and work-item records, the key-split partials and
// their counters) in one file-scope device array of fixed size instead of a
// caller-provided workspace.
//
// Set-up: the first call on a device (per CUDA context), with that device
// current, looks up the array's device address (cudaGetSymbolAddress) and
// keeps it for later calls.  With lazy module loading that first lookup may
// make the driver load this library's device code and reserve the array, so
// make the first call early, where the caller may still allocate, and before
// any stream capture.  When the device's context changes (after a
// cudaDeviceReset, say) the next call repeats the set-up instead of reusing
// an address of the old context.  The array (kNoAllocScratchBytes) stays
// resident on every device that loads the library until the process exits.
// Every call shares it and it keeps the last call's contents: each call
// clears the counters it needs, and calls that overlap on the GPU (different
// streams, no ordering between them) race on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/orca.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB

__device__ __align__(256) unsigned char g_attention_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  CUcontext ctx;  // the context the address belongs to
  void *addr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// cuCtxGetCurrent through the runtime's driver entry point (no libcuda link).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// Device address of the scratch array in the current device's context
// (looked up once per context).
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ORCA_ECUDA;
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (!get_ctx) return ORCA_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return ORCA_ECUDA;
  ScratchAddr &slot = g_scratch_addr[dev];
  if (!slot.addr || !ctx || ctx != slot.ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attention_scratch) != cudaSuccess || !p) return ORCA_ECUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return ORCA_ECUDA;  // made current by the lookup
    slot.ctx = ctx;
    slot.addr = p;
  }
  *out = slot.addr;
  return ORCA_OK;
}

}  // namespace

extern "C" int orca_attention_noalloc(int32_t dtype, int32_t n_heads, int32_t head_dim, int64_t n_slots,
                                      const void *q, const void *k_layer, const void *v_layer, void *out,
                                      int32_t n_batch, const int32_t *row_off, const int32_t *ctx,
                                      const int64_t *slot_base, int32_t *status_dev, void *stream) {
  if (n_batch <= 0 || !row_off) return ORCA_EINVAL;
  size_t need = 0;
  int rc = orca_attention_workspace_bytes(n_batch, row_off[n_batch], n_heads, head_dim, &need);
  if (rc) return rc;
  if (need > kNoAllocScratchBytes) return ORCA_EBATCH;  // batch too large for the static scratch
  void *scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc) return rc;
  return orca_attention(dtype, n_heads, head_dim, n_slots, q, k_layer, v_layer, out, n_batch, row_off, ctx, slot_base,
                        scratch, kNoAllocScratchBytes, status_dev, stream);
}
