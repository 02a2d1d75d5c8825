// skipsm_decode_noalloc: the Skip Softmax decode step for callers that cannot
// allocate device memory.
//
// The ordinary decode entry point asks its caller for a workspace (the per-split
// partial outputs and log-sum-exps).  Some callers cannot provide one: a plugin
// that runs inside a host framework owning every device allocation, a serving
// loop that must never call cudaMalloc (which can synchronise the device and
// stall other streams), or an embedding with no allocator at all.  This entry
// point keeps that workspace in a fixed array of device memory that belongs to
// the library, so the caller passes only inputs and outputs.
//
// Costs and rules of the fixed array:
//   * Every GPU that loads the library holds kScratchBytes (16 MiB) for as long
//     as the process lives.
//   * All calls share the one array.  Calls that can run at the same time on the
//     GPU (different streams, or different host threads, without ordering
//     between them) race on it and produce garbage; order them.
//   * The array keeps whatever the last call left in it.  Nothing in it needs
//     to start at zero: every partial that the combine step reads was written
//     by the split step of the same call.
//   * The first call on each device looks up the array's device address (one
//     cudaGetSymbolAddress with that device current).  Make that first call
//     before starting any stream capture on the device.  The address is kept
//     with the id of the context it belongs to; a call from another context
//     (or after a device reset recreated the primary context) looks it up again,
//     so such a call, too, must come before any capture.
#include <cstring>
#include <mutex>

#include "../../include/skipsm.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = SKIPSM_DECODE_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size keeps 256-byte alignment");

// The workspace of every skipsm_decode_noalloc call, on every device.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_lookup_mu;
struct ScratchSlot {
  unsigned long long ctx;  // id of the context the address belongs to
  void* ptr;
};
ScratchSlot g_scratch[64] = {};

// Device address of g_decode_scratch in the context current on this thread.  It is
// looked up once per device (cudaGetSymbolAddress with that device current) and again
// only if the current context is not the one it was looked up in (a device reset
// that recreated the primary context, or another context made current).
skipsm_status scratch_on_current_device(void** out, int* dev_out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return SKIPSM_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SKIPSM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_lookup_mu);
  unsigned long long ctx = skipsm::current_context_id();
  if (!g_scratch[dev].ptr || ctx == 0 || g_scratch[dev].ctx != ctx) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess || ptr == nullptr) return SKIPSM_ERR_CUDA;
    if (ctx == 0) ctx = skipsm::current_context_id();
    g_scratch[dev] = ScratchSlot{ctx, ptr};
  }
  *out = g_scratch[dev].ptr;
  *dev_out = dev;
  return SKIPSM_OK;
}

}  // namespace

extern "C" skipsm_status skipsm_decode_noalloc(const void* q, const void* k, const void* v,
                                               void* o, int B, int Hq, int Hkv, int Skv, int D,
                                               float lambda, uint64_t* skip_counts,
                                               void* stream) {
  const size_t need = skipsm_decode_workspace_size(B, Hq, Hkv, Skv, D, 0);
  if (need == 0) {
    // invalid sizes: let the ordinary entry point name the problem
    return skipsm_decode(q, k, v, o, B, Hq, Hkv, Skv, D, lambda, skip_counts, nullptr, 0, stream);
  }
  if (need > kScratchBytes) {
    // the message goes through the ordinary entry point's error path, which
    // reports the bytes needed; nothing is launched
    return skipsm_decode(q, k, v, o, B, Hq, Hkv, Skv, D, lambda, skip_counts, nullptr,
                         kScratchBytes, stream);
  }
  void* scratch = nullptr;
  int dev = -1;
  const skipsm_status st = scratch_on_current_device(&scratch, &dev);
  if (st != SKIPSM_OK) return st;
  return skipsm_decode(q, k, v, o, B, Hq, Hkv, Skv, D, lambda, skip_counts, scratch,
                       kScratchBytes, stream);
}
