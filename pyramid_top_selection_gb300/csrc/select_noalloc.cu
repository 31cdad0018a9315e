// Fixed scratch for pisa_select_noalloc: the selection's workspace lives in a file-scope
// device array of the library instead of a caller-provided buffer.
//
// The array is part of the library's device image. With CUDA's default lazy module loading,
// that image (the array and the selection kernels) is loaded on a device by the first call
// that needs it there, so the driver reserves the array's memory inside the first
// pisa_select_noalloc call on each device; callers that allow no device allocation while
// serving make one warm-up call per device at set-up (or run with CUDA_MODULE_LOADING=EAGER),
// and that first call should come before any stream capture on the device. The array's
// device address is looked up on every call (cheap once the image is loaded), with the
// calling device current, so a device reset in between leaves no stale address behind.
// All calls share the one array and it keeps the last call's contents: the selection clears
// the parts that must start at zero (its grouping counters) on the stream before use, and
// two calls whose GPU work overlaps (different streams, or different host threads on one
// device) race on the array.
#include "device.cuh"

namespace pisa {

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB

static __device__ __align__(256) unsigned char g_select_scratch[kNoAllocScratchBytes];

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device. In host code the array's name
// stands for a host-side shadow, not a device address, so the address is asked for here.
int noalloc_scratch(void** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_select_scratch);
  if (e != cudaSuccess) return static_cast<int>(e);
  *out = ptr;
  return 0;
}

}  // namespace pisa
