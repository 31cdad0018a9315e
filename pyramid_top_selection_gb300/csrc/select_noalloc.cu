// Fixed scratch for pisa_select_noalloc: the selection's workspace lives in a file-scope
// device array of the library instead of a caller-provided buffer.
//
// The array is part of the library's device image, so every GPU on which the library is
// loaded holds it (kNoAllocScratchBytes) until the process exits. Its device address is
// looked up once per device, on the first pisa_select_noalloc call made with that device
// current; that first call should therefore come before any stream capture on the device.
// All calls share the one array and it keeps the last call's contents: the selection clears
// the parts that must start at zero (its grouping counters) on the stream before use, and
// two calls whose GPU work overlaps (different streams, or different host threads on one
// device) race on the array.
#include <mutex>

#include "device.cuh"

namespace pisa {

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device (looked up on first use).
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_select_scratch);
    if (e != cudaSuccess) return static_cast<int>(e);
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return 0;
}

}  // namespace pisa
