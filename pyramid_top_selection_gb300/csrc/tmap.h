// Host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled, reached through the CUDA
// runtime's driver entry point so the library does not link the driver API directly).
#pragma once

#include <cuda.h>
#include <cstdint>

namespace pisa {

// Tiled map of a row-major tensor: dims/box innermost first, byte strides of dims 1..rank-1,
// 128-byte swizzle, zero fill out of bounds. Returns 0 or a cudaError_t-compatible code.
int encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace pisa
