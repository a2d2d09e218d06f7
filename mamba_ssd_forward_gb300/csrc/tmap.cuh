// Host-side construction of TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry-point query so the library does not
// link libcuda directly).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

// A rank-`rank` (<= 5) tiled map with 128-byte swizzling and zero fill for
// out-of-range elements.  dims[] are element extents, innermost first;
// strides[] the byte strides of dims 1..rank-1; box[] the tile extents
// (box[0] * element size must be <= 128 bytes).  Returns false on failure.
bool make_tmap_sw128(CUtensorMap *map, const void *base, bool bf16, int rank,
                     const uint64_t *dims, const uint64_t *strides, const uint32_t *box);

}  // namespace ssd
