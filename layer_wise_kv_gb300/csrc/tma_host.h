// Host-side construction of TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry-point query so the library does not link
// libcuda directly).
#pragma once

#include <cuda.h>
#include <cstdint>

namespace kvs {

// Tiled bf16 tensor map of rank 2..3 with 128-byte swizzle.  dims/strides are
// innermost first; strides[i] is the byte stride of dimension i + 1.  Returns
// false (and sets the error message) if the driver rejects it.
bool make_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* byte_strides, const uint32_t* box);

}  // namespace kvs
