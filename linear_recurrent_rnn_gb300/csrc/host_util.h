// Host utilities for the tensor-core kernels (see host_util.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rglru {

// Encodes a tiled TMA tensor map; dims / box are innermost first, strides_bytes has rank - 1
// entries (dims 1..rank-1).
cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        CUtensorMapSwizzle swizzle);

// Streaming multiprocessors of the current device (cached per device; 0 on error).
int sm_count();

}  // namespace rglru
