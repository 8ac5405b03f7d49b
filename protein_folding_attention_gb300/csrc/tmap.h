// Host-side construction of TMA tensor maps (cuTensorMapEncodeTiled through
// the runtime's driver entry point, so the library needs no link-time
// dependency on libcuda).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace evo {

// Returns the driver's cuTensorMapEncodeTiled, or nullptr if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Encodes a tiled bf16 tensor map.  dims/strides are innermost first; strides
// are in bytes for dims 1..rank-1 (dim 0 is contiguous).  `promotion` is the
// L2 fetch granularity of the box's rows.  Returns false if the driver
// rejects the map.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* byte_strides, const uint32_t* box,
                    CUtensorMapSwizzle swizzle,
                    CUtensorMapL2promotion promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

}  // namespace evo
