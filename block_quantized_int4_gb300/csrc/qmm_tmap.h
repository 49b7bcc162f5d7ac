// qmm_tmap.h -- TMA tensor descriptors for the streaming kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace qmm {

// Encode a 2D tiled TMA descriptor (row-major [outer][inner] tensor of
// `dt` elements, row pitch `row_bytes`) with the driver's encoder, fetched
// through the runtime; false if the encoder is unavailable or rejects it.
// Out-of-range boxes are zero-filled.
bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

// The same for a 3D view: dims[0] innermost (contiguous), strides in bytes
// of dims 1 and 2 (any order: a dim may step through memory more finely
// than the one inside it), box[i] elements along dim i.
bool make_tensor_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                        const uint64_t (&strides)[2], const uint32_t (&box)[3], CUtensorMapSwizzle sw);

}  // namespace qmm
