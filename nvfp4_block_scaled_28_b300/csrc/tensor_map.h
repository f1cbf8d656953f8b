// Tensor-map (TMA descriptor) construction shared by the GEMM kernels.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace nvfp4 {

// 2-D tensor of `rows` rows of `inner` elements, `row_bytes` apart, copied
// in boxes of box_inner x box_rows; out-of-range box elements read as zero.
// False when the driver entry point is missing or rejects the layout.
bool make_map_2d(CUtensorMap *map, CUtensorMapDataType type, const void *ptr, uint64_t inner,
                 uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swz);

// 3-D tensor: dims {inner, d1, d2}, byte strides s1 (between d1 rows) and
// s2 (between d2 planes), boxes of box_inner x box1 x box2, no swizzle.
bool make_map_3d(CUtensorMap *map, CUtensorMapDataType type, const void *ptr, uint64_t inner,
                 uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2, uint32_t box_inner,
                 uint32_t box1, uint32_t box2);

}  // namespace nvfp4
