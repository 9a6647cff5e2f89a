// tensor_map.h — encoding of TMA tensor maps through the driver entry point
// obtained from the runtime (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gb300 {

// 3-D tiled map over a [planes, rows, inner] tensor (inner contiguous, rows
// `inner` elements apart, planes `plane_rows` rows apart; 0 = rows) with a
// box of box_inner x box_rows x 1 and 128-byte swizzle; out-of-range
// elements (rows >= `rows` included) read as zero.  Returns false if the
// driver rejects the map.
bool encode_tiled_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                     uint64_t inner, uint64_t rows, uint64_t planes, uint32_t elem_bytes,
                     uint32_t box_inner, uint32_t box_rows, uint64_t plane_rows = 0);

// 4-D tiled map over a [batches, heads, rows, inner] tensor with element
// strides row_stride, head_stride, batch_stride (inner contiguous; each
// stride times elem_bytes a multiple of 16), box box_inner x box_rows x 1 x 1,
// 128-byte swizzle unless given; out-of-range elements read as zero.  Returns
// false if the driver rejects the map.
bool encode_tiled_4d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                     uint64_t inner, uint64_t rows, uint64_t heads, uint64_t batches,
                     uint32_t elem_bytes, uint32_t box_inner, uint32_t box_rows,
                     uint64_t row_stride, uint64_t head_stride, uint64_t batch_stride,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// The same with a box of box_heads heads (128-byte swizzle): the box lands
// as box_heads x box_rows rows of box_inner elements, heads outermost.
bool encode_tiled_4d_box(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                         uint64_t inner, uint64_t rows, uint64_t heads, uint64_t batches,
                         uint32_t elem_bytes, uint32_t box_inner, uint32_t box_rows,
                         uint32_t box_heads, uint64_t row_stride, uint64_t head_stride,
                         uint64_t batch_stride);

}  // namespace gb300
