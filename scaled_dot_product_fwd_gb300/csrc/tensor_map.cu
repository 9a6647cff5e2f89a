// tensor_map.cu — see tensor_map.h.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tensor_map.h"

namespace gb300 {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool encode_tiled_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                     uint64_t inner, uint64_t rows, uint64_t planes, uint32_t elem_bytes,
                     uint32_t box_inner, uint32_t box_rows, uint64_t plane_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  if (plane_rows == 0) plane_rows = rows;
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {inner * elem_bytes, inner * plane_rows * elem_bytes};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tiled_4d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                     uint64_t inner, uint64_t rows, uint64_t heads, uint64_t batches,
                     uint32_t elem_bytes, uint32_t box_inner, uint32_t box_rows,
                     uint64_t row_stride, uint64_t head_stride, uint64_t batch_stride,
                     CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {inner, rows, heads, batches};
  const cuuint64_t strides[3] = {row_stride * elem_bytes, head_stride * elem_bytes,
                                 batch_stride * elem_bytes};
  const cuuint32_t box[4] = {box_inner, box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dtype, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tiled_4d_box(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                         uint64_t inner, uint64_t rows, uint64_t heads, uint64_t batches,
                         uint32_t elem_bytes, uint32_t box_inner, uint32_t box_rows,
                         uint32_t box_heads, uint64_t row_stride, uint64_t head_stride,
                         uint64_t batch_stride) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {inner, rows, heads, batches};
  const cuuint64_t strides[3] = {row_stride * elem_bytes, head_stride * elem_bytes,
                                 batch_stride * elem_bytes};
  const cuuint32_t box[4] = {box_inner, box_rows, box_heads, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dtype, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace gb300
