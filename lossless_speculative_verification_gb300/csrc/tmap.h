// tmap.h -- host-side creation of TMA tensor maps (2-D bf16, 128-byte swizzle).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lsv {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box = 64 columns x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
inline bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if (rows == 0) rows = 1;  // an empty tensor still needs a valid map; nothing reads it
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Gate/up weights as pairs: the gate row r and its up row r + half_rows of a
// [.., cols] bf16 matrix, viewed as dims {cols, 2, rows}.  A box {64, 2, 64}
// stages 64 features as 128 interleaved rows (gate 0, up 0, gate 1, up 1, ...)
// with the 128-byte swizzle, so that an MMA puts each feature's gate and up
// products in neighbouring accumulator lanes.  Only rows r whose up row
// r + half_rows exists may be requested.
inline bool make_map_gu(CUtensorMap* m, const void* base, uint64_t rows, uint64_t half_rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if (rows == 0) rows = 1;
  if (half_rows == 0) half_rows = 1;
  const cuuint64_t dims[3] = {cols, 2, rows};
  const cuuint64_t strides[2] = {half_rows * cols * 2, cols * 2};
  const cuuint32_t box[3] = {64, 2, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace lsv
