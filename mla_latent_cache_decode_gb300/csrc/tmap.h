// Host-side TMA tensor-map encoding for libmla's kernels: the driver's
// cuTensorMapEncodeTiled, found through the runtime (no link against
// libcuda), and the views of the latent cache and of q the kernels load.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {
namespace tmap {

constexpr int kRowDim = MLA_ROW_DIM;  // 576 elements per cached row

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

// [rows x 576] bf16 (row stride 1152 B) read in boxes {64 columns, box_rows}.
inline bool encode_2d(CUtensorMap *m, const void *base, int64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kRowDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kRowDim * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same rows viewed as {64 columns, rows, 9 chunks of 64 columns}: a box
// {64, box_rows, chunks} lands in shared memory chunk after chunk, each chunk
// box_rows x 128 B.
inline bool encode_3d(CUtensorMap *m, const void *base, int64_t rows, uint32_t box_rows,
               uint32_t chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(kRowDim / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)kRowDim * 2, 128};
  cuuint32_t box[3] = {64, box_rows, chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// FP8 cache [rows x 576] bytes (row stride 576 B), unswizzled: a box
// {64 bytes, box_rows} lands as box_rows rows of 64 bytes.
inline bool encode_2d_u8(CUtensorMap *m, const void *base, int64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kRowDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kRowDim};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The FP8 rows viewed as {64 bytes, rows, 9 chunks of 64 bytes}: a box
// {64, box_rows, chunks} lands chunk after chunk, each box_rows x 64 bytes.
inline bool encode_3d_u8(CUtensorMap *m, const void *base, int64_t rows, uint32_t box_rows,
                  uint32_t chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(kRowDim / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)kRowDim, 64};
  cuuint32_t box[3] = {64, box_rows, chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Slot of a pointer in a small direct-mapped cache of tensor maps.
inline size_t slot_of_ptr(const void *p, size_t slots) {
  const uint64_t x = (uint64_t)(uintptr_t)p;
  return (size_t)((x >> 8) ^ (x >> 20) ^ (x >> 32)) % slots;
}

}  // namespace tmap
}  // namespace mla
