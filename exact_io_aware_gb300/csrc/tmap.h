// Host-side TMA tensor-map encoding for [heads, rows, cols] 16-bit tensors.
//
// The driver entry point cuTensorMapEncodeTiled is looked up once through the runtime, so the
// library does not link against libcuda directly.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

namespace ea {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Map over a contiguous [heads][rows][cols] tensor of 16-bit elements, read in boxes of
// box_rows x box_cols with the swizzle of width 2 * box_cols bytes.  Rows past `rows` read as
// zero.  Returns false if the driver rejects the encoding.
inline bool encode_tile_map(CUtensorMap* map, const void* base, bool bf16, uint64_t heads,
                            uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const uint32_t row_bytes = box_cols * 2;
  CUtensorMapSwizzle swz = row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                           : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                             : CU_TENSOR_MAP_SWIZZLE_NONE;
  cuuint64_t dims[3] = {cols, rows, heads};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Map over a contiguous [heads][rows][cols] tensor of 8-bit elements, read in boxes of box_rows
// x box_cols bytes (32, 64 or 128) with the swizzle of that width.  cols must be a multiple of
// 16 (the row stride of a map is a multiple of 16 bytes).
inline bool encode_byte_map(CUtensorMap* map, const void* base, uint64_t heads, uint64_t rows,
                            uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  CUtensorMapSwizzle swz = box_cols == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                           : box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                            : CU_TENSOR_MAP_SWIZZLE_NONE;
  cuuint64_t dims[3] = {cols, rows, heads};
  cuuint64_t strides[2] = {cols, rows * cols};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Map over a contiguous [heads][rows][cols] float32 tensor, addressed in boxes of box_rows x
// box_cols (16 or 32 columns: 64- or 128-byte rows with the swizzle of that width).  Used for
// reduce-add of float32 tiles.
inline bool encode_f32_map(CUtensorMap* map, const void* base, uint64_t heads, uint64_t rows,
                           uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, heads};
  cuuint64_t strides[2] = {cols * 4, rows * cols * 4};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   box_cols * 4 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace ea
