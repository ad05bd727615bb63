// Host helper: TMA tensor maps of the packed [S][H][d] bf16 tensors.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace ffa {

// Map of a bf16 tensor [seqlen][heads][d] as a 3-D tiled view (d, heads,
// seqlen) with a box of 64 x 1 x box_rows elements and the 128-byte swizzle:
// one box is a box_rows x 128-byte panel, exactly one K-major / MN-major
// swizzle column of the UMMA operand layouts.
inline bool make_tile_map(CUtensorMap* map, const void* ptr, int64_t seqlen, int32_t heads, int32_t d,
                          uint32_t box_rows = 128) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(seqlen)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of an fp32 tensor [seqlen][heads][d] (d <= 256) as (d, heads, seqlen)
// with a box of d x 1 x box_rows and no swizzle: one box is box_rows rows of
// d contiguous floats, the layout a reduce-add source tile is written in.
inline bool make_f32_row_map(CUtensorMap* map, const void* ptr, int64_t seqlen, int32_t heads, int32_t d,
                             uint32_t box_rows) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(seqlen)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(heads) * d * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 1, box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ffa
