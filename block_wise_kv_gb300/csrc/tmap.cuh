// tmap.cuh — host helpers to encode TMA tensor maps (2-D, 128-byte swizzle).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dllm {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).  Resolved once; nullptr if unavailable.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Row-major [rows][cols] tensor of elem_bytes-sized elements (rows densely
// packed), loaded in boxes of box_cols x box_rows with 128-byte swizzling
// (box_cols * elem_bytes must be 128).  Out-of-range rows read as zero.
inline cudaError_t encode_2d_sw128(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* ptr,
                                   uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Row-major [n2][n1][cols] tensor (cols innermost, all dense), loaded in
// boxes of box_cols x 1 x box_n2 with 128-byte swizzling: box_n2 rows of
// box_cols elements taken at a stride of n1 * cols (one fixed middle index).
// Out-of-range rows read as zero.
inline cudaError_t encode_3d_rows_sw128(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* ptr,
                                        uint64_t cols, uint64_t n1, uint64_t n2, uint32_t box_cols,
                                        uint32_t box_n2) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {cols, n1, n2};
  cuuint64_t strides[2] = {cols * static_cast<uint64_t>(elem_bytes), n1 * cols * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[3] = {box_cols, 1, box_n2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace dllm
