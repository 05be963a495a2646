// Host side of the tensor-memory-accelerator (TMA) copies: the driver's
// tensor-map encoder, looked up once per process through the runtime (no
// link against the driver library), and a 2-D bf16 map with 128-byte swizzle.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums
#include <cuda_runtime.h>
#include <stdint.h>

namespace qsa {

using TensorMapEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                       const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                       const cuuint32_t *, CUtensorMapInterleave,
                                       CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);

inline TensorMapEncodeFn tensor_map_encoder() {
  static const TensorMapEncodeFn fn = []() -> TensorMapEncodeFn {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<TensorMapEncodeFn>(p);
    cudaGetLastError();
    return nullptr;
  }();
  return fn;
}

// A row-major bf16 matrix [rows, cols] (row pitch `pitch_elems`) read in boxes
// of box_cols x box_rows with 128-byte swizzle; rows past `rows` read as zero.
// Returns false if the encoder is missing or refuses the shape.
inline bool encode_bf16_sw128(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                              uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows) {
  const TensorMapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch_elems * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qsa
