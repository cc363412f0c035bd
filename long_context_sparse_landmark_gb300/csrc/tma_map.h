// Host side of the TMA tensor maps used by the tensor-core kernels: the
// driver's cuTensorMapEncodeTiled, fetched once through the runtime, and the
// one map shape they use.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace msa {

constexpr int kMapD = 128;  // head dimension of every mapped tensor

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [rows, H, 128] bf16 tensor, boxes of 64 (d) x 1 (head) x box_rows (rows),
// 128-byte swizzle: each box lands as box_rows rows of 128 bytes, the
// canonical K-major SW128 layout for Q/K and the MN-major SW128 layout for V.
inline bool encode_map(EncodeTiledFn fn, CUtensorMap* m, const void* ptr, int64_t rows, int H,
                       uint32_t box_rows = 128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kMapD), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kMapD) * 2,
                           static_cast<cuuint64_t>(H) * kMapD * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows, H, 128] fp32 tensor, boxes of 32 (d) x 1 (head) x box_rows (rows),
// 128-byte swizzle: each box row is 128 bytes, as in the bf16 maps.
inline bool encode_map_f32(EncodeTiledFn fn, CUtensorMap* m, const void* ptr, int64_t rows, int H,
                           uint32_t box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kMapD), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kMapD) * 4,
                           static_cast<cuuint64_t>(H) * kMapD * 4};
  cuuint32_t box[3] = {32, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace msa
