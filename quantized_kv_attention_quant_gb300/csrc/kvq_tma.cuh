// Host side of the tensor memory accelerator: tensor maps for row-major
// [rows][heads][D] tensors of 16-bit values, read in 128-byte-swizzled boxes
// of 64 dims.  cuTensorMapEncodeTiled is taken from the driver through the
// runtime's entry-point query (no link against the driver library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace kvq {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A tensor [rows][heads][D] of 16-bit values (bf16 or f16) read in boxes of
// (64 dims, box_h heads, box_r rows), 128-byte swizzled; rows past the end
// read as zeros.  The base must be 16-byte aligned.
inline bool rows_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, int D, int heads, int rows,
                     int box_h, int box_r) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
  const cuuint32_t box[3] = {64u, (cuuint32_t)box_h, (cuuint32_t)box_r};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return fn(m, type, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace kvq
