// gdn_tmap.h -- tiled TMA tensor maps, encoded on the host through the CUDA runtime's entry
// point for the driver's cuTensorMapEncodeTiled (so the library does not link the driver
// library itself). Used by the dv-split decode (2-D boxes of the state pool) and the
// tensor-core prefill (3-D boxes of the token tensors).
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>

namespace gdn {

// `rank` dimensions, innermost first: `dims` elements each, `strides` the byte strides of
// dimensions 1 .. rank-1, `box` the box extent per dimension. No interleave, L2 promotion of
// 256 bytes, out-of-range elements read as zero. cudaErrorInvalidValue when the encoder
// rejects the arguments (alignment, extents).
inline cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, const void* base,
                                const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                                CUtensorMapSwizzle swizzle) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static std::atomic<Encode> fn{nullptr};
  Encode f = fn.load(std::memory_order_relaxed);
  if (f == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    const cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (err != cudaSuccess) return err;
    if (q != cudaDriverEntryPointSuccess || ptr == nullptr) return cudaErrorNotSupported;
    f = reinterpret_cast<Encode>(ptr);
    fn.store(f, std::memory_order_relaxed);
  }
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  const CUresult r = f(map, type, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace gdn
