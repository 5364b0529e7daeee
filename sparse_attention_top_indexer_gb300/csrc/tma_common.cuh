// Tensor-map (TMA) helpers shared by the bf16 tcgen05 GEMM kernels (the fused query
// projection and the upstream producers): 2-D tiled copies of bf16 row-major matrices in
// K-chunks of 64 elements (128 bytes, one 128-byte swizzle row), and the matching
// shared-memory matrix descriptor.
#pragma once

#include <cuda.h>   // CUtensorMap and its enums (the encoder comes through the runtime)
#include <cuda_runtime.h>

#include <cstdint>

namespace indexer {

constexpr int kTmaK = 64;   // bf16 elements per K-chunk: 128 bytes, one swizzle row

// 2-D tensor-map copy of the box at (x, y) into shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

// Shared-memory matrix descriptor, K-major with the 128-byte swizzle: rows of 128 bytes, 8-row
// groups 1024 bytes apart (the layout a 128-byte-swizzled tensor-map copy writes at a
// 1024-byte aligned address); bits 46-48 hold 0b001, layout type 2 in bits 61-63. The K
// steps of 16 elements inside a row advance the start address by 32 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}


// cuTensorMapEncodeTiled, looked up once through the runtime (no link against the driver).
typedef CUresult (*TensorMapEncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                         const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                         CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline TensorMapEncodeTiled lookup_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  return e == cudaSuccess && q == cudaDriverEntryPointSuccess ? reinterpret_cast<TensorMapEncodeTiled>(fn) : nullptr;
}

inline cudaError_t encode_bf16_rows(CUtensorMap* map, const void* base, long long rows, int cols, int box_rows) {
  static const TensorMapEncodeTiled encode = lookup_encode();   // looked up once, thread-safely
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTmaK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


}  // namespace indexer
