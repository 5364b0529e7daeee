// Conversions between row-major key rows (one 68-byte MXFP4 or 132-byte FP8 row per
// compressed position, the indexer cache as the attention.py page's
// DeepseekV4IndexerCache holds it: [num_blocks][block_size][row bytes]) and this
// library's 64-key pages, whose bytes are the same rows re-ordered into the tensor cores'
// core-matrix order (include/indexer.h states both formulas).
//
// One thread moves one 4-byte word: a row is 17 words (16 of codes, 1 of scales) in
// MXFP4 and 33 (32 + the f32 scale) in FP8. Every code word of a row stays within one
// 16-byte core-matrix row of the page, so a word is never split.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace indexer {

namespace {

template <bool FP8>
struct RowFmt {
  static constexpr int kRow = FP8 ? kRowBytesFp8 : kRowBytes;
  static constexpr int kCode = FP8 ? kCodeBytesFp8 : kCodeBytes;
  static constexpr int kGroup = FP8 ? kGroupBytesFp8 : kGroupBytes;
  static constexpr int kPage = FP8 ? kPageBytesFp8 : kPageBytes;
  static constexpr int kWords = kRow / 4;
};

// Byte offset within its page of word i of key m's row.
template <bool FP8>
__device__ __forceinline__ int page_word_offset(int m, int i) {
  using F = RowFmt<FP8>;
  const int j = 4 * i;
  if (j < F::kCode) return (m >> 3) * F::kGroup + (j >> 4) * 128 + (m & 7) * 16 + (j & 15);
  return (m >> 3) * F::kGroup + F::kCode * 8 + (m & 7) * 4;
}

template <bool FP8, bool TO_PAGES>
__global__ void __launch_bounds__(256) layout_kernel(const LayoutArgs a) {
  using F = RowFmt<FP8>;
  pdl_allow_next();
  pdl_wait();
  const long long n = (long long)a.n_seq * a.n_keys * F::kWords;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < n; g += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(g % F::kWords);
    const long long key = g / F::kWords;
    const int t = (int)(key % a.n_keys);
    const int b = (int)(key / a.n_keys);
    const size_t row_off = ((size_t)b * a.ld_rows + t) * F::kRow + 4 * i;
    const size_t page_off = ((size_t)b * (a.T_cap / kPageKeys) + t / kPageKeys) * F::kPage +
                            page_word_offset<FP8>(t % kPageKeys, i);
    if (TO_PAGES)
      *reinterpret_cast<uint32_t*>(a.pages + page_off) = *reinterpret_cast<const uint32_t*>(a.rows_in + row_off);
    else
      *reinterpret_cast<uint32_t*>(a.rows_out + row_off) = *reinterpret_cast<const uint32_t*>(a.pages_in + page_off);
  }
}

}  // namespace

cudaError_t launch_layout(const LayoutArgs& a, bool to_pages, cudaStream_t stream) {
  const long long words = (long long)a.n_seq * a.n_keys * (a.fp8 ? kRowBytesFp8 / 4 : kRowBytes / 4);
  if (words <= 0) return cudaSuccess;
  long long blocks = (words + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;   // grid-stride beyond 16 CTAs per SM
  const dim3 grid((unsigned)blocks), block(256);
  if (a.fp8)
    return to_pages ? launch_overlapped(layout_kernel<true, true>, grid, block, 0, stream, a)
                    : launch_overlapped(layout_kernel<true, false>, grid, block, 0, stream, a);
  return to_pages ? launch_overlapped(layout_kernel<false, true>, grid, block, 0, stream, a)
                  : launch_overlapped(layout_kernel<false, false>, grid, block, 0, stream, a);
}

}  // namespace indexer
