// Per-row selection kernels: the position-ordered top-k and the level-one candidate
// blocks. Both reduce to one CTA-wide primitive: among n order-preserving uint32 keys
// (0 = not selectable) keep the k largest, ties to the lower index, and emit their
// indices in ascending order.
//
// Selection is a most-significant-digit radix select (shared-memory histograms) that
// pins the k-th largest key K*, followed by an ordered compaction: every key > K* and the
// first `need` keys equal to K* (in index order) are written at their prefix-sum slot, so
// the output comes out sorted by position without a sort. The top-k kernel uses the
// register-resident form in select_common.cuh; the candidate-block kernel keeps its keys
// in shared memory.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"
#include "select_common.cuh"

namespace indexer {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;

// Adds 1 to hist[bin] for every lane whose `valid` is set, with one shared-memory atomic
// per distinct bin per warp (lanes holding the same bin are combined first, so a few hot
// bins do not serialise 32 atomics each). All 32 lanes of the warp must call it.
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t bin, bool valid) {
  const uint32_t tag = valid ? bin : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, tag);
  if (valid && (__ffs(peers) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

struct SelShared {
  uint32_t hist[256];
  uint32_t warp_tot[kSelWarps];
  uint32_t bcast[4];
};

// Exclusive prefix sum over the CTA (1024 threads); returns this thread's exclusive
// prefix and writes the total to *total.
__device__ __forceinline__ uint32_t cta_exclusive_scan(uint32_t v, uint32_t* total, SelShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sh.warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = sh.warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    sh.warp_tot[lane] = t;   // inclusive
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? sh.warp_tot[warp - 1] : 0u) + x - v;
  *total = sh.warp_tot[kSelWarps - 1];
  __syncthreads();
  return before;
}

// keys[0..n) in shared memory. Writes out[0..width): selected indices + offset in
// ascending order, then -1. k >= 1.
__device__ void cta_select(const uint32_t* keys, int n, int k, int32_t* out, int width, int offset,
                           SelShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kSelThreads - 1) / kSelThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);

  uint32_t nvalid_local = 0;
  for (int i = lo; i < hi; ++i) nvalid_local += keys[i] != 0u;
  uint32_t nvalid;
  cta_exclusive_scan(nvalid_local, &nvalid, sh);

  uint32_t kstar = 0u;        // select keys > kstar, plus `need` keys == kstar
  uint32_t need = 0u;
  if ((int)nvalid > k) {
    uint32_t prefix = 0u, mask = 0u;
    need = (uint32_t)k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) sh.hist[tid] = 0u;
      __syncthreads();
      for (int j = 0; j < per; ++j) {
        const int i = lo + j;
        const uint32_t key = i < hi ? keys[i] : 0u;
        hist_add_warp(sh.hist, (key >> shift) & 255u, key != 0u && (key & mask) == prefix);
      }
      __syncthreads();
      if (warp == 0) {
        // lane L owns bins 8L .. 8L+7; find the bin holding the need-th largest key
        uint32_t c[8], own = 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          c[q] = sh.hist[lane * 8 + q];
          own += c[q];
        }
        uint32_t incl = own;   // sum over lanes >= lane
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t y = __shfl_down_sync(0xffffffffu, incl, off);
          if (lane + off < 32) incl += y;
        }
        const uint32_t above = incl - own;
        if (above < need && need <= incl) {
          uint32_t acc = above;
          for (int q = 7; q >= 0; --q) {
            if (acc + c[q] >= need) {
              sh.bcast[0] = (uint32_t)(lane * 8 + q);
              sh.bcast[1] = acc;
              break;
            }
            acc += c[q];
          }
        }
      }
      __syncthreads();
      const uint32_t bin = sh.bcast[0];
      need -= sh.bcast[1];
      prefix |= bin << shift;
      mask |= 255u << shift;
      __syncthreads();
    }
    kstar = prefix;
  }

  // ordered compaction
  uint32_t eq_local = 0u, gt_local = 0u;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[i];
    gt_local += key > kstar;
    eq_local += (key == kstar && kstar != 0u);
  }
  uint32_t eq_total;
  const uint32_t eq_before = cta_exclusive_scan(eq_local, &eq_total, sh);
  const uint32_t eq_take = need > eq_before ? min(need - eq_before, eq_local) : 0u;
  uint32_t sel_total;
  uint32_t slot = cta_exclusive_scan(gt_local + eq_take, &sel_total, sh);
  uint32_t eq_seen = 0u;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[i];
    bool take = key > kstar;
    if (key == kstar && kstar != 0u) {
      take = eq_seen < eq_take;
      ++eq_seen;
    }
    if (take) out[slot++] = i + offset;
  }
  for (int i = (int)sel_total + tid; i < width; i += kSelThreads) out[i] = -1;
}

struct TopkKept {
  uint32_t kept[kCandMaxBlocks / 32];
};

// One CTA (1024 threads) per query row; thread t holds the keys of positions
// [t*KPT, (t+1)*KPT) in registers. Keys are the order-preserving images of the finite
// scores at t < vis (inside the kept candidate blocks, if any), 0 otherwise. Up to three
// radix passes pin the k_eff-th largest key and an ordered compaction writes the indices
// in position order (select_top). Rows with no candidate filter and vis <= k_eff take the
// short-context fill [0 .. vis).

template <int NT, int KPT>
__global__ void __launch_bounds__(NT, 1) topk_kernel(const TopkArgs a) {
  __shared__ SelectShared<NT> sh;
  __shared__ TopkKept kb;
  const int tid = threadIdx.x;
  pdl_allow_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int s = row % a.S;
  const int vis = min(a.T, (a.start_pos + s + 1) / a.ratio);
  const int k_eff = min(a.topk, a.T);
  int32_t* out = a.out + (size_t)row * a.topk;
  if (a.cand == nullptr && vis <= k_eff) {
    for (int i = tid; i < a.topk; i += NT) out[i] = i < vis ? i + a.offset : -1;
    return;
  }
  const int nblk_words = a.cand ? ((a.T + a.cbs - 1) / a.cbs + 31) / 32 : 0;
  if (a.cand) {
    for (int i = tid; i < nblk_words; i += NT) kb.kept[i] = 0u;
    __syncthreads();
    for (int i = tid; i < a.cbk; i += NT) {
      const int blk = a.cand[(size_t)row * a.cbk + i];
      if (blk >= 0 && blk < nblk_words * 32) atomicOr(&kb.kept[blk >> 5], 1u << (blk & 31));
    }
  }
  __syncthreads();

  const int base = tid * KPT;
  const float* src = a.scores + (size_t)row * a.T;
  auto make_key = [&](float f, int t) -> uint32_t {
    bool ok = t < vis && isfinite(f);
    if (ok && a.cand) {
      const int blk = t / a.cbs;
      ok = (kb.kept[blk >> 5] >> (blk & 31)) & 1u;
    }
    return ok ? order_key(f) : 0u;
  };
  uint32_t key[KPT];
  if ((a.T & 3) == 0) {   // rows start 16-byte aligned: float4 loads
#pragma unroll
    for (int j = 0; j < KPT; j += 4) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (base + j < vis) v = *reinterpret_cast<const float4*>(src + base + j);
      key[j] = make_key(v.x, base + j);
      key[j + 1] = make_key(v.y, base + j + 1);
      key[j + 2] = make_key(v.z, base + j + 2);
      key[j + 3] = make_key(v.w, base + j + 3);
    }
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j) key[j] = base + j < vis ? make_key(src[base + j], base + j) : 0u;
  }

  select_top<NT, KPT>(key, k_eff, out, a.topk, a.offset, sh, nullptr);
}

// One CTA per query row: block score = max finite score over the block's positions
// t < vis; ineligible blocks keep key 0; then cta_select over the blocks.
__global__ void __launch_bounds__(kSelThreads, 1) cand_kernel(const CandArgs a) {
  __shared__ uint32_t bkeys[kCandMaxBlocks];
  __shared__ SelShared sh;
  const int tid = threadIdx.x;
  pdl_allow_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int s = row % a.S;
  const int vis = min(a.T, (a.start_pos + s + 1) / a.ratio);
  const int nblk = (a.T + a.cbs - 1) / a.cbs;
  for (int i = tid; i < nblk; i += kSelThreads) bkeys[i] = 0u;
  __syncthreads();
  const float* src = a.scores + (size_t)row * a.T;
  for (int t = tid; t < vis; t += kSelThreads) {
    const float f = src[t];
    if (isfinite(f)) atomicMax(&bkeys[t / a.cbs], order_key(f));
  }
  __syncthreads();
  cta_select(bkeys, nblk, a.cbk, a.blocks + (size_t)row * a.cbk, a.cbk, 0, sh);
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  if (a.T <= kSelThreads * 8) {
    return launch_overlapped(topk_kernel<kSelThreads, 8>, dim3(a.rows), dim3(kSelThreads), 0, stream, a);
  } else if (a.T <= kSelThreads * 16) {
    return launch_overlapped(topk_kernel<kSelThreads, 16>, dim3(a.rows), dim3(kSelThreads), 0, stream, a);
  } else if (a.T <= kSelThreads * 32) {
    return launch_overlapped(topk_kernel<kSelThreads, 32>, dim3(a.rows), dim3(kSelThreads), 0, stream, a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_candidates(const CandArgs& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  return launch_overlapped(cand_kernel, dim3(a.rows), dim3(kSelThreads), 0, stream, a);
}

}  // namespace indexer
