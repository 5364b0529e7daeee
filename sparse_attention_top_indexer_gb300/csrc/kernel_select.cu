// Per-row selection kernels: the position-ordered top-k and the level-one candidate
// blocks. Both reduce to one CTA-wide primitive: among n order-preserving uint32 keys
// (0 = not selectable) keep the k largest, ties to the lower index, and emit their
// indices in ascending order.
//
// Selection is a most-significant-digit radix select (shared-memory histograms) that
// pins the k-th largest key K*, followed by an ordered compaction: every key > K* and the
// first `need` keys equal to K* (in index order) are written at their prefix-sum slot, so
// the output comes out sorted by position without a sort. Both kernels use the
// register-resident form in select_common.cuh.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"
#include "select_common.cuh"

namespace indexer {

namespace {

constexpr int kSelThreads = 1024;

// (vis, T) of a row: keys it may see and keys of its sequence, from the per-row metadata
// of a batch with per-sequence positions, or from the uniform S / start_pos.
__device__ __forceinline__ int2 row_extent(const RowInfo* ri, int row, int S, int T, int start_pos, int ratio) {
  if (ri != nullptr) {
    const RowInfo r = ri[row];
    const int t = max(0, min(r.T, T));
    return make_int2(max(0, min(r.vis, t)), t);
  }
  return make_int2(min(T, (start_pos + row % S + 1) / ratio), T);
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

// Many rows per SM: the 256-thread builds are register-capped so that more rows share an SM
// and hide more of each row's latency chain. 32 keys a thread at 40 registers (six CTAs; the
// large prefill 0.621 ms against 0.679 with four CTAs at 64 registers and 0.627 with five at
// 48, although the cap spills some keys to local memory, which stays in L1; eight CTAs at 32
// registers spill more and take 0.755 ms); 8 keys at 32 registers (eight CTAs, no spills;
// the 2048-key prefill 30.5 against 33.2 us with six).
constexpr int topk_min_ctas(int NT, int KPT) { return NT != 256 ? 1 : KPT == 32 ? 6 : KPT == 8 ? 8 : 1; }

template <int NT, int KPT>
__global__ void __launch_bounds__(NT, topk_min_ctas(NT, KPT)) topk_kernel(const TopkArgs a) {
  __shared__ SelectShared<NT> sh;
  __shared__ TopkKept kb;
  const int tid = threadIdx.x;
  pdl_allow_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int2 ext = row_extent(a.rinfo, row, a.S, a.T, a.start_pos, a.ratio);
  const int vis = ext.x;
  const int k_eff = min(a.topk, ext.y);
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

  // keys a thread holds: the row's visible positions spread over all threads, four at a time
  // (a row that sees fewer than NT * KPT positions then takes fewer instructions per thread
  // in every per-key loop, instead of leaving the threads past it idle)
  const int kpt = min(KPT, max(4, (((vis + NT - 1) / NT) + 3) & ~3));
  const int base = tid * kpt;
  const float* src = a.scores + (size_t)row * a.ld;
  auto make_key = [&](float f, int t) -> uint32_t { return t < vis && isfinite(f) ? order_key(f) : 0u; };
  uint32_t key[KPT];
#pragma unroll
  for (int j = 0; j < KPT; ++j) key[j] = 0u;
  if (base < vis) {   // threads past the visible positions hold no key
    if ((a.ld & 3) == 0) {   // rows start 16-byte aligned (base is a multiple of 4): float4 loads
      for_keys<KPT>(kpt, [&](int j) {
        if ((j & 3) == 0 && base + j < vis) {
          const float4 v = *reinterpret_cast<const float4*>(src + base + j);
          key[j] = make_key(v.x, base + j);
          key[j + 1] = make_key(v.y, base + j + 1);
          key[j + 2] = make_key(v.z, base + j + 2);
          key[j + 3] = make_key(v.w, base + j + 3);
        }
      });
    } else {
      for_keys<KPT>(kpt, [&](int j) {
        if (base + j < vis) key[j] = make_key(src[base + j], base + j);
      });
    }
    if (a.cand) {   // the candidate filter: positions outside the kept blocks hold no key
      for_keys<KPT>(kpt, [&](int j) {
        const int blk = (base + j) / a.cbs;   // < the row's blocks where key[j] != 0 (t < vis <= T)
        if (key[j] != 0u && !((kb.kept[blk >> 5] >> (blk & 31)) & 1u)) key[j] = 0u;
      });
    }
  }

  select_top<NT, KPT>(key, k_eff, out, a.topk, a.offset, sh, vis, kpt);
}

// Level two with one query row: the top-k over the kept candidate blocks only. The row's
// kept blocks (deduplicated, ascending) are gathered into a list of E = nb * cbs
// positions; thread t takes list entries [t*KPT, (t+1)*KPT) -- still in position order --
// and select_top returns list indices, which are then mapped back to positions. The
// selection equals topk_kernel's with the same filter: same keys, same order.
template <int NT>
struct SparseShared {
  SelectShared<NT> sel;
  uint32_t bits[kCandMaxBlocks / 32];
  int blist[kCandMaxBlocks];
  int nb;
};

template <int NT, int KPT>
__global__ void __launch_bounds__(NT, 1) topk_sparse_kernel(const TopkArgs a) {
  __shared__ SparseShared<NT> sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_allow_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int2 ext = row_extent(a.rinfo, row, a.S, a.T, a.start_pos, a.ratio);
  const int vis = ext.x;
  const int k_eff = min(a.topk, ext.y);
  int32_t* out = a.out + (size_t)row * a.topk;
  const int nblk = (a.T + a.cbs - 1) / a.cbs;
  const int nw = (nblk + 31) / 32;
  for (int i = tid; i < nw; i += NT) sh.bits[i] = 0u;
  __syncthreads();
  for (int i = tid; i < a.cbk; i += NT) {
    const int blk = a.cand[(size_t)row * a.cbk + i];
    if (blk >= 0 && blk < nblk) atomicOr(&sh.bits[blk >> 5], 1u << (blk & 31));
  }
  __syncthreads();
  if (warp == 0) {   // ascending list of the kept blocks
    int total = 0;
    for (int w0 = 0; w0 < nw; w0 += 32) {
      const uint32_t word = w0 + lane < nw ? sh.bits[w0 + lane] : 0u;
      const int cnt = __popc(word);
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      int slot = total + incl - cnt;
      for (uint32_t w = word; w; w &= w - 1) sh.blist[slot++] = (w0 + lane) * 32 + (__ffs(w) - 1);
      total += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sh.nb = total;
  }
  __syncthreads();
  const int E = sh.nb * a.cbs;
  const float* src = a.scores + (size_t)row * a.ld;
  auto pos_of = [&](int e) { return sh.blist[e / a.cbs] * a.cbs + e % a.cbs; };
  uint32_t key[KPT];
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int e = tid * KPT + j;
    key[j] = 0u;
    if (e < E) {
      const int t = pos_of(e);
      if (t < vis) {
        const float f = src[t];
        if (isfinite(f)) key[j] = order_key(f);
      }
    }
  }
  select_top<NT, KPT>(key, k_eff, out, a.topk, 0, sh.sel, E);
  __syncthreads();   // every list index is written
  for (int i = tid; i < a.topk; i += NT) {
    const int g = out[i];
    if (g >= 0) out[i] = pos_of(g) + a.offset;
  }
}

// One CTA per query row. Block score = max finite score over the block's positions
// t < vis; a block with none keeps key 0 (ineligible). Thread t loads the PPT positions
// [t*PPT, (t+1)*PPT) at once, folds them into a running maximum per block and merges each
// block it touches with one shared-memory atomicMax. The blocks' keys then go to
// registers (BPT consecutive blocks per thread) and select_top keeps the cbk best, ties to
// the lower block, in ascending block order.
union CandShared {
  uint32_t bkeys[kCandMaxBlocks];
  SelectShared<kSelThreads> sel;   // reused once the block keys are in registers
};

template <int PPT, int BPT>
__global__ void __launch_bounds__(kSelThreads, 1) cand_kernel(const CandArgs a) {
  __shared__ CandShared sh;
  const int tid = threadIdx.x;
  pdl_allow_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int vis = row_extent(a.rinfo, row, a.S, a.T, a.start_pos, a.ratio).x;
  const int nblk = (a.T + a.cbs - 1) / a.cbs;
  for (int i = tid; i < nblk; i += kSelThreads) sh.bkeys[i] = 0u;
  __syncthreads();
  const float* src = a.scores + (size_t)row * a.ld;
  const int t_begin = tid * PPT;
  uint32_t pk[PPT];   // this thread's position keys (0 = not a candidate value)
  if ((a.ld & 3) == 0) {   // rows start 16-byte aligned: float4 loads
#pragma unroll
    for (int j = 0; j < PPT; j += 4) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t_begin + j < vis) v = *reinterpret_cast<const float4*>(src + t_begin + j);
      const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) pk[j + u] = (t_begin + j + u < vis && isfinite(f[u])) ? order_key(f[u]) : 0u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < PPT; ++j) {
      const float f = t_begin + j < vis ? src[t_begin + j] : 0.f;
      pk[j] = (t_begin + j < vis && isfinite(f)) ? order_key(f) : 0u;
    }
  }
  if (t_begin < vis) {
    int blk = t_begin / a.cbs, bnd = (blk + 1) * a.cbs;   // positions advance by one: one boundary at a time
    uint32_t run = 0u;
#pragma unroll
    for (int j = 0; j < PPT; ++j) {
      if (t_begin + j >= bnd) {
        if (run) atomicMax(&sh.bkeys[blk], run);
        ++blk;
        bnd += a.cbs;
        run = 0u;
      }
      run = max(run, pk[j]);
    }
    if (run) atomicMax(&sh.bkeys[blk], run);
  }
  __syncthreads();
  uint32_t key[BPT];
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int bi = tid * BPT + j;
    key[j] = bi < nblk ? sh.bkeys[bi] : 0u;
  }
  __syncthreads();   // the block keys are in registers: the shared memory is reused below
  select_top<kSelThreads, BPT>(key, min(a.cbk, nblk), a.blocks + (size_t)row * a.cbk, a.cbk, 0, sh.sel);
}

// Level one of the two-level top-k without a filter of its own (the candidate source
// layer): the candidate blocks and the row's own top-k come from the same scores, so one
// CTA per row loads them into registers once, forms the block keys (cand_kernel's rule),
// keeps the cbk best blocks, then selects the k_eff best positions (topk_kernel's rule,
// including the short-context fill) with the same primitive.
union CandTopkShared {
  uint32_t bkeys[kCandMaxBlocks];
  SelectShared<kSelThreads> sel;   // reused once the block keys are in registers
};

template <int KPT, int BPT>
__global__ void __launch_bounds__(kSelThreads, 1) cand_topk_kernel(const CandArgs c, const TopkArgs a) {
  __shared__ CandTopkShared sh;
  const int tid = threadIdx.x;
  pdl_allow_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int2 ext = row_extent(a.rinfo, row, a.S, a.T, a.start_pos, a.ratio);
  const int vis = ext.x;
  const int k_eff = min(a.topk, ext.y);
  const int nblk = (a.T + c.cbs - 1) / c.cbs;
  for (int i = tid; i < nblk; i += kSelThreads) sh.bkeys[i] = 0u;
  __syncthreads();
  const int base = tid * KPT;
  const float* src = a.scores + (size_t)row * a.ld;
  uint32_t key[KPT];   // position keys: finite scores at t < vis, else 0
  if ((a.ld & 3) == 0) {   // rows start 16-byte aligned: float4 loads
#pragma unroll
    for (int j = 0; j < KPT; j += 4) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (base + j < vis) v = *reinterpret_cast<const float4*>(src + base + j);
      const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) key[j + u] = (base + j + u < vis && isfinite(f[u])) ? order_key(f[u]) : 0u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const float f = base + j < vis ? src[base + j] : 0.f;
      key[j] = (base + j < vis && isfinite(f)) ? order_key(f) : 0u;
    }
  }
  if (base < vis) {   // block maxima: positions advance by one, one block boundary at a time
    int blk = base / c.cbs, bnd = (blk + 1) * c.cbs;
    uint32_t run = 0u;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      if (base + j >= bnd) {
        if (run) atomicMax(&sh.bkeys[blk], run);
        ++blk;
        bnd += c.cbs;
        run = 0u;
      }
      run = max(run, key[j]);
    }
    if (run) atomicMax(&sh.bkeys[blk], run);
  }
  __syncthreads();
  uint32_t bk[BPT];
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int bi = tid * BPT + j;
    bk[j] = bi < nblk ? sh.bkeys[bi] : 0u;
  }
  __syncthreads();   // the block keys are in registers: the shared memory is reused below
  select_top<kSelThreads, BPT>(bk, min(c.cbk, nblk), c.blocks + (size_t)row * c.cbk, c.cbk, 0, sh.sel);
  __syncthreads();   // the selection's shared memory is reused for the top-k
  int32_t* out = a.out + (size_t)row * a.topk;
  if (vis <= k_eff) {   // short-context rule: every visible position, in order
    for (int i = tid; i < a.topk; i += kSelThreads) out[i] = i < vis ? i + a.offset : -1;
    return;
  }
  select_top<kSelThreads, KPT>(key, k_eff, out, a.topk, a.offset, sh.sel, vis);
}

// The candidate-block kernels and the sparse top-k launch in plain stream order, without the
// early start the other small grids take: the two-level decode step (8 rows over 32768 keys)
// measured 45.9 against 51.0 us with it.
template <int KPT>
cudaError_t launch_cand_topk_kpt(const CandArgs& c, const TopkArgs& a, int nblk, cudaStream_t stream) {
  const dim3 grid(a.rows), block(kSelThreads);
  if (nblk <= kSelThreads) return launch_kernel(false, cand_topk_kernel<KPT, 1>, grid, block, 0, stream, c, a);
  if (nblk <= 2 * kSelThreads) return launch_kernel(false, cand_topk_kernel<KPT, 2>, grid, block, 0, stream, c, a);
  if (nblk <= 4 * kSelThreads) return launch_kernel(false, cand_topk_kernel<KPT, 4>, grid, block, 0, stream, c, a);
  if (nblk <= 8 * kSelThreads) return launch_kernel(false, cand_topk_kernel<KPT, 8>, grid, block, 0, stream, c, a);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_cand_topk(const CandArgs& c, const TopkArgs& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  if (a.cand != nullptr || a.sparse || c.rows != a.rows || c.ld != a.ld) return cudaErrorInvalidValue;
  const int nblk = (a.T + c.cbs - 1) / c.cbs;
  if (a.T <= kSelThreads * 8) return launch_cand_topk_kpt<8>(c, a, nblk, stream);
  if (a.T <= kSelThreads * 16) return launch_cand_topk_kpt<16>(c, a, nblk, stream);
  if (a.T <= kSelThreads * 32) return launch_cand_topk_kpt<32>(c, a, nblk, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  const dim3 grid(a.rows);
  if (a.sparse) {   // kept positions only: at most cbk * cbs of them
    const long long E = (long long)a.cbk * a.cbs;
    if (a.cand == nullptr || E > (long long)kSelThreads * 8) return cudaErrorInvalidValue;
    if (E <= 256 * 8) return launch_kernel(false, topk_sparse_kernel<256, 8>, grid, dim3(256), 0, stream, a);
    if (E <= 512 * 8) return launch_kernel(false, topk_sparse_kernel<512, 8>, grid, dim3(512), 0, stream, a);
    return launch_kernel(false, topk_sparse_kernel<kSelThreads, 8>, grid, dim3(kSelThreads), 0, stream, a);
  }
  if (a.rows >= 4096 && a.T > 256 * 8 && a.T <= 256 * 32) {
    // many rows (prefill): 256 threads per row with up to 32 keys each, so several rows
    // share an SM; the latency of one row matters less than the rows per second
    if (a.T <= 256 * 16) return launch_overlapped(topk_kernel<256, 16>, grid, dim3(256), 0, stream, a);
    return launch_overlapped(topk_kernel<256, 32>, grid, dim3(256), 0, stream, a);
  }
  // eight keys per thread and no more threads than keys up to 8192 positions
  if (a.T <= 256 * 8) return launch_overlapped(topk_kernel<256, 8>, grid, dim3(256), 0, stream, a);
  if (a.T <= 512 * 8) return launch_overlapped(topk_kernel<512, 8>, grid, dim3(512), 0, stream, a);
  if (a.T <= kSelThreads * 8)
    return launch_overlapped(topk_kernel<kSelThreads, 8>, grid, dim3(kSelThreads), 0, stream, a);
  if (a.T <= kSelThreads * 16)
    return launch_overlapped(topk_kernel<kSelThreads, 16>, grid, dim3(kSelThreads), 0, stream, a);
  if (a.T <= kSelThreads * 32)
    return launch_overlapped(topk_kernel<kSelThreads, 32>, grid, dim3(kSelThreads), 0, stream, a);
  return cudaErrorInvalidValue;
}

template <int PPT>
cudaError_t launch_cand_ppt(const CandArgs& a, int nblk, cudaStream_t stream) {
  const dim3 grid(a.rows), block(kSelThreads);
  if (nblk <= kSelThreads) return launch_kernel(false, cand_kernel<PPT, 1>, grid, block, 0, stream, a);
  if (nblk <= 2 * kSelThreads) return launch_kernel(false, cand_kernel<PPT, 2>, grid, block, 0, stream, a);
  if (nblk <= 4 * kSelThreads) return launch_kernel(false, cand_kernel<PPT, 4>, grid, block, 0, stream, a);
  if (nblk <= 8 * kSelThreads) return launch_kernel(false, cand_kernel<PPT, 8>, grid, block, 0, stream, a);
  return cudaErrorInvalidValue;
}

cudaError_t launch_candidates(const CandArgs& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  const int nblk = (a.T + a.cbs - 1) / a.cbs;
  if (a.T <= kSelThreads * 8) return launch_cand_ppt<8>(a, nblk, stream);
  if (a.T <= kSelThreads * 16) return launch_cand_ppt<16>(a, nblk, stream);
  if (a.T <= kSelThreads * 32) return launch_cand_ppt<32>(a, nblk, stream);
  return cudaErrorInvalidValue;
}

}  // namespace indexer
