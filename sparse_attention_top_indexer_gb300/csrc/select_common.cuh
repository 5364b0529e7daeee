// CTA-wide top-k selection over order-preserving uint32 keys held in registers, shared by
// the top-k kernels (all positions, the kept candidate positions, the fused candidate
// blocks + top-k) and the candidate-block selection.
//
// Thread t holds the keys of positions [t*kpt, (t+1)*kpt) (kpt <= KPT, chosen per row);
// key 0 marks a position that cannot be selected. The k_eff largest keys are kept, ties to
// the lower position, and
// their positions (+offset) are written in ascending order, then -1 up to `width`.
// Up to three most-significant-digit radix passes (11 + 11 + 10 bits, 2048-bin
// shared-memory histograms) pin the k_eff-th largest key K*; a pass stops the search
// early once its bin holds exactly the keys still needed. With many rows per SM one warp
// searches each histogram (fewer instructions); with one row per SM all threads do (a
// shorter chain). One CTA-wide scan of packed (equal, greater) counts then gives every
// thread its output slot, and each thread writes its selected positions from a bit mask,
// so no sort is needed.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace indexer {

// Larger float -> larger key; every finite value maps to a key >= 0x00800000 > 0.
// -0.0 and +0.0 compare equal, so -0.0 is first folded onto +0.0 (x + 0 = +0 for x = -0).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(__fadd_rn(f, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kHistBins = 2048;

// Radix digits of the selection, most significant first: 11 + 11 + 10 bits. The first
// digit spreads typical score rows over ~100 bins; shared-memory atomics see little
// contention even when it does not (uniform scores in [1, 2), four bins: +8 % time).

template <int NT>
struct alignas(16) SelectShared {
  uint32_t hist[2][kHistBins];   // 16-byte aligned: the bin search reads four bins at a time
  uint32_t warp_tot[NT / 32];
  uint32_t bc[4];            // bin, count above the bin, count in the bin, count in all bins
};

// Sum over the CTA of v, and the sum over the threads before this one. Ends with the
// warp totals consumed (the caller may reuse sh.warp_tot after its next barrier).
template <int NT>
__device__ __forceinline__ uint32_t cta_scan(uint32_t v, uint32_t& total, SelectShared<NT>& sh) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) sh.warp_tot[warp] = incl;
  __syncthreads();
  const uint32_t wt = lane < NW ? sh.warp_tot[lane] : 0u;
  uint32_t before_w = lane < warp ? wt : 0u;
  uint32_t tot = wt;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    before_w += __shfl_xor_sync(0xffffffffu, before_w, off);
    tot += __shfl_xor_sync(0xffffffffu, tot, off);
  }
  total = tot;
  return before_w + incl - v;
}

// Warp 0 of the CTA: in histogram h (larger digit = larger keys) find the bin holding the
// need-th largest key (need >= 1) and set bc = {bin, keys in the bins above it, keys in it,
// keys in all bins}; with fewer than need keys in all, only bc[3]. Lane l sums the 64 bins
// below 2047 - 64 l as 16 four-bin chunks (16-byte loads), visiting them in an order rotated
// by l so that the eight lanes of each 128-byte phase read distinct banks; a scan of those
// sums from the top picks the lane holding the key, and the warp then scans that lane's 64
// bins two per lane. BATCH chunks are in flight at a time (four keep the register-capped
// builds from spilling more).
template <int BATCH>
__device__ __forceinline__ void warp_search(const uint32_t* h, uint32_t need, uint32_t* bc) {
  static_assert(BATCH % 4 == 0 && 16 % BATCH == 0, "whole batches of the four partial sums");
  const int lane = threadIdx.x & 31;
  const int top = kHistBins - 1 - 64 * lane;
  const uint4* hv = reinterpret_cast<const uint4*>(h + (top - 63));   // 16-byte aligned: top - 63 = 64 (31 - lane)
  uint32_t part[4] = {0u, 0u, 0u, 0u};   // four independent sums: a short add chain
#pragma unroll 1
  for (int m0 = 0; m0 < 16; m0 += BATCH) {
#pragma unroll
    for (int m = 0; m < BATCH; ++m) {
      const uint4 v = hv[(m0 + m + lane) & 15];
      part[m & 3] += (v.x + v.y) + (v.z + v.w);
    }
  }
  const uint32_t own = (part[0] + part[1]) + (part[2] + part[3]);
  uint32_t incl = own;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  const unsigned hit = __ballot_sync(0xffffffffu, incl - own < need && need <= incl);
  if (hit == 0u) {
    if (lane == 0) bc[3] = total;
    return;
  }
  const int L = __ffs(hit) - 1;
  const uint32_t above_l = __shfl_sync(0xffffffffu, incl - own, L);
  const int top_l = kHistBins - 1 - 64 * L;
  const uint32_t c0 = h[top_l - 2 * lane], c1 = h[top_l - 2 * lane - 1];
  uint32_t pair = c0 + c1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, pair, off);
    if (lane >= off) pair += y;
  }
  const uint32_t ab = above_l + pair - (c0 + c1);   // keys in the bins above this lane's two
  if (ab < need && need <= ab + c0 + c1) {          // exactly one lane
    const bool first = ab + c0 >= need;
    bc[0] = (uint32_t)(first ? top_l - 2 * lane : top_l - 2 * lane - 1);
    bc[1] = first ? ab : ab + c0;
    bc[2] = first ? c0 : c1;
    bc[3] = total;
  }
}

// The same search by all NT threads (BPT bins each): thread t owns bins hb, hb-1, ...,
// hb-BPT+1 with hb = 2047 - BPT*t, so a scan over threads in order counts the keys in the
// bins above a thread's bins. Shorter than warp_search when NT is large (one row per SM);
// ends without a barrier (bc is written by one thread).
template <int NT>
__device__ __forceinline__ void cta_search(const uint32_t* h, uint32_t need, SelectShared<NT>& sh) {
  constexpr int BPT = kHistBins / NT;
  static_assert(BPT >= 1 && kHistBins % NT == 0, "thread count must divide the bin count");
  const int hb = kHistBins - 1 - BPT * (int)threadIdx.x;
  uint32_t c[BPT], own = 0u;
#pragma unroll
  for (int q = 0; q < BPT; ++q) {
    c[q] = h[hb - q];
    own += c[q];
  }
  uint32_t total;
  const uint32_t above = cta_scan<NT>(own, total, sh);   // keys in bins above hb
  if (threadIdx.x == 0) sh.bc[3] = total;
  if (need <= total && above < need && need <= above + own) {
    uint32_t acc = above;
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
      if (acc + c[q] >= need) {
        sh.bc[0] = (uint32_t)(hb - q);
        sh.bc[1] = acc;
        sh.bc[2] = c[q];
        break;
      }
      acc += c[q];
    }
  }
}

// Calls fn(j) for the keys j < kpt of a thread, kpt a multiple of four (when KPT is): four at
// a time, with a jump past the chunks at or beyond kpt (kpt is the same in all threads of the
// CTA, so the jump is uniform and the skipped keys cost no issue slots).
template <int KPT, class Fn>
__device__ __forceinline__ void for_keys(int kpt, Fn&& fn) {
  if constexpr (KPT % 4 != 0) {
#pragma unroll
    for (int j = 0; j < KPT; ++j) fn(j);
  } else {
#pragma unroll
    for (int c = 0; c < KPT / 4; ++c) {
      if (4 * c >= kpt) break;
#pragma unroll
      for (int u = 0; u < 4; ++u) fn(4 * c + u);
    }
  }
}

// All NT threads must call it; it ends with every output written (256-thread CTAs with 16 or
// more keys a thread stage the indices in shared memory and write them after a barrier;
// otherwise each thread writes its own, with no trailing barrier). WARP_SEARCH: one warp searches the histograms (many rows per SM);
// otherwise all threads do (one row per SM, where the search's latency counts). Only
// threads with base < span may hold a nonzero key: the others skip the per-key loops.
//
// Instruction count is what bounds many rows per SM, so each step is lean: a valid key is
// >= 0x00800000, so the first digit of a valid key is >= 4 and the first pass needs no
// prefix test, and every later prefix is nonzero (a zero key never matches it); the
// compaction builds a bit mask of the thread's selected keys and visits only those.
// kpt: the keys a thread holds, positions [t*kpt, (t+1)*kpt) (a multiple of four, at most
// KPT, the same in all threads; KPT itself when KPT is not a multiple of four); the keys
// key[j] for j >= kpt are not read.
template <int NT, int KPT, bool WARP_SEARCH = (NT <= 256)>
__device__ void select_top(const uint32_t (&key)[KPT], int k_eff, int32_t* out, int width, int offset,
                           SelectShared<NT>& sh, int span = NT * KPT, int kpt = KPT) {
  static_assert(NT % 32 == 0 && NT >= 32, "whole warps");
  static_assert(KPT <= 32, "one bit per key in a 32-bit mask");
  const int tid = threadIdx.x;
  const int base = tid * kpt;
  const bool live = base < span;
  for (int i = tid; i < 2 * kHistBins / 4; i += NT) reinterpret_cast<uint4*>(&sh.hist[0][0])[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();

  auto search = [&](const uint32_t* h, uint32_t need) {
    if constexpr (WARP_SEARCH) {
      if (tid < 32) warp_search<4>(h, need, sh.bc);
    } else {
      cta_search<NT>(h, need, sh);
    }
    __syncthreads();
  };

  uint32_t need = (uint32_t)k_eff, kstar = 0u;
  // pass 0: the top 11 bits
  if (live) {
    for_keys<KPT>(kpt, [&](int j) {
      if (key[j] != 0u) atomicAdd(&sh.hist[0][key[j] >> 21], 1u);
    });
  }
  __syncthreads();
  search(sh.hist[0], need);
  if (sh.bc[3] <= need) {   // no more valid keys than k_eff: take them all
    need = 0u;
  } else {
    uint32_t prefix = sh.bc[0] << 21, mask = 0xFFE00000u;
    need -= sh.bc[1];
    bool settled = sh.bc[2] == need;   // the whole bin is taken: every key >= prefix
#pragma unroll 1
    for (int p = 1; p < 3 && !settled; ++p) {
      const int shift = p == 1 ? 10 : 0;
      const uint32_t dm = p == 1 ? 0x7FFu : 0x3FFu;
      uint32_t* h = sh.hist[p & 1];
      if (p == 2) {   // pass 0's histogram, read by its search before the last barrier
        for (int i = tid; i < kHistBins / 4; i += NT) reinterpret_cast<uint4*>(h)[i] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
      }
      if (live) {
        for_keys<KPT>(kpt, [&](int j) {
          if ((key[j] & mask) == prefix) atomicAdd(&h[(key[j] >> shift) & dm], 1u);
        });
      }
      __syncthreads();
      search(h, need);
      need -= sh.bc[1];
      prefix |= sh.bc[0] << shift;
      mask |= dm << shift;
      settled = sh.bc[2] == need;
    }
    if (settled) {
      kstar = prefix - 1u;   // prefix > 0 (see above)
      need = 0u;
    } else {
      kstar = prefix;        // all 32 bits fixed; `need` keys equal to it are still taken
    }
  }

  // ordered compaction: the keys above kstar, then the first `need` equal to it
  uint32_t gtm = 0u, eqm = 0u;
  if (live) {
    for_keys<KPT>(kpt, [&](int j) {
      gtm |= (key[j] > kstar ? 1u : 0u) << j;
      if (need != 0u) eqm |= (key[j] == kstar ? 1u : 0u) << j;
    });
  }
  const uint32_t packed = ((uint32_t)__popc(eqm) << 16) | (uint32_t)__popc(gtm);
  uint32_t total;
  const uint32_t before = cta_scan<NT>(packed, total, sh);   // (the passes read warp_tot before their last barrier)
  const uint32_t eq_before = before >> 16;
  // equal keys are taken in position order: this thread's first (need - eq_before) of them
  uint32_t take = need > eq_before ? need - eq_before : 0u;
  uint32_t sel = gtm;
  for (uint32_t m = eqm; m != 0u && take != 0u; m &= m - 1u, --take) sel |= m & (0u - m);
  uint32_t slot = (before & 0xFFFFu) + min(eq_before, need);
  const int sel_total = (int)((total & 0xFFFFu) + min(total >> 16, need));
  if constexpr (NT == 256 && KPT >= 16) {
    if (width <= 2 * kHistBins) {
      // many long rows per SM: stage the row's indices in the (now free) histogram memory and
      // write them out in order, a warp's stores covering consecutive addresses (each thread's
      // own run of slots would touch a sector per index): large prefill 0.802 -> 0.681 ms; the
      // 2048-key rows (8 keys a thread, 512 indices) were faster without (33.3 against 34.7 us)
      int32_t* stage = reinterpret_cast<int32_t*>(&sh.hist[0][0]);
      for (; sel != 0u; sel &= sel - 1u) stage[slot++] = base + (__ffs(sel) - 1) + offset;
      __syncthreads();
      for (int i = tid; i < width; i += NT) out[i] = i < sel_total ? stage[i] : -1;
      return;
    }
  }
  for (; sel != 0u; sel &= sel - 1u) out[slot++] = base + (__ffs(sel) - 1) + offset;
  for (int i = sel_total + tid; i < width; i += NT) out[i] = -1;
}

}  // namespace indexer
