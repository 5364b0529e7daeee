// CTA-wide top-k selection over order-preserving uint32 keys held in registers, shared by
// the stand-alone top-k kernel and the fused decode kernel.
//
// Thread t holds the keys of positions [t*KPT, (t+1)*KPT); key 0 marks a position that
// cannot be selected. The k_eff largest keys are kept, ties to the lower position, and
// their positions (+offset) are written in ascending order, then -1 up to `width`.
// Up to three most-significant-digit radix passes (11 + 11 + 10 bits, 2048-bin
// shared-memory histograms) pin the k_eff-th largest key K*; a pass stops the search
// early once its bin holds exactly the keys still needed. With many rows per SM one warp
// searches each histogram (fewer instructions); with one row per SM all threads do (a
// shorter chain). One CTA-wide scan of packed (equal, greater) counts then gives every
// thread its output slot, so no sort is needed.
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
// digit spreads typical score rows over ~100 bins, so plain shared-memory atomics see
// little contention.
__device__ __forceinline__ int digit_shift(int p) { return p == 0 ? 21 : (p == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t digit_mask(int p) { return p == 2 ? 0x3FFu : 0x7FFu; }

template <int NT>
struct SelectShared {
  uint32_t hist[2][kHistBins];
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
// below 2047 - 64 l, visiting them in an order rotated by l so that the lanes read 32
// different banks; a scan of those sums from the top picks the lane holding the key, and
// the warp then scans that lane's 64 bins two per lane.
__device__ __forceinline__ void warp_search(const uint32_t* h, uint32_t need, uint32_t* bc) {
  const int lane = threadIdx.x & 31;
  const int top = kHistBins - 1 - 64 * lane;
  uint32_t own = 0u;
#pragma unroll 16
  for (int i = 0; i < 64; ++i) own += h[top - ((i + lane) & 63)];
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

// All NT threads must call it; it ends with every output written by its thread (no
// trailing barrier). WARP_SEARCH: one warp searches the histograms (many rows per SM);
// otherwise all threads do (one row per SM, where the search's latency counts).
template <int NT, int KPT, bool WARP_SEARCH = (NT <= 256)>
__device__ void select_top(const uint32_t (&key)[KPT], int k_eff, int32_t* out, int width, int offset,
                           SelectShared<NT>& sh) {
  static_assert(NT % 32 == 0 && NT >= 32, "whole warps");
  const int tid = threadIdx.x;
  const int base = tid * KPT;
  for (int i = tid; i < 2 * kHistBins; i += NT) (&sh.hist[0][0])[i] = 0u;
  __syncthreads();

  uint32_t prefix = 0u, mask = 0u, need = (uint32_t)k_eff, kstar = 0u;
  bool select_all = false, settled = false;
#pragma unroll 1
  for (int p = 0; p < 3; ++p) {
    const int shift = digit_shift(p);
    const uint32_t dm = digit_mask(p);
    uint32_t* h = sh.hist[p & 1];
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const uint32_t k = key[j];
      if (k != 0u && (k & mask) == prefix) atomicAdd(&h[(k >> shift) & dm], 1u);
    }
    __syncthreads();
    if constexpr (WARP_SEARCH) {
      if (tid < 32) warp_search(h, need, sh.bc);
    } else {
      cta_search<NT>(h, need, sh);
    }
    __syncthreads();
    if (p == 0 && sh.bc[3] <= need) {   // no more valid keys than k_eff: take them all
      select_all = true;
      break;
    }
    const uint32_t bin = sh.bc[0];
    need -= sh.bc[1];
    prefix |= bin << shift;
    mask |= dm << shift;
    if (sh.bc[2] == need) {   // the whole bin is taken: every key >= prefix
      kstar = (prefix > 0u ? prefix : 1u) - 1u;
      need = 0u;
      settled = true;
      break;
    }
    // zero this histogram for the pass after next (its atomics follow the next barrier)
    for (int i = tid; i < kHistBins; i += NT) h[i] = 0u;
  }
  if (select_all) {
    kstar = 0u;
    need = 0u;
  } else if (!settled) {
    kstar = prefix;          // all 32 bits fixed; `need` keys equal to it are still taken
  }

  // ordered compaction: one scan of (equal << 16 | greater) per thread
  uint32_t gt = 0u, eq = 0u;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    gt += key[j] > kstar;
    eq += (need != 0u && key[j] == kstar);
  }
  const uint32_t packed = (eq << 16) | gt;
  uint32_t total;
  const uint32_t before = cta_scan<NT>(packed, total, sh);   // (the passes read warp_tot before their last barrier)
  const uint32_t eq_before = before >> 16;
  uint32_t slot = (before & 0xFFFFu) + min(eq_before, need);
  uint32_t eq_seen = eq_before;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t k = key[j];
    if (k > kstar) {
      out[slot++] = base + j + offset;
    } else if (need != 0u && k == kstar) {
      if (eq_seen < need) out[slot++] = base + j + offset;
      ++eq_seen;
    }
  }
  const int sel_total = (int)((total & 0xFFFFu) + min(total >> 16, need));
  for (int i = sel_total + tid; i < width; i += NT) out[i] = -1;
}

}  // namespace indexer
