// Index scoring on the 5th-generation tensor cores (tcgen05, kind::mxf4 block-scaled).
//
// score[b,s,t] = sum_h w'[b,s,h] * relu( qhat[b,s,h,:] . khat[b,t,:] )
// ("DeepSeek V4.1" index-keys page, Indexer.forward: einsum bshd,btd->bsht, relu,
// times weights, sum over heads), with t >= vis(s) = (start_pos + s + 1) / ratio
// masked to -inf and, for a level-two layer, -inf outside the candidate blocks.
//
// One CTA (256 threads) takes a group of QG query rows of one sequence and a run of
// 128-key tiles (two 64-key pages each) of the paged key cache. A page already holds its
// codes in the tensor cores' K-major core-matrix order, so the MMA reads the A operand
// straight from the stage buffer the tile was bulk-copied into (cp.async.bulk: one copy
// when the tile's two pages are adjacent in the pool, else one per page; a ring of NSTAGE
// stages):
//   * MMA warpgroup (warps 0-3): rewrites the group's quantised query rows into the same
//     core-matrix order once (the B operand, N = QG * H padded to 16) and stores their
//     scale factors in tensor memory; then, per page, each warp stores the A scale factors
//     of its 32 keys (tcgen05.st into its lane quadrant), the four warps meet at a named
//     barrier, and one thread issues two block-scaled MMAs (K = 64 each) into one of NACC
//     f32 accumulators, committed to an mbarrier;
//   * epilogue warpgroup (warps 4-7): thread m owns key t0 + m (TMEM lane m); it reads the
//     N head dot products with tcgen05.ld, releases the accumulator, and forms
//     sum_h w' * max(dot, 0) per query row in f32 -- no shuffles, because keys, not heads,
//     sit on the lanes. Once a page's MMA has completed, its stage is refilled from here.
// Every lane of a waiting warp polls the mbarrier (bounded) and the warp agrees on the
// outcome with __all_sync. Several query rows per group run in score_rows_kernel below.
//
// Tensor-memory scale layout: the MMA reads the scale factors of A row m from lane m,
// column m / 32 of the scale set, and those of B row n = 32 j + i from column j, lane i of
// any 32-lane quadrant. Each 32-bit column holds the two UE8M0 scales an MMA of K = 64
// needs in its low two bytes (scale-factor id 0), so a key's scale word is split into
// bytes 0/1 (first MMA) and bytes 2/3 (second MMA) in two 4-column halves of its set.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace indexer {

namespace {

constexpr int kTileKeys = 2 * kPageKeys;             // one MMA M-tile: two 64-key pages side by side
// Key formats: MXFP4 rows (68 bytes; block-scaled MMA, scales in tensor memory) and FP8
// rows (132 bytes; e4m3 MMA, the per-row scales multiply in the epilogue).
struct FmtMxfp4 {
  static constexpr bool kFp8 = false;
  static constexpr int kCode = kCodeBytes, kRow = kRowBytes, kPage = kPageBytes, kGroup = kGroupBytes;
  static constexpr int kStage = 9216;    // two pages (8704 B) padded to a 1 KB multiple
};
struct FmtFp8 {
  static constexpr bool kFp8 = true;
  static constexpr int kCode = kCodeBytesFp8, kRow = kRowBytesFp8, kPage = kPageBytesFp8, kGroup = kGroupBytesFp8;
  static constexpr int kStage = 17408;   // two pages (16896 B) padded to a 1 KB multiple
};
constexpr int kEpiThreads = 128;                     // one epilogue warpgroup
constexpr int kEpiWarps = 4;
// The lanes of a converged warp are done (their earlier shared-memory and tensor-memory
// accesses ordered by the warp synchronisation); one lane arrives for the warp.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
constexpr int kMaxPages = 32768 / kPageKeys;         // pages of the longest row a sparse launch takes
constexpr int kMaxTilesCta = 256;                    // tiles one CTA takes at most

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ constexpr uint32_t pow2_cols(int n) {
  return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : n <= 256 ? 256u : 512u;
}

// most accumulators (at most 4) whose columns, with their A scale sets and the B
// scales, fit in `budget` tensor-memory columns
__host__ __device__ constexpr int max_acc(int NP, int SB, int budget) {
  return 4 * (NP + 8) + 2 * SB <= budget ? 4 : 3 * (NP + 8) + 2 * SB <= budget ? 3
       : 2 * (NP + 8) + 2 * SB <= budget ? 2 : 1 * (NP + 8) + 2 * SB <= budget ? 1 : 0;
}

// FP8 accumulators: at most 4; N <= 64 keeps them within 256 columns (two CTAs per SM),
// larger N takes the 512 columns of one CTA per SM (its epilogue reads 128 columns at once)
constexpr int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }

__host__ __device__ constexpr int acc_f8(int NP) {
  return NP <= 64 ? (256 / NP < 4 ? 256 / NP : 4) : (512 / NP < 4 ? 512 / NP : 4);
}

// EPI epilogue warpgroups (warps 4 .. 4*EPI+3) take alternate pages.
template <int H, int QG, int EPI, class F>
struct ScoreCfg {
  static constexpr int THREADS = 128 * (1 + EPI);
  static constexpr int N = QG * H;
  static constexpr int NP = round_up(N, 16);                 // MMA N
  static constexpr int NCB = (NP + 31) / 32;                 // B scale columns per half
  static constexpr int SB = round_up(NCB, 4);
  // tensor memory: NACC accumulators of NP columns, NACC A scale sets of 8 columns, two
  // halves of SB B scale columns; every scale address is a multiple of 4 columns. Two or
  // more accumulators within 256 columns let two CTAs share an SM.
  static constexpr int NSTAGE = F::kFp8 ? 5 : 8;
  static constexpr int NACC = F::kFp8 ? acc_f8(NP)
                                      : max_acc(NP, SB, 256) >= 2 ? max_acc(NP, SB, 256) : max_acc(NP, SB, 512);
  static constexpr int SFA_COL = NACC * NP;
  static constexpr int SFB_COL = SFA_COL + 8 * NACC;
  static constexpr int TMEM_NEED = F::kFp8 ? NACC * NP : SFB_COL + 2 * SB;
  static constexpr uint32_t TMEM_COLS = pow2_cols(TMEM_NEED);
  static constexpr int OFF_QB = 0;
  static constexpr int OFF_STG = round_up(NP * F::kCode, 1024);
  static constexpr int OFF_QSTG = OFF_STG + NSTAGE * F::kStage;             // raw query rows
  static constexpr int OFF_W = OFF_QSTG + round_up(N * F::kRow, 16);
  static constexpr int OFF_SFW = OFF_W + round_up(N * 4, 16);
  // barriers: full per stage; done per accumulator and epilogue warpgroup (the MMA of tile i
  // commits to the barrier of the warpgroup that reads it, so each done barrier's phases are
  // consumed in order by one warpgroup: with one per accumulator, a warpgroup taking every
  // other tile would skip phases and a parity wait could pass on a phase two rounds old);
  // empty per accumulator; the query rows
  static constexpr int LDONE = NACC / gcd_int(NACC, EPI) * EPI;   // tiles per round of (accumulator, warpgroup) pairs
  static constexpr int NBAR = NSTAGE + NACC * EPI + NACC + 1;
  static constexpr int OFF_BAR = round_up(OFF_SFW + NCB * 32 * 4, 8);
  static constexpr int OFF_INFO = OFF_BAR + NBAR * 8;                         // tmem base, counters
  static constexpr int OFF_PTAB = round_up(OFF_INFO + 16, 16);   // pool page of each half of this CTA's tiles
  static constexpr int OFF_PLIST = OFF_PTAB + 2 * kMaxTilesCta * 4;   // sparse: the row's pages (+ bitmap)
  static constexpr int OFF_CAND = OFF_PLIST + (QG == 1 ? kMaxPages * 4 + kMaxPages / 8 : 0);
  static_assert(N <= 256, "MMA N is at most 256");
  static_assert(NACC >= 1, "tensor memory budget");
  static_assert(NBAR <= 32, "barriers are initialised by the lanes of one warp");
  static_assert(SFA_COL % 4 == 0 && SFB_COL % 4 == 0 && SB % 4 == 0, "scale sets must be 4-column aligned");
  static_assert(TMEM_NEED <= (int)TMEM_COLS && TMEM_COLS <= 512u, "tensor memory budget");
};

// Pool page of logical page lp of sequence b: through the block table, or the sequence's
// own run of pages. -1: no page (lp < 0); -2: a block-table entry outside the pool.
__device__ __forceinline__ int pool_page(const ScoreArgs& a, int b, int lp) {
  if (lp < 0) return -1;
  if (a.block_table == nullptr) return b * a.pages_per_seq + lp;
  const int p = a.block_table[(size_t)b * a.bt_stride + lp];
  return (p >= 0 && p < a.num_pages) ? p : -2;
}

// Requests the two pages of a tile into a stage (a missing half is not copied; its keys
// are never stored); adjacent pool pages come in one copy.
template <class F>
__device__ __forceinline__ void issue_tile_load(const ScoreArgs& a, int p0, int p1, uint32_t stage_addr,
                                                uint32_t bar) {
  constexpr int PB = F::kPage;
  mbar_arrive_expect_tx(bar, (uint32_t)((p0 >= 0 ? PB : 0) + (p1 >= 0 ? PB : 0)));
  if (p0 >= 0 && p1 == p0 + 1) {
    bulk_g2s(stage_addr, a.k_pool + (size_t)p0 * PB, (uint32_t)(2 * PB), bar);
    return;
  }
  if (p0 >= 0) bulk_g2s(stage_addr, a.k_pool + (size_t)p0 * PB, (uint32_t)PB, bar);
  if (p1 >= 0) bulk_g2s(stage_addr + PB, a.k_pool + (size_t)p1 * PB, (uint32_t)PB, bar);
}

// The query rows of a group -> the MMA's B operand (core-matrix order: 8-row groups of
// 8 * code bytes, 16-byte core-matrix rows 128 bytes apart along K) and, for MXFP4, each
// row's scale word into sfw (rows past nrows are zero, their scales 2^0).
template <class F, int NCB32, int NP>
__device__ __forceinline__ void build_b_operand(const uint8_t* qstg, uint8_t* qB, uint32_t* sfw, int nrows,
                                                int tid) {
  for (int n = tid; n < NCB32; n += 128) {
    uint32_t w[F::kCode / 4];
    uint32_t sc = 0x7F7F7F7Fu;
    if (n < nrows) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(qstg + n * F::kRow);
#pragma unroll
      for (int i = 0; i < F::kCode / 4; ++i) w[i] = src[i];
      if (!F::kFp8) sc = src[F::kCode / 4];
    } else {
#pragma unroll
      for (int i = 0; i < F::kCode / 4; ++i) w[i] = 0u;
    }
    if (n < NP) {
#pragma unroll
      for (int c = 0; c < F::kCode / 16; ++c)
        *reinterpret_cast<uint4*>(qB + (n >> 3) * (8 * F::kCode) + c * 128 + (n & 7) * 16) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
    if (!F::kFp8) sfw[n] = sc;
  }
}

// {x0 + |x0|, x1 + |x1|} = 2 max(x, 0) of two values with one packed add (exact: x + x = 2x,
// x + |x| = +0 for x <= 0).
__device__ __forceinline__ float2 twice_relu2(float x0, float x1) {
  return __fadd2_rn(make_float2(x0, x1), make_float2(fabsf(x0), fabsf(x1)));
}

// One tile's MMAs: MXFP4 -- two block-scaled MMAs of K = 64; FP8 -- four e4m3 MMAs of K = 32.
template <class F, int NP>
__device__ __forceinline__ void issue_tile_mma(uint32_t acc, uint32_t pa, uint32_t qb, uint32_t sfa, uint32_t sfb,
                                               int SB) {
  if constexpr (F::kFp8) {
    const uint32_t idesc = idesc_f8(128, NP);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mma_f8(acc, smem_desc(pa + 256 * k, 128, F::kGroup), smem_desc(qb + 256 * k, 128, 8 * F::kCode), idesc,
             k > 0 ? 1u : 0u);
  } else {
    const uint32_t idesc = idesc_mxf4(128, NP);
    mma_mxf4(acc, smem_desc(pa, 128, F::kGroup), smem_desc(qb, 128, 8 * F::kCode), idesc, sfa, sfb, 0u);
    mma_mxf4(acc, smem_desc(pa + 256, 128, F::kGroup), smem_desc(qb + 256, 128, 8 * F::kCode), idesc, sfa + 4,
             sfb + SB, 1u);
  }
}

// The whole warp waits (bounded) for the phase, converged: every lane polls, and the warp
// agrees on the result (a single polling lane followed by a shuffle measured ~20 % slower in
// the score kernels). Warp-uniform result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  const bool ok = mbar_wait(bar, parity, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// The whole warp waits (bounded) for two phases (the second only when `need2`): both polls
// are issued before the warp branches on them, so a wait whose phases have completed costs one
// poll's latency, not two. Warp-uniform result.
__device__ __forceinline__ bool warp_wait2(uint32_t bar1, uint32_t par1, uint32_t bar2, uint32_t par2, bool need2,
                                           uint64_t limit_ns) {
  bool ok1 = mbar_try_wait(bar1, par1);
  bool ok2 = !need2 || mbar_try_wait(bar2, par2);
  if (!(ok1 && ok2)) {
    const uint64_t t0 = global_ns();
    while (!(ok1 && ok2)) {
      if (!ok1) ok1 = mbar_try_wait(bar1, par1);
      if (!ok2) ok2 = mbar_try_wait(bar2, par2);
      if (!(ok1 && ok2) && global_ns() - t0 > limit_ns) break;
    }
  }
  return __all_sync(0xffffffffu, ok1 && ok2);
}

template <int H, int QG, int EPI, class F>
__global__ void __launch_bounds__(ScoreCfg<H, QG, EPI, F>::THREADS,
                                  ScoreCfg<H, QG, EPI, F>::TMEM_COLS <= 256 && ScoreCfg<H, QG, EPI, F>::THREADS <= 256
                                      ? 2 : 1)
    score_kernel(const ScoreArgs a) {
  using C = ScoreCfg<H, QG, EPI, F>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1024-byte aligned base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_allow_next();
  // this CTA's query rows: nq consecutive rows (row0 ..) of sequence b, the first at
  // position pos0; the sequence has Tb keys
  int b, row0, nq, pos0, Tb;
  if (a.groups == nullptr) {
    b = blockIdx.z;
    const int s0 = blockIdx.y * QG;
    nq = min(QG, a.S - s0);
    row0 = b * a.S + s0;
    pos0 = a.start_pos + s0;
    Tb = a.T;
  } else {
    const int g = blockIdx.z * gridDim.y + blockIdx.y;
    if (g >= a.n_groups) return;
    pdl_wait();   // the groups were written by the kernels before
    const RowGroup rg = a.groups[g];
    b = rg.b;
    row0 = rg.row0;
    nq = min(rg.nq, QG);
    pos0 = rg.pos0;
    Tb = min(rg.T, a.T);
  }
  int* plist = reinterpret_cast<int*>(smem + C::OFF_PLIST);   // sparse: the row's pages, ascending
  int* ptab = reinterpret_cast<int*>(smem + C::OFF_PTAB);     // pool page of each half of this CTA's tiles
  uint32_t* info = reinterpret_cast<uint32_t*>(smem + C::OFF_INFO);   // [0] tmem, [1] tiles issued, [2] mma issued,
                                                                       // [3] sparse: pages of the row
  const bool sparse = QG == 1 && a.sparse_pages;
  int npages = (Tb + kPageKeys - 1) / kPageKeys;   // logical pages to score, two per tile
  if (sparse) {
    // level two with one query row: only the pages holding a kept candidate block are
    // scored. Warp 0 marks them in a bitmap and lists them in ascending order.
    pdl_wait();
    if (warp == 0) {
      uint32_t* bits = reinterpret_cast<uint32_t*>(plist + kMaxPages);
      const int nw = (npages + 31) / 32;
      for (int i = lane; i < nw; i += 32) bits[i] = 0u;
      __syncwarp();
      const int32_t* cand = a.cand + (size_t)row0 * a.cbk;
      for (int e = lane; e < a.cbk; e += 32) {
        const int blk = cand[e];
        if (blk < 0 || (long long)blk * a.cbs >= Tb) continue;
        const int p0 = (int)(((long long)blk * a.cbs) / kPageKeys);
        const int p1 = (int)(min((long long)(blk + 1) * a.cbs, (long long)Tb) - 1) / kPageKeys;
        for (int pg = p0; pg <= p1; ++pg) atomicOr(&bits[pg >> 5], 1u << (pg & 31));
      }
      __syncwarp();
      int total = 0;
      for (int w0 = 0; w0 < nw; w0 += 32) {
        const uint32_t word = w0 + lane < nw ? bits[w0 + lane] : 0u;
        const int cnt = __popc(word);
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += y;
        }
        int slot = total + incl - cnt;
        for (uint32_t w = word; w; w &= w - 1) plist[slot++] = (w0 + lane) * 32 + (__ffs(w) - 1);
        total += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) info[3] = (uint32_t)total;
    }
    __syncthreads();
    npages = (int)info[3];
  }
  const int ntiles = (npages + 1) / 2;
  const int tile0 = blockIdx.x * a.tiles_per_cta;
  const int tile1 = min(tile0 + a.tiles_per_cta, ntiles);
  if (nq <= 0 || tile0 >= tile1) return;
  // logical page of half h of tile i (-1: none)
  auto lpage = [&](int i, int h) {
    const int k = 2 * i + h;
    return k < npages ? (sparse ? plist[k] : k) : -1;
  };
  // keys the group's last row can see; tiles at or past it are fully masked (a sparse
  // launch has one row, which sees every key)
  const int vis_hi = min(Tb, (pos0 + nq) / a.ratio);
  const int tile_vis = sparse ? tile1 : min(tile1, (vis_hi + kTileKeys - 1) / kTileKeys);
  if (!sparse && a.groups == nullptr && a.block_table == nullptr && warp == 0) {
    // the CTA's pages are known before the kernels before finish: warm L2 with them
    // while they run (a hint; the copies below read after pdl_wait)
    for (int i = tile0 + lane; i < tile_vis; i += 32) {
      const int lp = 2 * i, n = min(2, npages - lp);
      prefetch_l2_bulk(a.k_pool + ((size_t)b * a.pages_per_seq + lp) * F::kPage, (uint32_t)(n * F::kPage));
    }
  }
  pdl_wait();   // the query rows, weights and pages of the kernels before are complete
  // -inf over the tiles no row of the group can see (by the epilogue warps while they wait
  // for the first accumulator, or here when the CTA has nothing to score)
  auto fill_masked = [&](int first_thread, int nthreads) {
    if (sparse) return;
    const int t_begin = max(tile0, tile_vis) * kTileKeys, t_end = min(tile1 * kTileKeys, Tb);
    for (int qi = 0; qi < nq; ++qi) {
      float* dst = a.scores + (size_t)(row0 + qi) * a.ld;
      for (int t = t_begin + first_thread; t < t_end; t += nthreads) dst[t] = -__int_as_float(0x7f800000);
    }
  };
  if (tile_vis <= tile0) {
    if (a.fill_masked) fill_masked(tid, C::THREADS);
    return;
  }
  const int nt = tile_vis - tile0;   // tiles this CTA scores

  uint8_t* qB = smem + C::OFF_QB;
  const uint8_t* stg = smem + C::OFF_STG;
  const uint8_t* qstg = smem + C::OFF_QSTG;
  float* wq = reinterpret_cast<float*>(smem + C::OFF_W);
  uint32_t* sfw = reinterpret_cast<uint32_t*>(smem + C::OFF_SFW);
  uint32_t* cand_bits = reinterpret_cast<uint32_t*>(smem + C::OFF_CAND);
  const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
  auto bar_full = [&](int st) { return bar0 + 8u * (uint32_t)st; };
  // tile i's accumulator i % NACC, read by epilogue warpgroup i % EPI
  auto bar_done = [&](int i) { return bar0 + 8u * (uint32_t)(C::NSTAGE + (i % C::NACC) * EPI + i % EPI); };
  auto bar_empty = [&](int c) { return bar0 + 8u * (uint32_t)(C::NSTAGE + C::NACC * EPI + c); };
  const uint32_t bar_q = bar0 + 8u * (uint32_t)(C::NBAR - 1);
  const uint32_t stg0 = smem_u32(stg);
  // pool pages of tile i's halves into ptab (an entry outside the pool is reported and its
  // keys score -inf)
  auto fill_ptab = [&](int i) {
    int p[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      p[h] = pool_page(a, b, lpage(tile0 + i, h));
      if (p[h] == -2) atomicOr(a.status, kStatusBadMeta);
      ptab[2 * i + h] = p[h];
    }
    return make_int2(p[0], p[1]);
  };

  // Setup: warp 0 initialises the barriers and requests the group's query rows and head
  // weights, then the first NSTAGE tiles (one lane per tile); warp 1 allocates tensor
  // memory meanwhile; warps 2-3 look up the pool pages of the remaining tiles.
  const size_t qrow0 = (size_t)row0 * H;   // first query-head row of the group
  const int first = min(nt, C::NSTAGE);
  if (warp == 0) {
    if (lane < C::NBAR) {
      const bool empty_bar = lane >= C::NSTAGE + C::NACC * EPI && lane < C::NSTAGE + C::NACC * EPI + C::NACC;
      mbar_init(bar0 + 8u * (uint32_t)lane, empty_bar ? (uint32_t)kEpiThreads : 1u);
      fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0) {
      const uint32_t qbytes = (uint32_t)(nq * H * F::kRow), wbytes = (uint32_t)(nq * H * 4);
      mbar_arrive_expect_tx(bar_q, qbytes + wbytes);
      bulk_g2s(smem_u32(qstg), a.q_rows + qrow0 * F::kRow, qbytes, bar_q);
      bulk_g2s(smem_u32(wq), a.w_prime + qrow0, wbytes, bar_q);
      info[1] = (uint32_t)first;
      info[2] = 0u;
    }
    __syncwarp();
    if (lane < first) {
      const int2 p = fill_ptab(lane);
      issue_tile_load<F>(a, max(p.x, -1), max(p.y, -1), stg0 + lane * F::kStage, bar_full(lane));
    }
    __syncwarp();
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&info[0]), C::TMEM_COLS);
    tmem_relinquish();
  } else if (warp < 4) {
    for (int i = first + tid - 64; i < nt; i += 64) fill_ptab(i);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = info[0];
  const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);   // this warp's lane quadrant

  bool failed = false;
  if (warp < 4) {
    // ------------------------------------------------------------ MMA warpgroup
    // query rows -> B operand (core-matrix order) and B scales
    failed = !named_bar_and(1, 128, warp_wait(bar_q, 0u));
    if (!failed) {
      build_b_operand<F, C::NCB * 32, C::NP>(qstg, qB, sfw, nq * H, tid);
      fence_proxy_async_smem();   // the B operand was written by ordinary stores
      named_bar_sync(1, 128);
      if constexpr (!F::kFp8) {
#pragma unroll
        for (int j = 0; j < C::NCB; ++j) {
          const uint32_t wd = sfw[32 * j + lane];
          tmem_st_x1(tq + C::SFB_COL + j, wd & 0xFFFFu);
          tmem_st_x1(tq + C::SFB_COL + C::SB + j, wd >> 16);
        }
      }
    }
    const uint32_t qb = smem_u32(qB);
    const int key = (warp << 5) | lane;   // this thread's key (TMEM lane) within a page
    for (int i = 0; i < nt && !failed; ++i) {
      const int st = i % C::NSTAGE, c = i % C::NACC;
      // the page has landed, and accumulator c (with its scale set) has been drained
      bool ok = warp_wait(bar_full(st), (uint32_t)(i / C::NSTAGE) & 1u);
      if (ok && i >= C::NACC) ok = warp_wait(bar_empty(c), (uint32_t)((i - C::NACC) / C::NACC) & 1u);
      if (ok) {
        tc_fence_after();
        if constexpr (!F::kFp8) {   // the tile's A scales
          const uint32_t w = *reinterpret_cast<const uint32_t*>(stg + st * F::kStage + page_scale_offset(key));
          const uint32_t lo = w & 0xFFFFu, hi = w >> 16;
          tmem_st_x8(tq + (uint32_t)(C::SFA_COL + 8 * c), lo, lo, lo, lo, hi, hi, hi, hi);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      // one barrier: the four warps' scales are stored, and they agree that every wait ended
      if (!named_bar_and(1, 128, ok)) {
        failed = true;
        break;
      }
      if (tid == 0) {
        tc_fence_after();
        const uint32_t pa = stg0 + (uint32_t)(st * F::kStage);
        const uint32_t acc = tmem + (uint32_t)(c * C::NP);
        const uint32_t sfa = tmem + (uint32_t)(C::SFA_COL + 8 * c);
        issue_tile_mma<F, C::NP>(acc, pa, qb, sfa, tmem + C::SFB_COL, C::SB);
        tc_commit(bar_done(i));
        info[2] = (uint32_t)(i + 1);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue warpgroup
    constexpr int P = H >= 32 ? 4 : 2;   // independent partial sums per row (pairs of heads)
    static_assert(C::N % 4 == 0 && H % 4 == 0 && C::NCB <= 4, "epilogue column grouping");
    const int grp = (warp - 4) >> 2;              // this warp's epilogue warpgroup
    const int et = (tid - 128) & (kEpiThreads - 1);   // key within the page == TMEM lane
    const int ge = tid - 128;                     // index among all epilogue threads
    // level-two candidate filter: one bit per block of cbs positions, per query row
    const int cand_words = a.cand ? ((a.T + a.cbs - 1) / a.cbs + 31) / 32 : 0;
    if (a.cand) {
      for (int i = ge; i < QG * cand_words; i += EPI * kEpiThreads) cand_bits[i] = 0u;
      named_bar_sync(2, EPI * kEpiThreads);
      for (int i = ge; i < nq * a.cbk; i += EPI * kEpiThreads) {
        const int qi = i / a.cbk;
        const int blk = a.cand[(size_t)(row0 + qi) * a.cbk + (i % a.cbk)];
        if (blk >= 0 && blk < cand_words * 32) atomicOr(&cand_bits[qi * cand_words + (blk >> 5)], 1u << (blk & 31));
      }
    }
    // head weights (rows past S weigh nothing)
    failed = !warp_wait(bar_q, 0u);
    if (!failed) {
      for (int n = nq * H + ge; n < C::N; n += EPI * kEpiThreads) wq[n] = 0.f;
      if constexpr (F::kFp8)   // fold each query row's scale into its head weight
        for (int n = ge; n < nq * H; n += EPI * kEpiThreads)
          wq[n] *= *reinterpret_cast<const float*>(qstg + n * F::kRow + F::kCode);
    }
    named_bar_sync(2, EPI * kEpiThreads);
    if (a.fill_masked) fill_masked(ge, EPI * kEpiThreads);
    for (int i = grp; i < nt && !failed; i += EPI) {   // this group's pages
      const int c = i % C::NACC;
      bool ok = warp_wait(bar_done(i), (uint32_t)(i / C::LDONE) & 1u);
      float sk = 1.f;   // FP8: this key's scale, read before the stage is refilled
      if constexpr (F::kFp8) {
        if (ok) sk = *reinterpret_cast<const float*>(stg + (i % C::NSTAGE) * F::kStage + page_scale_offset_fp8(et));
        ok = named_bar_and(3 + grp, kEpiThreads, ok);   // the warpgroup agrees (and has read its scales)
      }
      if (!ok) {
        failed = true;
        break;
      }
      tc_fence_after();
      // the whole accumulator in one tensor-memory read, then release it
      float v[C::NCB * 32];
      if constexpr (C::NCB == 1) tmem_ld32(tq + (uint32_t)(c * C::NP), v);
      else if constexpr (C::NCB == 2) tmem_ld64(tq + (uint32_t)(c * C::NP), v);
      else tmem_ld128(tq + (uint32_t)(c * C::NP), v);
      tc_fence_before();
      mbar_arrive(bar_empty(c));   // accumulator c and its scale set may be reused
      // sum_h w' * max(dot, 0) per query row: column pairs (two heads of one row) with packed
      // f32x2 FMAs into P independent partial sums per row
      float part[QG][P];
#pragma unroll
      for (int qi = 0; qi < QG; ++qi)
#pragma unroll
        for (int p = 0; p < P; ++p) part[qi][p] = 0.f;
#pragma unroll
      for (int n = 0; n < C::N; n += 4) {
        const float4 w4 = *reinterpret_cast<const float4*>(wq + n);
        const int qi = n / H, p0 = (n % P), p1 = ((n + 2) % P);
        const float2 r01 = twice_relu2(v[n], v[n + 1]);   // 2 max(dot, 0), halved at the row's sum
        const float2 r23 = twice_relu2(v[n + 2], v[n + 3]);
        ffma2(part[qi][p0], part[qi][p0 + 1], w4.x, w4.y, r01.x, r01.y);
        ffma2(part[(n + 2) / H][p1], part[(n + 2) / H][p1 + 1], w4.z, w4.w, r23.x, r23.y);
      }
      if (et == 0 && i + C::NSTAGE < nt) {
        // the MMA that read this page's stage has completed: refill it
        const int nx = i + C::NSTAGE;
        issue_tile_load<F>(a, max(ptab[2 * nx], -1), max(ptab[2 * nx + 1], -1), stg0 + (i % C::NSTAGE) * F::kStage,
                        bar_full(i % C::NSTAGE));
        atomicMax(&info[1], (uint32_t)(i + C::NSTAGE + 1));
      }
      // this thread's key: key et % 64 of the tile's half et / 64
      const int h = et >> 6;
      const int lp = lpage(tile0 + i, h);
      const int t = lp * kPageKeys + (et & (kPageKeys - 1));
      if (lp >= 0 && t < Tb) {
        const bool present = ptab[2 * i + h] >= 0;   // else a block-table entry outside the pool
#pragma unroll
        for (int qi = 0; qi < QG; ++qi) {
          if (qi < nq) {
            float acc = part[qi][0];
#pragma unroll
            for (int p = 1; p < P; ++p) acc += part[qi][p];
            acc *= 0.5f;   // the partial sums hold twice the head sum
            const int vis = min(Tb, (pos0 + qi + 1) / a.ratio);
            bool keep = present && t < vis;
            if (a.cand) {
              const int blk = t / a.cbs;
              keep = keep && ((cand_bits[qi * cand_words + (blk >> 5)] >> (blk & 31)) & 1u);
            }
            if constexpr (F::kFp8) acc *= sk;
            a.scores[(size_t)(row0 + qi) * a.ld + t] = keep ? acc : -__int_as_float(0x7f800000);
          }
        }
      }
      __syncwarp();
    }
  }
  __syncwarp();
  if (failed && (tid == 0 || tid == 128)) atomicOr(a.status, tid == 0 ? kStatusLoadTimeout : kStatusMmaTimeout);
  // On success every copy and MMA has been waited for by its consumer; after a failure,
  // bounded waits for whatever may still be in flight before shared and tensor memory go.
  const bool any_failed = __syncthreads_or(failed);
  if (any_failed) {
    if (tid == 0) {
      const int issued = (int)info[1], mmas = (int)info[2];
      mbar_wait(bar_q, 0u);
      for (int st = 0; st < C::NSTAGE && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / C::NSTAGE) * C::NSTAGE;   // last page loaded into st
        mbar_wait(bar_full(st), (uint32_t)(last / C::NSTAGE) & 1u);
      }
      if (mmas > 0) mbar_wait(bar_done(mmas - 1), (uint32_t)((mmas - 1) / C::LDONE) & 1u);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ============================================================================ several rows
// Query groups of several rows (prefill, chunked prefill, mixed batches): a persistent CTA
// per SM runs one pipeline over many groups, so the set-up (barriers, tensor memory, the
// first pages' latency) is paid once per SM instead of once per group. Groups are fetched
// from a counter in the workspace (a uniform batch hands out the groups with the most
// visible keys first), which balances the causal triangle across SMs.
// Tiles are numbered across all of a CTA's groups; a role that takes every k-th tile keeps
// its ring positions (stage, accumulator, scale set and their phases) as counters. The SM's
// issue slots are the limit, so every role does as little per tile as it can:
//   * producer warp (the last warp): fetches the next group, writes its descriptor and
//     requests its query rows and w' into one of two query buffers (once the other roles
//     have released the buffer's previous group), then streams the group's tiles through a
//     ring of NSTAGE stages, PBATCH tiles at a time: the lane that looked up a tile's pages
//     polls that stage's barrier (the MMA that last read it has completed) and issues its copy;
//   * scale warpgroup (warps 0-3): per group, rewrites the query rows into the B operand
//     (core-matrix order, one of two buffers) and stores their scales in tensor memory (one
//     of two sets); per tile, once the tile has landed, the four warps store the tile's A
//     scales into the scale set of its stage (each warp its own lane quadrant; the MMA that last
//     read the set completed before the stage was refilled) and signal the set's "ready"
//     mbarrier, two tiles per poll, so the scale warps run ahead of the accumulators;
//   * NMMA MMA warps, warp m taking tiles m, m + NMMA, ...: once the tile's scale set is
//     ready and its accumulator (j % NACC) has been drained, one thread issues the two
//     block-scaled MMAs and commits to the stage's mbarrier, which frees the stage for the
//     producer and the scale set for the scale warps and hands the accumulator to the epilogue
//     (NSTAGE > NACC). The two waits are polled together: a wait on a completed mbarrier still
//     costs the poll's latency (~150 cycles when the warp branches on it);
//   * EPI epilogue warpgroups, warpgroup g taking tiles g, g + EPI, ...: read the accumulator
//     in 32-column pieces, release it, form sum_h w' * max(dot, 0) per row and store; after
//     its last tile of a group every epilogue warp releases the query buffer of that group.
// Position of a tile in a ring of M slots: the slot (tile number mod M) and the parity of the
// ring's round (tile number / M), advanced by a stride of at most M without dividing.
template <int M>
struct RingPos {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ explicit RingPos(uint32_t t) : slot((int)(t % M)), phase((t / M) & 1u) {}
  template <int K>
  __device__ __forceinline__ void advance() {
    static_assert(K >= 1 && K <= M, "one wrap at most");
    slot += K;
    if (slot >= M) {
      slot -= M;
      phase ^= 1u;
    }
  }
};

template <int H, int QG, int EPI, int NMMA, class F>
struct RowsCfg {
  static constexpr int THREADS = 128 * (1 + EPI) + 32 * NMMA + 32;
  static constexpr int MMA_WARP = 4 * (1 + EPI);              // the first of NMMA MMA warps
  static constexpr int PRODUCER_WARP = MMA_WARP + NMMA;
  static constexpr int QFREE_COUNT = 4 * (1 + EPI) + NMMA;    // warps: scale warpgroup, epilogue, MMA
  static constexpr int N = QG * H;
  static constexpr int NP = round_up(N, 16);
  static constexpr int NCB = (NP + 31) / 32;
  static constexpr int SB = round_up(NCB, 4);
  static constexpr int NSTAGE = F::kFp8 ? 8 : 12;
  static constexpr int PBATCH = 4;   // tiles the producer requests per poll of the stage barriers
  // NSC key-scale sets (8 columns each), one per stage: tile j's A scales go into set
  // j % NSTAGE, last read by the MMA of tile j - NSTAGE, which had completed before the
  // producer refilled the stage with tile j; so once tile j has landed its set is free, and
  // the scale warps wait on the tile's barrier alone
  static constexpr int NSC = NSTAGE;
  // NACC accumulators (MXFP4: then the NSC A scale sets and two B scale sets, one per query
  // buffer; FP8: no scale sets)
  static constexpr int NACC = F::kFp8 ? (512 / NP < 4 ? 512 / NP : 4)
                            : 3 * NP + 8 * NSC + 4 * SB <= 512 ? 3 : 2 * NP + 8 * NSC + 4 * SB <= 512 ? 2 : 1;
  static constexpr int SFA_COL = NACC * NP;
  static constexpr int SFB_COL = SFA_COL + 8 * NSC;   // set q: columns SFB_COL + 2*SB*q ..
  static constexpr int TMEM_NEED = F::kFp8 ? NACC * NP : SFB_COL + 4 * SB;
  static constexpr uint32_t TMEM_COLS = pow2_cols(TMEM_NEED);
  static constexpr int QB_STRIDE = round_up(NP * F::kCode, 1024);
  static constexpr int QSTG_STRIDE = round_up(N * F::kRow, 16);
  static constexpr int W_STRIDE = round_up(N * 4, 16);
  static constexpr int OFF_QB = 0;
  static constexpr int OFF_STG = 2 * QB_STRIDE;
  static constexpr int OFF_QSTG = OFF_STG + NSTAGE * F::kStage;
  static constexpr int OFF_W = OFF_QSTG + 2 * QSTG_STRIDE;
  static constexpr int OFF_WS = OFF_W + 2 * W_STRIDE;                    // FP8: w' times the row's scale
  static constexpr int OFF_SFW = OFF_WS + (F::kFp8 ? 2 * W_STRIDE : 0);
  static constexpr int OFF_GD = round_up(OFF_SFW + NCB * 32 * 4, 16);   // two group descriptors
  // barriers: full and free per stage, empty per accumulator and MMA warp, qfull and qfree per
  // query buffer, ready per scale set; FP8: scales read (per stage), scaled w' ready.
  // Accumulator c's release after tile j goes to the barrier of the MMA warp that issues tile
  // j + NACC, so each empty barrier's phases are consumed in order by one MMA warp: with one
  // barrier per accumulator, an MMA warp that takes every other tile skips every other phase
  // and a parity wait could pass on a phase two rounds old (the epilogue then still reading
  // the accumulator), which large groups of slow epilogues (16 query rows a tile) hit
  static constexpr int NEMPTY = NACC * NMMA;
  static constexpr int B_FULL = 0, B_FREE = NSTAGE, B_EMPTY = 2 * NSTAGE, B_QFULL = B_EMPTY + NEMPTY;
  static constexpr int B_QFREE = B_QFULL + 2, B_READY = B_QFREE + 2, B_SREAD = B_READY + NSC;
  static constexpr int B_WS = B_SREAD + (F::kFp8 ? NSTAGE : 0);
  static constexpr int NBAR = B_WS + (F::kFp8 ? 2 : 0);
  static constexpr int OFF_BAR = OFF_GD + 2 * 32;
  static constexpr int OFF_INFO = OFF_BAR + NBAR * 8;   // tmem, tiles issued, q phases, each MMA warp's tiles
  static constexpr int SMEM = OFF_INFO + 4 * (3 + NMMA);
  static_assert(N <= 256, "MMA N is at most 256");
  static_assert(NMMA >= 1 && 3 + NMMA <= 8, "MMA warps");
  static_assert(TMEM_NEED <= (int)TMEM_COLS && TMEM_COLS <= 512u, "tensor memory budget");
  static_assert(SFA_COL % 4 == 0 && SFB_COL % 4 == 0 && SB % 4 == 0, "scale sets must be 4-column aligned");
  static_assert(NBAR <= 64, "barriers are initialised by the lanes of two passes of one warp");
  static_assert(QFREE_COUNT < (1 << 20), "mbarrier arrival count");
  static_assert(NSTAGE > NACC, "the epilogue waits on a stage's barrier for its accumulator");
  static_assert(NSC == NSTAGE, "a tile's scale set is freed by the refill of its stage");
  static_assert(PBATCH <= 32 && PBATCH < NSTAGE, "a batch of stages, one lane each");
  static_assert(OFF_GD + 64 + NBAR * 8 + 16 + 1024 <= 227 * 1024, "shared memory budget");
};

struct GroupDesc {   // one query group, as the producer hands it to the other roles
  int b, row0, nq, pos0;
  int Tb, nt, ntiles, live;   // keys of the sequence, tiles to score, tiles of the sequence, 0 = no more groups
};

template <int H, int QG, int EPI, int NMMA, class F>
__global__ void __launch_bounds__(RowsCfg<H, QG, EPI, NMMA, F>::THREADS, 1) score_rows_kernel(const ScoreArgs a) {
  using C = RowsCfg<H, QG, EPI, NMMA, F>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_allow_next();
  GroupDesc* gdesc = reinterpret_cast<GroupDesc*>(smem + C::OFF_GD);
  // [0] tmem, [1] tiles issued, [2] q phases, [3 + m] tiles MMA warp m has issued (last + 1)
  uint32_t* info = reinterpret_cast<uint32_t*>(smem + C::OFF_INFO);
  const uint8_t* stg = smem + C::OFF_STG;
  const uint32_t stg0 = smem_u32(stg);
  uint32_t* sfw = reinterpret_cast<uint32_t*>(smem + C::OFF_SFW);
  const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
  auto bar_full = [&](int st) { return bar0 + 8u * (uint32_t)(C::B_FULL + st); };
  auto bar_free = [&](int st) { return bar0 + 8u * (uint32_t)(C::B_FREE + st); };
  auto bar_empty = [&](int c, int m) { return bar0 + 8u * (uint32_t)(C::B_EMPTY + c * NMMA + m); };
  auto bar_qfull = [&](int q) { return bar0 + 8u * (uint32_t)(C::B_QFULL + q); };
  auto bar_qfree = [&](int q) { return bar0 + 8u * (uint32_t)(C::B_QFREE + q); };
  auto bar_ready = [&](int sc) { return bar0 + 8u * (uint32_t)(C::B_READY + sc); };
  auto bar_sread = [&](int st) { return bar0 + 8u * (uint32_t)(C::B_SREAD + st); };
  auto bar_wsready = [&](int q) { return bar0 + 8u * (uint32_t)(C::B_WS + q); };
  if (warp == 0) {
    for (int i = lane; i < C::NBAR; i += 32) {
      const bool empty_bar = i >= C::B_EMPTY && i < C::B_EMPTY + C::NEMPTY;
      const bool qfree_bar = i >= C::B_QFREE && i < C::B_QFREE + 2;
      const bool ready_bar = i >= C::B_READY && i < C::B_READY + C::NSC;
      const bool sread_bar = F::kFp8 && i >= C::B_SREAD && i < C::B_SREAD + C::NSTAGE;
      const bool ws_bar = F::kFp8 && i >= C::B_WS;
      // a query buffer is released by the scale warpgroup and the MMA warp (once they have
      // read it) and by every epilogue thread (once the group's last accumulator has been
      // read); an accumulator's scales are ready once the four scale warps have stored them;
      // FP8: a stage's key scales have been read by the epilogue warpgroup of its tile, and
      // a query buffer's scaled head weights have been written by all epilogue threads
      mbar_init(bar0 + 8u * (uint32_t)i, empty_bar || ready_bar || sread_bar ? (uint32_t)kEpiWarps
                                         : qfree_bar ? (uint32_t)C::QFREE_COUNT
                                         : ws_bar ? (uint32_t)(EPI * kEpiWarps) : 1u);
    }
    fence_mbar_init();
    if (lane >= 1 && lane < 3 + NMMA) info[lane] = 0u;   // info[0] is the allocation's, written by warp 1
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&info[0]), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = info[0];
  bool failed = false;
  const uint64_t wait_ns = a.wait_ns ? a.wait_ns : kWaitLimitNs;
  // every role waits for the kernels before (query rows, w', pages, the group list; the
  // scores they read) before its first bounded wait, so that no wait's clock starts while
  // the dependency is still running (a kernel before that runs longer than the limit would
  // otherwise make these waits run out)
  pdl_wait();

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ producer warp
    // (a test of the bounded waits holds this role back: no group, copy or MMA is ever
    // issued and every other role's first wait runs out)
    if (!a.hold_producer) {
    const int gps = (a.S + QG - 1) / QG;                       // uniform batch: groups per sequence
    const long long total = a.groups ? (long long)a.n_groups : (long long)gps * a.B;
    uint32_t j = 0;                                            // tiles issued
    for (int k = 0;; ++k) {
      const int qb = k & 1;
      if (k >= 2 && !warp_wait(bar_qfree(qb), (uint32_t)((k - 2) >> 1) & 1u, wait_ns)) {
        failed = true;
        break;
      }
      // next group with rows (the lanes agree through lane 0's fetch)
      GroupDesc d{};
      for (;;) {
        uint32_t f = 0u;
        if (lane == 0) f = atomicAdd(a.sched, 1u);
        f = __shfl_sync(0xffffffffu, f, 0);
        if ((long long)f >= total) break;
        if (a.groups == nullptr) {
          const int si = gps - 1 - (int)(f / (uint32_t)a.B);   // most visible keys first
          d.b = (int)(f % (uint32_t)a.B);
          const int s0 = si * QG;
          d.nq = min(QG, a.S - s0);
          d.row0 = d.b * a.S + s0;
          d.pos0 = a.start_pos + s0;
          d.Tb = a.T;
        } else {
          const RowGroup rg = a.groups[f];
          d.b = rg.b;
          d.row0 = rg.row0;
          d.nq = min(rg.nq, QG);
          d.pos0 = rg.pos0;
          d.Tb = min(rg.T, a.T);
        }
        if (d.nq > 0) {
          d.live = 1;
          break;
        }
      }
      if (d.live) {
        d.ntiles = (d.Tb + kTileKeys - 1) / kTileKeys;
        const int vis_hi = min(d.Tb, (d.pos0 + d.nq) / a.ratio);
        d.nt = min(d.ntiles, (vis_hi + kTileKeys - 1) / kTileKeys);
      }
      if (lane == 0) {
        gdesc[qb] = d;
        if (d.live) {
          const uint32_t qbytes = (uint32_t)(d.nq * H * F::kRow), wbytes = (uint32_t)(d.nq * H * 4);
          mbar_arrive_expect_tx(bar_qfull(qb), qbytes + wbytes);
          bulk_g2s(smem_u32(smem + C::OFF_QSTG + qb * C::QSTG_STRIDE), a.q_rows + (size_t)d.row0 * H * F::kRow,
                   qbytes, bar_qfull(qb));
          bulk_g2s(smem_u32(smem + C::OFF_W + qb * C::W_STRIDE), a.w_prime + (size_t)d.row0 * H, wbytes,
                   bar_qfull(qb));
        } else {
          mbar_arrive(bar_qfull(qb));   // no more groups: the other roles stop here
        }
        info[2] = (uint32_t)(k + 1);
      }
      __syncwarp();
      if (!d.live) break;
      const int npages = (d.Tb + kPageKeys - 1) / kPageKeys;
      for (int i0 = 0; i0 < d.nt && !failed; i0 += 32) {
        int p0 = -1, p1 = -1;   // this lane's tile: its two pool pages (looked up in parallel)
        if (i0 + lane < d.nt) {
          const int lp = 2 * (i0 + lane);
          p0 = pool_page(a, d.b, lp);
          p1 = pool_page(a, d.b, lp + 1 < npages ? lp + 1 : -1);
          if (p0 == -2 || p1 == -2) atomicOr(a.status, kStatusBadMeta);
        }
        const int n = min(32, d.nt - i0);
        // C::PBATCH tiles at a time, each requested by the lane that looked up its pages: the
        // lanes poll their stages' barriers together, so a batch pays one poll's latency (a
        // completed barrier still costs ~150 cycles to branch on) instead of one per tile
        for (int u0 = 0; u0 < n; u0 += C::PBATCH) {
          const int nb = min(C::PBATCH, n - u0);
          const bool mine = lane >= u0 && lane < u0 + nb;
          const uint32_t jj = j + (uint32_t)(lane - u0);   // this lane's tile (when mine)
          const int st = (int)(jj % C::NSTAGE);
          // the stage's previous tile: its MMA has completed (FP8: and its key scales were read)
          bool ok = true;
          if (mine && jj >= (uint32_t)C::NSTAGE)
            ok = mbar_wait(F::kFp8 ? bar_sread(st) : bar_free(st), ((jj / C::NSTAGE) - 1) & 1u, wait_ns);
          if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
            break;
          }
          if (mine) issue_tile_load<F>(a, max(p0, -1), max(p1, -1), stg0 + st * F::kStage, bar_full(st));
          j += (uint32_t)nb;
          if (lane == 0) info[1] = j;
          __syncwarp();
        }
      }
      if (failed) break;
    }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ scale warpgroup
    const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);   // this warp's lane quadrant
    const int key = tid;   // this thread's key (TMEM lane) within a tile
    uint32_t j = 0;
    for (int k = 0;; ++k) {
      const int qb = k & 1;
      // the four warps agree at every group start (a warp that gave up inside the previous
      // group has skipped its remaining waits and arrives here with failed set)
      if (!named_bar_and(1, 128, !failed && warp_wait(bar_qfull(qb), (uint32_t)(k >> 1) & 1u, wait_ns))) {
        failed = true;
        break;
      }
      const GroupDesc d = gdesc[qb];
      if (!d.live) break;
      if (d.nt == 0) {
        warp_arrive(bar_qfree(qb));
        continue;
      }
      // query rows -> B operand buffer qb (core-matrix order) and B scale set qb
      uint8_t* qB = smem + C::OFF_QB + qb * C::QB_STRIDE;
      const uint8_t* qstg = smem + C::OFF_QSTG + qb * C::QSTG_STRIDE;
      build_b_operand<F, C::NCB * 32, C::NP>(qstg, qB, sfw, d.nq * H, tid);
      fence_proxy_async_smem();   // the B operand was written by ordinary stores
      named_bar_sync(1, 128);
      // done with the buffer's descriptor and raw rows (the B operand itself stays in use
      // until the group's MMAs complete, which the epilogue's release covers)
      warp_arrive(bar_qfree(qb));
      const uint32_t sfb = (uint32_t)(C::SFB_COL + qb * 2 * C::SB);
      if constexpr (!F::kFp8) {
#pragma unroll
        for (int jj = 0; jj < C::NCB; ++jj) {
          const uint32_t wd = sfw[32 * jj + lane];
          tmem_st_x1(tq + sfb + jj, wd & 0xFFFFu);
          tmem_st_x1(tq + sfb + C::SB + jj, wd >> 16);
        }
      }
      // tile j's stage and scale set, kept as a counter (one set per stage). Two tiles per
      // poll: the warps pay one poll's latency (a wait on completed barriers still costs ~180
      // cycles) and one loop's bookkeeping for both
      RingPos<C::NSTAGE> rs(j);
      for (int i = 0; i < d.nt;) {
        const bool two = i + 1 < d.nt;   // (warp-uniform)
        RingPos<C::NSTAGE> rs1 = rs;
        rs1.template advance<1>();
        if (!failed) {   // after a failure no more waits; the next group start reports it
          // the tiles have landed, so their scale sets are free; each warp goes on by itself
          // and arrives on the sets' "ready" barriers
          if (!warp_wait2(bar_full(rs.slot), rs.phase, bar_full(rs1.slot), rs1.phase, two, wait_ns)) {
            failed = true;
          } else {
            tc_fence_after();
            if constexpr (!F::kFp8) {   // the tiles' A scales
              const uint32_t w = *reinterpret_cast<const uint32_t*>(stg + rs.slot * F::kStage + page_scale_offset(key));
              const uint32_t lo = w & 0xFFFFu, hi = w >> 16;
              tmem_st_x8(tq + (uint32_t)(C::SFA_COL + 8 * rs.slot), lo, lo, lo, lo, hi, hi, hi, hi);
              if (two) {
                const uint32_t w1 =
                    *reinterpret_cast<const uint32_t*>(stg + rs1.slot * F::kStage + page_scale_offset(key));
                const uint32_t lo1 = w1 & 0xFFFFu, hi1 = w1 >> 16;
                tmem_st_x8(tq + (uint32_t)(C::SFA_COL + 8 * rs1.slot), lo1, lo1, lo1, lo1, hi1, hi1, hi1, hi1);
              }
            }
            tmem_wait_st();   // (also the group's B scales, for its first tile)
            tc_fence_before();
            warp_arrive(bar_ready(rs.slot));
            if (two) warp_arrive(bar_ready(rs1.slot));
          }
        }
        if (two) {
          i += 2;
          j += 2;
          rs.template advance<2>();
        } else {
          i += 1;
          j += 1;
          rs = rs1;
        }
      }
    }
  } else if (warp >= C::MMA_WARP && warp < C::PRODUCER_WARP) {
    // ------------------------------------------------------------ MMA warps (tile j is warp j % NMMA's)
    const int mid = warp - C::MMA_WARP;
    uint32_t j = 0;
    // this warp's tiles: global numbers mid, mid + NMMA, ... across all groups
    uint32_t jt = (uint32_t)mid;
    RingPos<C::NSTAGE> rst(jt);
    RingPos<C::NACC> rc(jt);
    RingPos<C::NSC> rsc(jt);
    uint32_t eph = 0u;   // bit c: parity of this warp's next wait on accumulator c's barrier
    for (int k = 0; !failed; ++k) {
      const int qb = k & 1;
      if (!warp_wait(bar_qfull(qb), (uint32_t)(k >> 1) & 1u, wait_ns)) {
        failed = true;
        break;
      }
      const GroupDesc d = gdesc[qb];
      if (!d.live) break;
      warp_arrive(bar_qfree(qb));   // the descriptor is in registers
      const uint32_t qbaddr = smem_u32(smem + C::OFF_QB + qb * C::QB_STRIDE);
      const uint32_t sfb = (uint32_t)(C::SFB_COL + qb * 2 * C::SB);
      // this warp's tiles of the group
      const uint32_t jend = j + (uint32_t)d.nt;
      for (; jt < jend; jt += NMMA, rst.template advance<NMMA>(), rc.template advance<NMMA>(), rsc.template advance<NMMA>()) {
        const int st = rst.slot, c = rc.slot, sc = rsc.slot;
        // the tile's scale set is ready (the scale warps arrive only after they have seen the
        // tile's copy land, so the tile is in place too) and accumulator c has been drained by
        // the epilogue of tile jt - NACC (the accumulator's previous round)
        // (this warp's barrier for accumulator c: its phases are the releases of the tiles
        // before this warp's tiles on c, in order; bit c of eph is the next one's parity)
        const bool reuse = jt >= (uint32_t)C::NACC;
        const bool ok = warp_wait2(bar_ready(sc), rsc.phase, bar_empty(c, mid), (eph >> c) & 1u, reuse, wait_ns);
        if (!ok) {
          failed = true;
          break;
        }
        if (reuse) eph ^= 1u << c;
        if (lane == 0) {
          tc_fence_after();
          const uint32_t pa = stg0 + (uint32_t)(st * F::kStage);
          const uint32_t acc = tmem + (uint32_t)(c * C::NP);
          const uint32_t sfa = tmem + (uint32_t)(C::SFA_COL + 8 * sc);
          issue_tile_mma<F, C::NP>(acc, pa, qbaddr, sfa, tmem + sfb, C::SB);
          tc_commit(bar_free(st));   // the stage may be refilled and the accumulator read
          info[3 + mid] = jt + 1;
        }
        __syncwarp();
      }
      j = jend;
    }
  } else if (warp >= 4 && warp < C::MMA_WARP) {
    // ------------------------------------------------------------ epilogue warpgroups
    constexpr int P = H >= 32 ? 4 : 2;   // independent partial sums per row (pairs of heads)
    const int grp = (warp - 4) >> 2;
    const int et = (tid - 128) & (kEpiThreads - 1);   // key within the tile == TMEM lane
    const int ge = tid - 128;
    const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t j = 0;
    // this warpgroup's tiles: global numbers grp, grp + EPI, ... across all groups
    uint32_t jt = (uint32_t)grp;
    RingPos<C::NSTAGE> rst(jt);
    RingPos<C::NACC> rc(jt);
    for (int k = 0; !failed; ++k) {
      const int qb = k & 1;
      if (!warp_wait(bar_qfull(qb), (uint32_t)(k >> 1) & 1u, wait_ns)) {
        failed = true;
        break;
      }
      const GroupDesc d = gdesc[qb];
      if (!d.live) break;
      const float* wq = reinterpret_cast<const float*>(smem + C::OFF_W + qb * C::W_STRIDE);
      if constexpr (F::kFp8) {
        // w' times each query row's scale, written by all epilogue threads (bounded wait
        // on the buffer's barrier before use)
        float* ws = reinterpret_cast<float*>(smem + C::OFF_WS + qb * C::W_STRIDE);
        const uint8_t* qstg = smem + C::OFF_QSTG + qb * C::QSTG_STRIDE;
        for (int n = ge; n < C::N; n += EPI * kEpiThreads)
          ws[n] = n < d.nq * H ? wq[n] * *reinterpret_cast<const float*>(qstg + n * F::kRow + F::kCode) : 0.f;
        warp_arrive(bar_wsready(qb));
        if (!warp_wait(bar_wsready(qb), (uint32_t)(k >> 1) & 1u, wait_ns)) {
          failed = true;
          break;
        }
        wq = ws;
      }
      if (a.fill_masked) {   // -inf over the tiles no row of the group can see
        const int t_begin = d.nt * kTileKeys;
        for (int qi = 0; qi < d.nq; ++qi) {
          float* dst = a.scores + (size_t)(d.row0 + qi) * a.ld;
          for (int t = t_begin + ge; t < d.Tb; t += EPI * kEpiThreads) dst[t] = -__int_as_float(0x7f800000);
        }
      }
      // keys each row of the group may see
      int visq[QG];
#pragma unroll
      for (int qi = 0; qi < QG; ++qi) visq[qi] = min(d.Tb, (d.pos0 + qi + 1) / a.ratio);
      // this warpgroup's tiles of the group
      const uint32_t jend = j + (uint32_t)d.nt;
      for (; jt < jend && !failed; jt += EPI, rst.template advance<EPI>(), rc.template advance<EPI>()) {
        const int i = (int)(jt - j);   // the tile within the group
        const int c = rc.slot, st = rst.slot;
        // tile jt's MMA has completed (its stage's barrier; the stage cannot be refilled and
        // complete again before this accumulator is released, as NSTAGE > NACC)
        if (!warp_wait(bar_free(st), rst.phase, wait_ns)) {
          failed = true;
          break;
        }
        float sk = 1.f;   // FP8: this key's scale; the stage may be refilled once all are read
        if constexpr (F::kFp8) {
          sk = *reinterpret_cast<const float*>(stg + st * F::kStage + page_scale_offset_fp8(et));
          warp_arrive(bar_sread(st));
        }
        tc_fence_after();
        float part[QG][P];
#pragma unroll
        for (int qi = 0; qi < QG; ++qi)
#pragma unroll
          for (int p = 0; p < P; ++p) part[qi][p] = 0.f;
        // 32-column pieces of the accumulator, read one at a time (reading each piece ahead of
        // the previous piece's arithmetic took more instructions and time); the accumulator is
        // released once the last piece is in registers
        constexpr int NH = C::NCB;
        const uint32_t acc_addr = tq + (uint32_t)(c * C::NP);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          uint32_t cur[32];
          tmem_ld32_issue(acc_addr + (uint32_t)(32 * h), cur);
          tmem_ld32_wait(cur);
          if (h + 1 == NH) {
            tc_fence_before();
            // accumulator c may take tile jt + NACC (issued by MMA warp (jt + NACC) % NMMA)
            warp_arrive(bar_empty(c, (int)((jt + (uint32_t)C::NACC) % (uint32_t)NMMA)));
          }
#pragma unroll
          for (int u = 0; u < 32; u += 4) {
            const int n = 32 * h + u;
            if (n < C::N) {
              const float4 w4 = *reinterpret_cast<const float4*>(wq + n);
              const int qi = n / H, p0 = (n % P), p1 = ((n + 2) % P);
              // 2 max(dot, 0) = dot + |dot| for two elements at once (the halving is applied to
              // the row's sum: exact, a power of two)
              const float2 r01 = twice_relu2(__uint_as_float(cur[u]), __uint_as_float(cur[u + 1]));
              const float2 r23 = twice_relu2(__uint_as_float(cur[u + 2]), __uint_as_float(cur[u + 3]));
              ffma2(part[qi][p0], part[qi][p0 + 1], w4.x, w4.y, r01.x, r01.y);
              ffma2(part[(n + 2) / H][p1], part[(n + 2) / H][p1 + 1], w4.z, w4.w, r23.x, r23.y);
            }
          }
        }
        const int t = i * kTileKeys + et;
        if (t < d.Tb) {
#pragma unroll
          for (int qi = 0; qi < QG; ++qi) {
            if (qi < d.nq) {
              float acc = part[qi][0];
#pragma unroll
              for (int p = 1; p < P; ++p) acc += part[qi][p];
              acc *= 0.5f;   // the partial sums hold twice the head sum
              if constexpr (F::kFp8) acc *= sk;
              a.scores[(size_t)(d.row0 + qi) * a.ld + t] = t < visq[qi] ? acc : -__int_as_float(0x7f800000);
            }
          }
        }
        __syncwarp();
      }
      j = jend;
      if (failed) break;
      warp_arrive(bar_qfree(qb));   // this warp is done with the group's query buffer
    }
  }
  __syncwarp();
  if (failed && lane == 0)
    atomicOr(a.status, warp >= 4 && warp < C::MMA_WARP ? kStatusMmaTimeout : kStatusLoadTimeout);
  // on failure, bounded waits for whatever may still be in flight before shared and tensor
  // memory go
  const bool any_failed = __syncthreads_or(failed);
  if (any_failed && tid == 0) {
    const int issued = (int)info[1], qph = (int)info[2];
    for (int st = 0; st < C::NSTAGE && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / C::NSTAGE) * C::NSTAGE;
      mbar_wait(bar_full(st), (uint32_t)(last / C::NSTAGE) & 1u, wait_ns);
    }
    for (int q = 0; q < 2 && q < qph; ++q) {
      const int last = q + ((qph - 1 - q) / 2) * 2;
      mbar_wait(bar_qfull(q), (uint32_t)(last >> 1) & 1u, wait_ns);
    }
    for (int m = 0; m < NMMA; ++m) {   // each MMA warp's last tile (its commit tracks all its MMAs)
      const int mmas = (int)info[3 + m];
      if (mmas > 0) mbar_wait(bar_free((mmas - 1) % C::NSTAGE), (uint32_t)((mmas - 1) / C::NSTAGE) & 1u, wait_ns);
    }
  }
  __syncthreads();
  if (tid == 0) {   // the last CTA to finish rewinds the group counter for the next launch
    __threadfence();
    if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
      a.sched[0] = 0u;
      a.sched[1] = 0u;
      __threadfence();
    }
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}


template <int H, int QG, int EPI, class F>
cudaError_t launch_cfg(ScoreArgs a, cudaStream_t stream) {
  using C = ScoreCfg<H, QG, EPI, F>;
  const int cand_words = a.cand ? ((a.T + a.cbs - 1) / a.cbs + 31) / 32 : 0;
  const size_t smem = (size_t)C::OFF_CAND + (size_t)QG * cand_words * 4 + 1024;   // + base alignment slack
  if (a.sparse_pages && (QG != 1 || (a.groups == nullptr && a.S != 1) || a.cand == nullptr ||
                         (a.T + kPageKeys - 1) / kPageKeys > kMaxPages))
    return cudaErrorInvalidValue;
  // the attributes are set once per device and kernel (the dynamic size only grows)
  static int set_bytes[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || set_bytes[dev] < (int)smem) {
    err = cudaFuncSetAttribute(score_kernel<H, QG, EPI, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(score_kernel<H, QG, EPI, F>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) set_bytes[dev] = (int)smem;
  }
  int ntiles = (a.T + kTileKeys - 1) / kTileKeys;
  if (a.sparse_pages) {   // at most the pages of the kept blocks, two per tile
    const long long pages = (long long)a.cbk * ((a.cbs + kPageKeys - 1) / kPageKeys + 1);
    ntiles = (int)min((long long)ntiles, (pages + 1) / 2);
  }
  const long long base = a.groups ? (long long)a.n_groups : (long long)((a.S + QG - 1) / QG) * a.B;
  if (base <= 0) return cudaSuccess;
  // resident CTAs per SM: tensor memory (512 columns) and shared memory (227 KB) both bound it
  const int by_tmem = 512 / (int)C::TMEM_COLS;
  const int by_smem = (int)((227 * 1024) / (smem + 1024));
  const int per_sm = by_tmem < by_smem ? by_tmem : by_smem;
  const long long target = (long long)sm_count() * (per_sm > 0 ? per_sm : 1);
  // few query groups (decode): split each sequence's tiles over CTAs, one wave in total
  int tpc = ntiles;
  if (base < target) {
    tpc = (int)((ntiles * base + target - 1) / target);
    if (tpc < 1) tpc = 1;
    while (tpc < ntiles && (long long)((ntiles + tpc - 1) / tpc) * base > target) ++tpc;
  }
  if (tpc > kMaxTilesCta) tpc = kMaxTilesCta;
  a.tiles_per_cta = tpc;
  dim3 grid((ntiles + tpc - 1) / tpc, 1, 1);
  if (a.groups) {   // group g = blockIdx.z * gridDim.y + blockIdx.y
    grid.y = (unsigned)min(base, 65535ll);
    grid.z = (unsigned)((base + grid.y - 1) / grid.y);
  } else {
    grid.y = (unsigned)((a.S + QG - 1) / QG);
    grid.z = (unsigned)a.B;
  }
  return launch_overlapped(score_kernel<H, QG, EPI, F>, grid, dim3(C::THREADS), smem, stream, a);
}

template <int H, int QG, int EPI, int NMMA, class F>
cudaError_t launch_rows(ScoreArgs a, cudaStream_t stream) {
  using C = RowsCfg<H, QG, EPI, NMMA, F>;
  const size_t smem = (size_t)C::SMEM + 1024;   // + base alignment slack
  static int set_bytes[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || set_bytes[dev] < (int)smem) {
    err = cudaFuncSetAttribute(score_rows_kernel<H, QG, EPI, NMMA, F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(score_rows_kernel<H, QG, EPI, NMMA, F>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) set_bytes[dev] = (int)smem;
  }
  const long long groups = a.groups ? (long long)a.n_groups : (long long)((a.S + QG - 1) / QG) * a.B;
  if (groups <= 0) return cudaSuccess;
  const long long ctas = groups < sm_count() ? groups : sm_count();   // one persistent CTA per SM
  // plain stream order: started early, the persistent CTAs measured slower steps (the large
  // prefill 3.017 against 2.988 ms; their work runs for milliseconds, their start-up for
  // microseconds)
  return launch_kernel(false, score_rows_kernel<H, QG, EPI, NMMA, F>, dim3((unsigned)ctas), dim3(C::THREADS), smem,
                       stream, a);
}

// The several-row kernel's epilogue warpgroups and MMA warps: three epilogue warpgroups for
// every head count (64 heads: 2048-key prefill scores 85.6 against 93.9 us with two, 8192-key
// rows 2.058 against 2.392 ms; 8, 32 and 128 heads over 8192-key rows 10-14 % faster than
// with two), two MMA warps (a third: 2.069 ms).
constexpr int kRowsEpi = 3, kRowsMma = 2;

template <class F>
cudaError_t launch_scores_fmt(const ScoreArgs& a, cudaStream_t stream) {
  // S == 1: one query row per group (a uniform batch of single rows, or row groups planned
  // with score_group_rows(H, true))
  const bool single = a.S == 1;
  if (!single && a.cand == nullptr && a.sched != nullptr) {
    // several rows per group: the persistent kernel (N = 128, kRowsEpi epilogue warpgroups,
    // kRowsMma MMA warps taking alternate tiles)
    switch (a.H) {
      case 8: return launch_rows<8, 16, kRowsEpi, kRowsMma, F>(a, stream);
      case 16: return launch_rows<16, 8, kRowsEpi, kRowsMma, F>(a, stream);
      case 32: return launch_rows<32, 4, kRowsEpi, kRowsMma, F>(a, stream);
      case 64: return launch_rows<64, 2, kRowsEpi, kRowsMma, F>(a, stream);
      case 128: return launch_rows<128, 1, kRowsEpi, kRowsMma, F>(a, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.H) {
    // decode: one query row, N = H, two CTAs per SM; several rows with a level-two filter:
    // N = 128 and two epilogue warpgroups
    case 8: return single ? launch_cfg<8, 1, 1, F>(a, stream) : launch_cfg<8, 16, 2, F>(a, stream);
    case 16: return single ? launch_cfg<16, 1, 1, F>(a, stream) : launch_cfg<16, 8, 2, F>(a, stream);
    case 32: return single ? launch_cfg<32, 1, 1, F>(a, stream) : launch_cfg<32, 4, 2, F>(a, stream);
    case 64: return single ? launch_cfg<64, 1, 1, F>(a, stream) : launch_cfg<64, 2, 2, F>(a, stream);
    case 128: return single ? launch_cfg<128, 1, 1, F>(a, stream) : launch_cfg<128, 1, 2, F>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_scores(const ScoreArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  return a.fp8 ? launch_scores_fmt<FmtFp8>(a, stream) : launch_scores_fmt<FmtMxfp4>(a, stream);
}

int score_group_rows(int H, bool single) {
  if (single) return 1;
  switch (H) {
    case 8: return 16;
    case 16: return 8;
    case 32: return 4;
    case 64: return 2;
    default: return 1;
  }
}

}  // namespace indexer
