// Index scoring on the 5th-generation tensor cores (tcgen05, kind::mxf4 block-scaled).
//
// score[b,s,t] = sum_h w'[b,s,h] * relu( qhat[b,s,h,:] . khat[b,t,:] )
// ("DeepSeek V4.1" index-keys page, Indexer.forward: einsum bshd,btd->bsht, relu,
// times weights, sum over heads), with t >= vis(s) = (start_pos + s + 1) / ratio
// masked to -inf and, for a level-two layer, -inf outside the candidate blocks.
//
// One CTA (128 threads) takes a group of QG query rows of one sequence and a run of
// 128-key tiles:
//   * A operand (M = 128): the key tile. Its 68-byte cache rows arrive by one bulk TMA
//     copy (cp.async.bulk) into a staging buffer; thread m rewrites row m into the
//     K-major no-swizzle core-matrix layout (8 rows x 16 bytes per core matrix) and
//     its 4 UE8M0 scale bytes into tensor memory.
//   * B operand (N = QG * H, padded to 16): the group's quantised query heads, loaded
//     once per CTA in the same layout; scales in tensor memory.
//   * Two MMAs (K = 64 each, scale blocks {0,1} then {2,3}) accumulate the 128 x N f32
//     head dot products in tensor memory; the next tile's copy is in flight meanwhile.
//   * Epilogue: thread m owns key t0 + m (TMEM lane m) and reads its N head scores with
//     tcgen05.ld; for every query row it forms sum_h w' * max(dot, 0) in f32 -- the
//     head reduction needs no shuffles because keys, not heads, sit on the lanes.
//
// Scale-factor placement in tensor memory (per 32-bit column, bytes 0/1 = the two
// scale blocks of one K = 64 MMA): B row n = 32j + i sits in column j of lane i of every
// 32-lane quadrant; A row m is written to lane m of all four columns of its set.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace indexer {

namespace {

constexpr int kTileKeys = 128;
constexpr int kStageBytes = kTileKeys * kRowBytes;   // 8704
constexpr int kABytes = kTileKeys * kCodeBytes;      // 8192

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

template <int H, int QG>
struct ScoreCfg {
  static constexpr int N = QG * H;
  static constexpr int NP = round_up(N, 16);         // MMA N
  static constexpr int NCB = (NP + 31) / 32;         // scale columns per set
  // Every scale-factor set starts on a 4-column boundary (an MMA given a scale set at an
  // odd column faulted with a misaligned address).
  static constexpr int SB = round_up(NCB, 4);        // column stride between the two B sets
  static constexpr int SFA_COL = NP;                 // 2 sets x 4 columns
  static constexpr int SFB_COL = NP + 8;             // 2 sets x SB columns
  static constexpr int TMEM_NEED = NP + 8 + 2 * SB;
  static_assert(SFA_COL % 4 == 0 && SFB_COL % 4 == 0 && SB % 4 == 0, "scale sets must be 4-column aligned");
  static constexpr uint32_t TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128
                                        : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int OFF_QB = 0;
  static constexpr int OFF_KA = round_up(NP * kCodeBytes, 1024);
  static constexpr int OFF_STG = OFF_KA + kABytes;
  static constexpr int OFF_W = OFF_STG + 2 * kStageBytes;
  static constexpr int OFF_SFW = OFF_W + round_up(N * 4, 16);
  static constexpr int OFF_BAR = OFF_SFW + NCB * 32 * 4;
  static constexpr int OFF_TSLOT = OFF_BAR + 3 * 8;
  static constexpr int OFF_CAND = round_up(OFF_TSLOT + 4, 16);
  static_assert(N <= 256, "MMA N is at most 256");
};

__device__ __forceinline__ void issue_tile_load(const ScoreArgs& a, int b, int tile, uint32_t stage_addr,
                                                uint32_t bar) {
  const int t0 = tile * kTileKeys;
  const int nv = min(kTileKeys, a.T - t0);
  const uint32_t bytes = (uint32_t)(round_up(nv, 4) * kRowBytes);   // multiple of 16; stays below T_cap
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s(stage_addr, a.k_cache + ((size_t)b * a.T_cap + t0) * kRowBytes, bytes, bar);
}

template <int H, int QG>
__global__ void __launch_bounds__(128, 1) score_kernel(const ScoreArgs a) {
  using C = ScoreCfg<H, QG>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1024-byte aligned base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z;
  const int s0 = blockIdx.y * QG;
  const int nq = min(QG, a.S - s0);
  const int ntiles = (a.T + kTileKeys - 1) / kTileKeys;
  const int tiles_per_cta = (ntiles + gridDim.x - 1) / gridDim.x;
  const int tile0 = blockIdx.x * tiles_per_cta;
  const int tile1 = min(tile0 + tiles_per_cta, ntiles);
  if (nq <= 0 || tile0 >= tile1) return;
  // keys the group's last row can see; tiles at or past it are fully masked
  const int vis_hi = min(a.T, (a.start_pos + s0 + nq) / a.ratio);
  const int tile_vis = min(tile1, (vis_hi + kTileKeys - 1) / kTileKeys);
  if (a.fill_masked) {
    const int t_begin = max(tile0, tile_vis) * kTileKeys, t_end = min(tile1 * kTileKeys, a.T);
    for (int qi = 0; qi < nq; ++qi) {
      float* dst = a.scores + ((size_t)b * a.S + s0 + qi) * a.T;
      for (int t = t_begin + tid; t < t_end; t += 128) dst[t] = -__int_as_float(0x7f800000);
    }
  }
  if (tile_vis <= tile0) return;

  uint8_t* qB = smem + C::OFF_QB;
  uint8_t* kA = smem + C::OFF_KA;
  uint8_t* stg = smem + C::OFF_STG;
  float* wq = reinterpret_cast<float*>(smem + C::OFF_W);
  uint32_t* sfw = reinterpret_cast<uint32_t*>(smem + C::OFF_SFW);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::OFF_TSLOT);
  uint32_t* cand_bits = reinterpret_cast<uint32_t*>(smem + C::OFF_CAND);
  const uint32_t bar_ld[2] = {smem_u32(&bars[0]), smem_u32(&bars[1])};
  const uint32_t bar_mma = smem_u32(&bars[2]);
  const uint32_t stg_addr[2] = {smem_u32(stg), smem_u32(stg + kStageBytes)};

  if (tid == 0) {
    mbar_init(bar_ld[0], 1);
    mbar_init(bar_ld[1], 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), C::TMEM_COLS);
    tmem_relinquish();
  }
  // head weights of the group (0 for rows past S)
  for (int n = tid; n < C::N; n += 128) {
    const int qi = n / H;
    wq[n] = qi < nq ? a.w_prime[((size_t)b * a.S + s0 + qi) * H + (n % H)] : 0.f;
  }
  // quantised query rows -> B operand (core-matrix layout) and scale words
  for (int n = tid; n < C::NCB * 32; n += 128) {
    uint32_t w[16];
    uint32_t sc = 0x7F7F7F7Fu;
    if (n < C::N && n / H < nq) {
      const uint32_t* src =
          reinterpret_cast<const uint32_t*>(a.q_rows + (((size_t)b * a.S + s0 + n / H) * H + (n % H)) * kRowBytes);
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = src[i];
      sc = src[16];
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = 0u;
    }
    if (n < C::NP) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(qB + (n >> 3) * 512 + c * 128 + (n & 7) * 16) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
    sfw[n] = sc;
  }
  // level-two candidate filter: one bit per block of cbs positions, per query row
  const int cand_words = a.cand ? ((a.T + a.cbs - 1) / a.cbs + 31) / 32 : 0;
  if (a.cand) {
    for (int i = tid; i < QG * cand_words; i += 128) cand_bits[i] = 0u;
    __syncthreads();
    for (int i = tid; i < nq * a.cbk; i += 128) {
      const int qi = i / a.cbk;
      const int blk = a.cand[((size_t)b * a.S + s0 + qi) * a.cbk + (i % a.cbk)];
      if (blk >= 0 && blk < cand_words * 32) atomicOr(&cand_bits[qi * cand_words + (blk >> 5)], 1u << (blk & 31));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(warp * 32) << 16);   // this warp's lane quadrant
#pragma unroll
  for (int j = 0; j < C::NCB; ++j) {
    const uint32_t wd = sfw[32 * j + lane];
    tmem_st_x1(tq + C::SFB_COL + j, wd & 0xFFFFu);
    tmem_st_x1(tq + C::SFB_COL + C::SB + j, wd >> 16);
  }
  if (tid == 0) issue_tile_load(a, b, tile0, stg_addr[0], bar_ld[0]);

  const uint32_t idesc = idesc_mxf4(128, C::NP);
  const uint32_t qb_addr = smem_u32(qB), ka_addr = smem_u32(kA);
  bool load_pending = true;   // tile0's copy
  int pending_stage = 0, pending_parity = 0;
  bool ok = true;
  int it = 0;
  for (int tile = tile0; tile < tile_vis; ++tile, ++it) {
    const int st = it & 1;
    const int t0 = tile * kTileKeys;
    const int nv = min(kTileKeys, a.T - t0);
    const bool got = mbar_wait(bar_ld[st], (it >> 1) & 1);
    if (__syncthreads_and(got) == 0) {
      if (tid == 0) atomicOr(a.status, kStatusLoadTimeout);
      ok = false;
      break;
    }
    load_pending = false;
    // A operand: key row tid -> core-matrix layout; scale word -> tensor memory
    uint32_t w[17];
    if (tid < nv) {
      const uint32_t* raw = reinterpret_cast<const uint32_t*>(stg + st * kStageBytes + tid * kRowBytes);
#pragma unroll
      for (int i = 0; i < 17; ++i) w[i] = raw[i];
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = 0u;
      w[16] = 0x7F7F7F7Fu;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(kA + (tid >> 3) * 512 + c * 128 + (tid & 7) * 16) =
          make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    const uint32_t s01 = w[16] & 0xFFFFu, s23 = w[16] >> 16;
    tmem_st_x8(tq + C::SFA_COL, s01, s01, s01, s01, s23, s23, s23, s23);
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      if (tile + 1 < tile_vis) issue_tile_load(a, b, tile + 1, stg_addr[st ^ 1], bar_ld[st ^ 1]);
      mma_mxf4(tmem, smem_desc(ka_addr, 128, 512), smem_desc(qb_addr, 128, 512), idesc, tmem + C::SFA_COL,
               tmem + C::SFB_COL, 0u);
      mma_mxf4(tmem, smem_desc(ka_addr + 256, 128, 512), smem_desc(qb_addr + 256, 128, 512), idesc,
               tmem + C::SFA_COL + 4, tmem + C::SFB_COL + C::SB, 1u);
      tc_commit(bar_mma);
    }
    if (tile + 1 < tile_vis) {
      load_pending = true;
      pending_stage = st ^ 1;
      pending_parity = ((it + 1) >> 1) & 1;
    }
    const bool done = mbar_wait(bar_mma, it & 1);
    if (__syncthreads_and(done) == 0) {
      if (tid == 0) atomicOr(a.status, kStatusMmaTimeout);
      ok = false;
      mbar_wait(bar_mma, it & 1);   // one more bounded wait before the tensor memory is released
      break;
    }
    tc_fence_after();

    // epilogue: key t0 + tid, all N head scores of the group
    float acc[QG];
#pragma unroll
    for (int qi = 0; qi < QG; ++qi) acc[qi] = 0.f;
#pragma unroll
    for (int c = 0; c < C::NCB; ++c) {
      float v[32];
      tmem_ld32(tq + 32 * c, v);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int n = 32 * c + jj;
        if (n < C::N) acc[n / H] = fmaf(wq[n], fmaxf(v[jj], 0.f), acc[n / H]);
      }
    }
    if (tid < nv) {
      const int t = t0 + tid;
#pragma unroll
      for (int qi = 0; qi < QG; ++qi) {
        if (qi < nq) {
          const int s = s0 + qi;
          const int vis = min(a.T, (a.start_pos + s + 1) / a.ratio);
          bool keep = t < vis;
          if (a.cand) {
            const int blk = t / a.cbs;
            keep = keep && ((cand_bits[qi * cand_words + (blk >> 5)] >> (blk & 31)) & 1u);
          }
          a.scores[((size_t)b * a.S + s) * a.T + t] = keep ? acc[qi] : -__int_as_float(0x7f800000);
        }
      }
    }
    tc_fence_before();
  }
  if (!ok && load_pending) mbar_wait(bar_ld[pending_stage], pending_parity);   // bounded
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int H, int QG>
cudaError_t launch_cfg(const ScoreArgs& a, cudaStream_t stream) {
  using C = ScoreCfg<H, QG>;
  const int cand_words = a.cand ? ((a.T + a.cbs - 1) / a.cbs + 31) / 32 : 0;
  const size_t smem = (size_t)C::OFF_CAND + (size_t)QG * cand_words * 4 + 1024;   // + base alignment slack
  cudaError_t err = cudaFuncSetAttribute(score_kernel<H, QG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int ntiles = (a.T + kTileKeys - 1) / kTileKeys;
  const int groups = (a.S + QG - 1) / QG;
  // decode-like shapes (few query groups): split the keys of a sequence over CTAs
  int chunks = 1;
  const long long base_ctas = (long long)groups * a.B;
  if (base_ctas < 600) {
    chunks = (int)((600 + base_ctas - 1) / base_ctas);
    if (chunks > ntiles) chunks = ntiles;
    if (chunks < 1) chunks = 1;
  }
  dim3 grid(chunks, groups, a.B);
  score_kernel<H, QG><<<grid, 128, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scores(const ScoreArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const bool single = a.S == 1;
  switch (a.H) {
    case 8: return single ? launch_cfg<8, 1>(a, stream) : launch_cfg<8, 32>(a, stream);
    case 16: return single ? launch_cfg<16, 1>(a, stream) : launch_cfg<16, 16>(a, stream);
    case 32: return single ? launch_cfg<32, 1>(a, stream) : launch_cfg<32, 8>(a, stream);
    case 64: return single ? launch_cfg<64, 1>(a, stream) : launch_cfg<64, 4>(a, stream);
    case 128: return single ? launch_cfg<128, 1>(a, stream) : launch_cfg<128, 2>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace indexer
