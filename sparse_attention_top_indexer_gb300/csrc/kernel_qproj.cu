// Query projection fused with query prep ("DeepSeek V4.1" index-keys page, Indexer.forward:
// q = wq_b(qr) unflattened to [H][128], RoPE on the last rope_dim dims at the row's
// position, fp4_act_quant): the bf16 projection runs on the 5th-generation tensor cores and
// its epilogue writes the 68-byte query rows and w' directly, so the bf16 q never goes
// through HBM.
//
// One persistent CTA per SM takes output tiles of 128 query rows x 256 features (two heads):
//   * warps 0-3 (producers) copy the K-chunks of 64 of qr (A, 128 x 64) and wq_b (B,
//     256 x 64) with 16-byte cp.async into the no-swizzle K-major core-matrix layout (8 rows
//     x 16 bytes per core matrix, 128 B apart along K, 1024 B apart along M/N), four stages
//     deep; before it waits for a stage to be released, each thread signals the "full"
//     barrier of the chunk it issued two chunks earlier (its own copies of it have landed;
//     then a proxy fence), so a chunk's MMAs never wait on the completion of the chunk
//     before them;
//   * warp 4 (MMA) issues four tcgen05.mma.kind::f16 (bf16 x bf16 -> f32, M 128, N 256,
//     K 16) per stage into one of two accumulators (2 x 256 tensor-memory columns) and
//     commits the stage back to the producers and, after the last chunk, the accumulator to
//     the epilogue;
//   * warps 5-8 (epilogue): thread m owns query row m0 + m (tensor-memory lane m) and takes
//     its two heads a 32-column block at a time: the accumulator rounded to bf16 (q as the
//     Linear's bf16 output; optionally stored for parity checks), RoPE on the rope blocks
//     with the same f32 rotation as the query-prep kernels, the block's e8m0 scale and
//     e2m1 codes; then w' = w * head_dim^-0.5 * H^-0.5 for the row's two heads.
// Every wait on an mbarrier is bounded; a role that gives up reports through the status word.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace indexer {

namespace {

constexpr int kQpM = 128;                 // query rows per tile
constexpr int kQpN = 256;                 // output features per tile (two heads)
constexpr int kQpK = 64;                  // K per stage
constexpr int kQpStages = 4;
constexpr int kQpLag = 2;                 // chunks between a chunk's copies and its "full" signal
constexpr int kQpAStage = kQpM * kQpK * 2;            // 16 KB
constexpr int kQpBStage = kQpN * kQpK * 2;            // 32 KB
constexpr int kQpStage = kQpAStage + kQpBStage;
constexpr int kQpPieces = (kQpM + kQpN) * kQpK * 2 / 16;   // 16-byte copies per stage
constexpr int kQpProducers = 128;
constexpr int kQpThreads = kQpProducers + 32 + 128;
constexpr int kQpMmaWarp = 4;
constexpr int kQpNBar = 2 * kQpStages + 4;          // full, empty per stage; acc full, acc empty
constexpr int kQpSmem = 1024 + kQpStages * kQpStage + kQpNBar * 8 + 16;
static_assert(kQpPieces % kQpProducers == 0, "whole copies per producer thread");
static_assert(kQpLag >= 1 && kQpLag < kQpStages, "a chunk is handed over before its stage comes round again");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Offset of the 16-byte piece (row r, K group g) of a K-major no-swizzle tile.
__device__ __forceinline__ uint32_t core_offset(int r, int g) {
  return (uint32_t)((r >> 3) * 1024 + g * 128 + (r & 7) * 16);
}

__global__ void __launch_bounds__(kQpThreads, 1) qproj_prep_kernel(const QprojArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_allow_next();
  const uint32_t stg0 = smem_u32(smem);
  const uint32_t bar0 = stg0 + kQpStages * kQpStage;
  uint32_t* info = reinterpret_cast<uint32_t*>(smem + kQpStages * kQpStage + kQpNBar * 8);
  auto bar_full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (uint32_t)(kQpStages + s); };
  auto bar_accfull = [&](int x) { return bar0 + 8u * (uint32_t)(2 * kQpStages + x); };
  auto bar_accempty = [&](int x) { return bar0 + 8u * (uint32_t)(2 * kQpStages + 2 + x); };
  if (warp == 0) {
    if (lane < kQpNBar) {
      // a stage is full once all producer threads' copies of it have landed; an accumulator
      // is free once the 128 epilogue threads have read it
      const bool by_threads = lane < kQpStages || lane >= 2 * kQpStages + 2;
      mbar_init(bar0 + 8u * (uint32_t)lane, by_threads ? 128u : 1u);
    }
    fence_mbar_init();
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&info[0]), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = info[0];
  const int tiles_n = a.H / 2, tiles_m = (a.R + kQpM - 1) / kQpM;
  const int n_tiles = tiles_m * tiles_n;
  const int kchunks = a.Kq / kQpK;
  bool failed = false;
  pdl_wait();   // qr, wq_b and w may come from the kernels before

  if (warp < kQpMmaWarp) {
    // ------------------------------------------------------------ producers
    uint32_t g = 0;   // stages filled so far
    for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
      const int m0 = (t / tiles_n) * kQpM, n0 = (t % tiles_n) * kQpN;
      for (int c = 0; c < kchunks; ++c, ++g) {
        const int st = (int)(g % kQpStages);
        if (g >= (uint32_t)kQpLag) {   // chunk g - kQpLag has landed: hand it to the MMA warp
          cp_async_wait<kQpLag - 1>();
          fence_proxy_async_smem();
          mbar_arrive(bar_full((int)((g - kQpLag) % kQpStages)));
        }
        // the stage's previous chunk has been read by its MMAs (whose commit completes it)
        if (g >= (uint32_t)kQpStages && !warp_wait_bounded(bar_empty(st), ((g / kQpStages) - 1) & 1u)) {
          failed = true;
          break;
        }
        const uint32_t sa = stg0 + (uint32_t)(st * kQpStage), sb = sa + kQpAStage;
#pragma unroll 4
        for (int u = 0; u < kQpPieces / kQpProducers; ++u) {
          const int p = tid + kQpProducers * u;
          if (p < kQpM * 8) {   // qr rows m0.., rows past R read nothing (zero-filled)
            const int r = p >> 3, gk = p & 7, row = m0 + r;
            const bool live = row < a.R;
            const uint16_t* src = a.qr + (size_t)(live ? row : 0) * a.Kq + c * kQpK + gk * 8;
            cp_async16(sa + core_offset(r, gk), src, live ? 16u : 0u);
          } else {              // wq_b rows n0 .. n0 + 255 (H * 128 is a multiple of 256)
            const int q = p - kQpM * 8, r = q >> 3, gk = q & 7;
            cp_async16(sb + core_offset(r, gk), a.wq_b + (size_t)(n0 + r) * a.Kq + c * kQpK + gk * 8, 16u);
          }
        }
        cp_async_commit();
      }
    }
    cp_async_wait<0>();   // no copy stays in flight past this point
    fence_proxy_async_smem();
    for (uint32_t d = g >= (uint32_t)kQpLag ? g - kQpLag : 0u; d < g; ++d) mbar_arrive(bar_full((int)(d % kQpStages)));
  } else if (warp == kQpMmaWarp) {
    // ------------------------------------------------------------ MMA warp
    const uint32_t idesc = idesc_bf16(kQpM, kQpN);
    uint32_t g = 0;
    int ti = 0;
    for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++ti) {
      const int acc = ti & 1;
      if (ti >= 2 && !warp_wait_bounded(bar_accempty(acc), (uint32_t)((ti >> 1) - 1) & 1u)) {
        failed = true;
        break;
      }
      tc_fence_after();
      for (int c = 0; c < kchunks; ++c, ++g) {
        const int st = (int)(g % kQpStages);
        if (!warp_wait_bounded(bar_full(st), (g / kQpStages) & 1u)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sa = stg0 + (uint32_t)(st * kQpStage), sb = sa + kQpAStage;
#pragma unroll
          for (int kk = 0; kk < kQpK / 16; ++kk)   // K 16 per MMA: two core matrices along K
            mma_bf16(tmem + (uint32_t)(acc * kQpN), smem_desc(sa + 256 * kk, 128, 1024),
                     smem_desc(sb + 256 * kk, 128, 1024), idesc, (c | kk) != 0 ? 1u : 0u);
          tc_commit(bar_empty(st));
          if (c == kchunks - 1) tc_commit(bar_accfull(acc));
        }
        __syncwarp();
      }
    }
    // the last MMAs have completed before the tensor memory goes
    if (g > 0) mbar_wait(bar_empty((int)((g - 1) % kQpStages)), ((g - 1) / kQpStages) & 1u);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                 // this warp's tensor-memory lane quadrant
    const int m = quad * 32 + lane;            // the query row within the tile
    const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);
    const int rstart = kHeadDim - a.rope_dim;
    int ti = 0;
    for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++ti) {
      const int acc = ti & 1;
      const int m0 = (t / tiles_n) * kQpM, h0 = (t % tiles_n) * 2;
      const int row = m0 + m;
      const bool live = row < a.R;
      if (!warp_wait_bounded(bar_accfull(acc), (uint32_t)(ti >> 1) & 1u)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const int pos = a.start_pos + (live ? row % a.S : 0);
      const float2* cs_row = reinterpret_cast<const float2*>(a.rope_cs) + (size_t)pos * (a.rope_dim / 2);
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int h = h0 + hh;
        uint8_t* qrow = a.q_rows + ((size_t)row * a.H + h) * kRowBytes;
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
          float v[32];
          tmem_ld32(tq + (uint32_t)(acc * kQpN + hh * 128 + 32 * b), v);
          if (hh == 1 && b == 3) {
            tc_fence_before();
            mbar_arrive(bar_accempty(acc));   // the accumulator may take the tile after next
          }
          // q: the projection's bf16 output
          uint32_t qb[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) qb[i] = bf16x2_rne(v[2 * i], v[2 * i + 1]);
          if (a.q_out != nullptr && live) {
            uint4* dst = reinterpret_cast<uint4*>(a.q_out + (size_t)row * a.H * kHeadDim + h * kHeadDim + 32 * b);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(qb[4 * i], qb[4 * i + 1], qb[4 * i + 2], qb[4 * i + 3]);
          }
          float x[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            x[2 * i] = __uint_as_float(qb[i] << 16);
            x[2 * i + 1] = __uint_as_float(qb[i] & 0xFFFF0000u);
          }
          if (32 * b + 32 > rstart) {   // RoPE on the block's pairs at or past rstart
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int e0 = 32 * b + 2 * i;
              if (e0 >= rstart) rope_pair_bf16(x[2 * i], x[2 * i + 1], cs_row[(e0 - rstart) >> 1]);
            }
          }
          float am = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(x[i]));
          const int e = e8m0_exponent(__float_as_uint(am) >> 16);
          const float sc = pow2_neg(e);
          uint32_t wd[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            wd[i] = 0u;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              wd[i] |= e2m1x2(__fmul_rn(x[8 * i + 2 * k], sc), __fmul_rn(x[8 * i + 2 * k + 1], sc)) << (8 * k);
          }
          if (live) {   // 68-byte rows: 4-byte aligned
            uint32_t* dw = reinterpret_cast<uint32_t*>(qrow + 16 * b);
#pragma unroll
            for (int i = 0; i < 4; ++i) dw[i] = wd[i];
            qrow[kCodeBytes + b] = (uint8_t)(e + 127);
          }
        }
        if (live) a.w_prime[(size_t)row * a.H + h] = bf16_to_f32(a.w[(size_t)row * a.H + h]) * a.w_scale;
      }
    }
  }
  __syncwarp();
  if (failed && lane == 0 && a.status) atomicOr(a.status, kStatusLoadTimeout);
  // a role that gave up may leave the MMA warp waiting (bounded) on it; every role has
  // finished its own asynchronous work before this barrier
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_qproj(const QprojArgs& a, cudaStream_t stream) {
  if (a.R <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(qproj_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQpSmem);
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)((a.R + kQpM - 1) / kQpM) * (a.H / 2);
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  return launch_overlapped(qproj_prep_kernel, dim3(grid), dim3(kQpThreads), (size_t)kQpSmem, stream, a);
}

}  // namespace indexer
