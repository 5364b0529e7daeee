// Query projection fused with query prep ("DeepSeek V4.1" index-keys page, Indexer.forward:
// q = wq_b(qr) unflattened to [H][128], RoPE on the last rope_dim dims at the row's
// position, fp4_act_quant): the bf16 projection runs on the 5th-generation tensor cores and
// its epilogue writes the 68-byte query rows and w' directly, so the bf16 q never goes
// through HBM.
//
// One persistent CTA per SM takes output tiles of 128 query rows x 256 features (two heads):
//   * warp 0 (producer): one thread loads each K-chunk of 64 of qr (A, 128 x 64) and wq_b
//     (B, 256 x 64) with two tensor-map copies (cp.async.bulk.tensor, 128-byte swizzle; rows
//     past R are zero-filled by the copy) into a four-stage ring;
//   * warp 1 (MMA): four tcgen05.mma.kind::f16 (bf16 x bf16 -> f32, M 128, N 256, K 16, both
//     operands K-major with the 128-byte swizzle) per stage into one of two accumulators
//     (2 x 256 tensor-memory columns); each stage is committed back to the producer and,
//     after the last chunk, the accumulator to the epilogue;
//   * warps 2-5 (epilogue): thread m owns query row m0 + m (tensor-memory lane m) and takes
//     its two heads a 32-column block at a time: the accumulator rounded to bf16 (q as the
//     Linear's bf16 output; optionally stored for parity checks), RoPE on the rope blocks
//     with the same f32 rotation as the query-prep kernels, the block's e8m0 scale and
//     e2m1 codes; then w' = w * head_dim^-0.5 * H^-0.5 for the row's two heads.
// Every wait on an mbarrier is bounded; a role that gives up reports through the status word.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"
#include "tma_common.cuh"

namespace indexer {

namespace {

constexpr int kQpM = 128;                 // query rows per tile
constexpr int kQpN = 256;                 // output features per tile (two heads)
constexpr int kQpK = 64;                  // K per stage: 128 bytes of bf16, one swizzle row
constexpr int kQpStages = 4;
constexpr int kQpAStage = kQpM * kQpK * 2;            // 16 KB
constexpr int kQpBStage = kQpN * kQpK * 2;            // 32 KB
constexpr int kQpStage = kQpAStage + kQpBStage;
constexpr int kQpThreads = 32 + 32 + 128;
constexpr int kQpNBar = 2 * kQpStages + 4;          // full, empty per stage; acc full, acc empty
constexpr int kQpSmem = 1024 + kQpStages * kQpStage + kQpNBar * 8 + 16;
static_assert(kQpAStage % 1024 == 0 && kQpStage % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");

struct QprojParams {
  CUtensorMap map_a;   // qr: [R][Kq] bf16, boxes of 64 x 128, 128-byte swizzle
  CUtensorMap map_b;   // wq_b: [H * 128][Kq] bf16, boxes of 64 x 256, 128-byte swizzle
  QprojArgs a;
};

__global__ void __launch_bounds__(kQpThreads, 1) qproj_prep_kernel(const __grid_constant__ QprojParams prm) {
  const QprojArgs& a = prm.a;
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
    if (lane < kQpNBar) {   // an accumulator is free once the 128 epilogue threads have read it
      mbar_init(bar0 + 8u * (uint32_t)lane, lane >= 2 * kQpStages + 2 ? 128u : 1u);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t g = 0;   // chunks issued
    for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
      const int m0 = (t / tiles_n) * kQpM, n0 = (t % tiles_n) * kQpN;
      for (int c = 0; c < kchunks; ++c, ++g) {
        const int st = (int)(g % kQpStages);
        // the stage's previous chunk has been read by its MMAs (whose commit completes it)
        if (g >= (uint32_t)kQpStages && !warp_wait_bounded(bar_empty(st), ((g / kQpStages) - 1) & 1u)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          const uint32_t sa = stg0 + (uint32_t)(st * kQpStage);
          mbar_arrive_expect_tx(bar_full(st), (uint32_t)kQpStage);
          tma_load_2d(sa, &prm.map_a, c * kQpK, m0, bar_full(st));
          tma_load_2d(sa + kQpAStage, &prm.map_b, c * kQpK, n0, bar_full(st));
        }
        __syncwarp();
      }
    }
    // no copy stays in flight past the final barrier: wait (bounded) for the last stages
    if (lane == 0)
      for (uint32_t d = g > (uint32_t)kQpStages ? g - kQpStages : 0u; d < g; ++d)
        mbar_wait(bar_full((int)(d % kQpStages)), (d / kQpStages) & 1u);
    __syncwarp();
  } else if (warp == 1) {
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
          for (int kk = 0; kk < kQpK / 16; ++kk)   // K 16 per MMA: 32 bytes along the swizzled row
            mma_bf16(tmem + (uint32_t)(acc * kQpN), smem_desc_sw128(sa + 32 * kk), smem_desc_sw128(sb + 32 * kk),
                     idesc, (c | kk) != 0 ? 1u : 0u);
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
      // what does not come from the accumulator is fetched before waiting for it: the row's
      // two head weights, and its RoPE table row (rope_dim * 4 bytes) into L1
      const int pos = a.start_pos + (live ? row % a.S : 0);
      const float2* cs_row = reinterpret_cast<const float2*>(a.rope_cs) + (size_t)pos * (a.rope_dim / 2);
      uint32_t wbits0 = 0u, wbits1 = 0u;
      if (live) {
        wbits0 = a.w[(size_t)row * a.H + h0];
        wbits1 = a.w[(size_t)row * a.H + h0 + 1];
        for (int o = 0; o < a.rope_dim * 4; o += 128)
          asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<const char*>(cs_row) + o));
      }
      if (!warp_wait_bounded(bar_accfull(acc), (uint32_t)(ti >> 1) & 1u)) {
        failed = true;
        break;
      }
      tc_fence_after();
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
        if (live) a.w_prime[(size_t)row * a.H + h] = bf16_to_f32(hh == 0 ? wbits0 : wbits1) * a.w_scale;
      }
    }
  }
  __syncwarp();
  if (failed && lane == 0 && a.status) atomicOr(a.status, kStatusLoadTimeout);
  // a role that gave up may leave another waiting (bounded) on it; every role has finished
  // its own asynchronous work before this barrier
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_qproj(const QprojArgs& a, cudaStream_t stream) {
  if (a.R <= 0) return cudaSuccess;
  QprojParams p{};
  p.a = a;
  cudaError_t e = encode_bf16_rows(&p.map_a, a.qr, a.R, a.Kq, kQpM);
  if (e == cudaSuccess) e = encode_bf16_rows(&p.map_b, a.wq_b, (long long)a.H * kHeadDim, a.Kq, kQpN);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(qproj_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQpSmem);
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)((a.R + kQpM - 1) / kQpM) * (a.H / 2);
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  return launch_overlapped(qproj_prep_kernel, dim3(grid), dim3(kQpThreads), (size_t)kQpSmem, stream, p);
}

}  // namespace indexer
