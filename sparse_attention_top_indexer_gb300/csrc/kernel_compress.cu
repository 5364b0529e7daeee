// The producers upstream of the indexer, fused over one pass of the hidden states x:
//   * the Compressor's latent ("Module compress" page, compressor: softmax pooling of ratio
//     tokens into one latent, a plain projection at ratio 1, f32 until its RMSNorm casts to
//     bf16; attention.py patch page: kv_score = hidden_states @ fused_wkv_wgate^T in f32):
//     kv = x Wkv^T and score = x Wgate^T per token, per latent dim the softmax over the
//     group's ratio tokens of score weighting kv, then RMSNorm with its weight, to bf16;
//   * the latent through the fp4 quantiser with e4m3 scales ("Module compress" page,
//     fp4_quant_e4m3_inplace, LATENT_BLOCK: blocks of 16, amax floored at 6 * 2^-9, scale
//     amax / 6 rounded through e4m3, e2m1 values, dequantised back to bf16);
//   * the head weights w = weights_proj(x) ("DeepSeek V4.1" index-keys page, a bf16 Linear
//     dim -> n_heads), rounded once to bf16.
//
// One persistent CTA per SM takes tiles of 128 token rows:
//   * warp 0 (producer): per K-chunk of 64, tensor-map copies (128-byte swizzle) of x (A,
//     128 x 64), Wkv and Wgate (B1, 256 x 64: the two 128-row boxes side by side) and
//     weights_proj (B2, NP2 x 64, rows past H zero-filled) into a three-stage ring;
//   * warp 1 (MMA): per chunk four tcgen05.mma.kind::f16 of N 256 into the kv|gate
//     accumulator and four of N NP2 into the weights accumulator (f32, tensor memory);
//   * warps 2-5 (epilogue): thread m owns token row m0 + m (tensor-memory lane m). The
//     weights are rounded to bf16 and stored; the kv|gate columns are pooled across the
//     ratio lanes of each group with warp shuffles (groups never straddle a warp: ratio
//     divides 32), every lane of a group ends with the whole pooled vector, normalises it
//     and writes its 128 / ratio dims of the latent and of the quantised latent.
// Every mbarrier wait is bounded; a role that gives up reports through the status word.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"
#include "tma_common.cuh"

namespace indexer {

namespace {

constexpr int kCmM = 128;                      // token rows per tile
constexpr int kCmD = 128;                      // latent width (kv and gate: 128 features each)
constexpr int kCmStages = 3;
constexpr int kCmAStage = kCmM * kTmaK * 2;    // 16 KB
constexpr int kCmB1Stage = 2 * kCmD * kTmaK * 2;   // 32 KB
constexpr int kCmThreads = 32 + 32 + 128;
constexpr int kCmNBar = 2 * kCmStages + 2;     // full, empty per stage; accumulator full, empty

__host__ __device__ constexpr int cm_np2(int H) { return H < 16 ? 16 : H; }
__host__ __device__ constexpr int cm_stage_bytes(int NP2) { return kCmAStage + kCmB1Stage + NP2 * kTmaK * 2; }
__host__ __device__ constexpr int cm_smem(int NP2) { return 1024 + kCmStages * cm_stage_bytes(NP2) + kCmNBar * 8 + 16; }

struct CompressParams {
  CUtensorMap map_x;      // x: [R][dim], boxes 64 x 128
  CUtensorMap map_kv;     // Wkv: [128][dim], boxes 64 x 128
  CUtensorMap map_gate;   // Wgate: [128][dim], boxes 64 x 128
  CUtensorMap map_proj;   // weights_proj: [H][dim], boxes 64 x NP2 (rows past H read as zero)
  CompressArgs a;
};

// The value of a 4-bit e2m1 code (sign in bit 3): magnitude codes 0, 1 are 0 and 0.5; from
// 2 on, exponent (code >> 1) - 1 and one mantissa bit (code & 1): 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t mc = code & 7u;
  const float v = mc >= 2u ? __uint_as_float(((126u + (mc >> 1)) << 23) | ((mc & 1u) << 22)) : 0.5f * (float)mc;
  return (code & 8u) ? -v : v;
}

// The nearest e4m3 value (ties to the even code, saturating at 448) of a non-negative f32.
__device__ __forceinline__ float e4m3_round_f32(float y) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %1; cvt.u32.u16 %0, t; }" : "=r"(r) : "f"(y));
  uint32_t h;   // back to f32 through f16x2 (e4m3 values are exact in f16)
  asm("{ .reg .b16 t; .reg .b32 u; mov.b16 t, %1; cvt.rn.f16x2.e4m3x2 u, t; mov.b32 %0, u; }" : "=r"(h)
      : "h"((unsigned short)(r & 0xFFFFu)));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// Stores SLICE bf16 values (SLICE / 2 packed words) at dst: 16-byte stores, or one 8-byte
// store for a slice of 4 (dst is aligned to the slice's size).
template <int SLICE>
__device__ __forceinline__ void store_slice(uint16_t* dst, const uint32_t (&v)[SLICE / 2]) {
  if constexpr (SLICE >= 8) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < SLICE / 8; ++i) d[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    *reinterpret_cast<uint2*>(dst) = make_uint2(v[0], v[1]);
  }
}

template <int RATIO>
__global__ void __launch_bounds__(kCmThreads, 1) compress_kernel(const __grid_constant__ CompressParams prm) {
  const CompressArgs& a = prm.a;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_allow_next();
  const int NP2 = cm_np2(a.H);
  const int stage_bytes = cm_stage_bytes(NP2);
  const uint32_t stg0 = smem_u32(smem);
  const uint32_t bar0 = stg0 + kCmStages * stage_bytes;
  uint32_t* info = reinterpret_cast<uint32_t*>(smem + kCmStages * stage_bytes + kCmNBar * 8);
  auto bar_full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (uint32_t)(kCmStages + s); };
  const uint32_t bar_accfull = bar0 + 8u * (uint32_t)(2 * kCmStages);
  const uint32_t bar_accempty = bar_accfull + 8u;
  if (warp == 0) {
    if (lane < kCmNBar) mbar_init(bar0 + 8u * (uint32_t)lane, lane == 2 * kCmStages + 1 ? 128u : 1u);
    fence_mbar_init();
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&info[0]), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = info[0];
  const int n_tiles = (a.R + kCmM - 1) / kCmM;
  const int kchunks = a.dim / kTmaK;
  bool failed = false;
  pdl_wait();   // x and the weights may come from the kernels before

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t g = 0;
    for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
      const int m0 = t * kCmM;
      for (int c = 0; c < kchunks; ++c, ++g) {
        const int st = (int)(g % kCmStages);
        if (g >= (uint32_t)kCmStages && !warp_wait_bounded(bar_empty(st), ((g / kCmStages) - 1) & 1u)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          const uint32_t sa = stg0 + (uint32_t)(st * stage_bytes);
          mbar_arrive_expect_tx(bar_full(st), (uint32_t)stage_bytes);
          tma_load_2d(sa, &prm.map_x, c * kTmaK, m0, bar_full(st));
          tma_load_2d(sa + kCmAStage, &prm.map_kv, c * kTmaK, 0, bar_full(st));
          tma_load_2d(sa + kCmAStage + kCmB1Stage / 2, &prm.map_gate, c * kTmaK, 0, bar_full(st));
          tma_load_2d(sa + kCmAStage + kCmB1Stage, &prm.map_proj, c * kTmaK, 0, bar_full(st));
        }
        __syncwarp();
      }
    }
    if (lane == 0)   // no copy stays in flight past the final barrier
      for (uint32_t d = g > (uint32_t)kCmStages ? g - kCmStages : 0u; d < g; ++d)
        mbar_wait(bar_full((int)(d % kCmStages)), (d / kCmStages) & 1u);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA warp
    const uint32_t idesc1 = idesc_bf16(kCmM, 2 * kCmD), idesc2 = idesc_bf16(kCmM, NP2);
    uint32_t g = 0;
    int ti = 0;
    for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++ti) {
      // the epilogue has read the previous tile's accumulators
      if (ti >= 1 && !warp_wait_bounded(bar_accempty, (uint32_t)(ti - 1) & 1u)) {
        failed = true;
        break;
      }
      tc_fence_after();
      for (int c = 0; c < kchunks; ++c, ++g) {
        const int st = (int)(g % kCmStages);
        if (!warp_wait_bounded(bar_full(st), (g / kCmStages) & 1u)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sa = stg0 + (uint32_t)(st * stage_bytes), sb1 = sa + kCmAStage, sb2 = sb1 + kCmB1Stage;
#pragma unroll
          for (int kk = 0; kk < kTmaK / 16; ++kk) {
            const uint32_t acc = (c | kk) != 0 ? 1u : 0u;
            mma_bf16(tmem, smem_desc_sw128(sa + 32 * kk), smem_desc_sw128(sb1 + 32 * kk), idesc1, acc);
            mma_bf16(tmem + (uint32_t)(2 * kCmD), smem_desc_sw128(sa + 32 * kk), smem_desc_sw128(sb2 + 32 * kk),
                     idesc2, acc);
          }
          tc_commit(bar_empty(st));
          if (c == kchunks - 1) tc_commit(bar_accfull);
        }
        __syncwarp();
      }
    }
    if (g > 0) mbar_wait(bar_empty((int)((g - 1) % kCmStages)), ((g - 1) / kCmStages) & 1u);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int m = quad * 32 + lane;
    const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);
    constexpr int SLICE = kCmD / RATIO;        // latent dims this lane writes
    constexpr int BL = SLICE < 16 ? SLICE : 16;   // its part of a 16-block of the quantiser
    const int j = lane % RATIO;                // this lane's place in its group
    int ti = 0;
    for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++ti) {
      const int row = t * kCmM + m;
      const bool live = row < a.R;
      if (!warp_wait_bounded(bar_accfull, (uint32_t)ti & 1u)) {
        failed = true;
        break;
      }
      tc_fence_after();
      // weights_proj: bf16 of the f32 accumulation
      for (int b = 0; b < NP2; b += 32) {
        float v[32];
        tmem_ld32(tq + (uint32_t)(2 * kCmD + b), v);
        if (live) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(a.w_out + (size_t)row * a.H + b);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (b + 2 * i < a.H) dst[i] = bf16x2_rne(v[2 * i], v[2 * i + 1]);
        }
      }
      // kv | gate: softmax pooling over the group's lanes, 32 dims at a time; every lane gets
      // every pooled value (for the norm) and keeps its own slice
      float ps[SLICE];
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < kCmD / 32; ++c) {
        float kv[32], gt[32];
        tmem_ld32(tq + (uint32_t)(32 * c), kv);
        tmem_ld32(tq + (uint32_t)(kCmD + 32 * c), gt);
        if (c == kCmD / 32 - 1) {
          tc_fence_before();
          mbar_arrive(bar_accempty);   // the accumulators may take the next tile
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float mx = gt[i];
#pragma unroll
          for (int o = 1; o < RATIO; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const float e = expf(gt[i] - mx);
          float se = e, sn = e * kv[i];
#pragma unroll
          for (int o = 1; o < RATIO; o <<= 1) {
            se += __shfl_xor_sync(0xffffffffu, se, o);
            sn += __shfl_xor_sync(0xffffffffu, sn, o);
          }
          const float pv = sn / se;
          ss = fmaf(pv, pv, ss);
          const int d = 32 * c + i;
          if (d / SLICE == j) ps[d % SLICE] = pv;
        }
      }
      const float r = 1.0f / sqrtf(ss / (float)kCmD + a.eps);
      const int grp = row / RATIO;
      const int lo = j * SLICE;
      // latent: bf16((w * p) * r) over this lane's slice
      uint32_t y[SLICE / 2];
#pragma unroll
      for (int d = 0; d < SLICE; d += 2)
        y[d / 2] = bf16x2_rne((bf16_to_f32(a.norm_w[lo + d]) * ps[d]) * r,
                              (bf16_to_f32(a.norm_w[lo + d + 1]) * ps[d + 1]) * r);
      if (live) store_slice<SLICE>(a.latent + (size_t)grp * kCmD + lo, y);
      if (a.latent_q != nullptr) {
        // fp4 with e4m3 scales over blocks of 16 of the bf16 latent, dequantised to bf16; a
        // block wider than the slice takes its amax across the lanes that share it
        uint32_t yq[SLICE / 2];
#pragma unroll
        for (int b0 = 0; b0 < SLICE; b0 += BL) {
          float xv[BL];
          float am = 0.f;
#pragma unroll
          for (int i = 0; i < BL / 2; ++i) {
            const uint32_t w2 = y[(b0 / 2) + i];
            xv[2 * i] = __uint_as_float(w2 << 16);
            xv[2 * i + 1] = __uint_as_float(w2 & 0xFFFF0000u);
            am = fmaxf(am, fmaxf(fabsf(xv[2 * i]), fabsf(xv[2 * i + 1])));
          }
#pragma unroll
          for (int o = 1; o < 16 / BL; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
          am = fmaxf(am, 6.0f * 0x1p-9f);
          const float s = e4m3_round_f32(__fdiv_rn(am, 6.0f));
#pragma unroll
          for (int i = 0; i < BL / 2; ++i) {
            const uint32_t c2 = e2m1x2(__fdiv_rn(xv[2 * i], s), __fdiv_rn(xv[2 * i + 1], s));
            yq[(b0 / 2) + i] = bf16x2_rne(e2m1_value(c2 & 0xFu) * s, e2m1_value(c2 >> 4) * s);
          }
        }
        if (live) store_slice<SLICE>(a.latent_q + (size_t)grp * kCmD + lo, yq);
      }
    }
  }
  __syncwarp();
  if (failed && lane == 0 && a.status) atomicOr(a.status, kStatusLoadTimeout);
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int RATIO>
cudaError_t launch_ratio(const CompressParams& p, cudaStream_t stream) {
  const int smem = cm_smem(cm_np2(p.a.H));
  cudaError_t e = cudaFuncSetAttribute(compress_kernel<RATIO>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int tiles = (p.a.R + kCmM - 1) / kCmM;
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  return launch_overlapped(compress_kernel<RATIO>, dim3(grid), dim3(kCmThreads), (size_t)smem, stream, p);
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t stream) {
  if (a.R <= 0) return cudaSuccess;
  CompressParams p{};
  p.a = a;
  const int NP2 = cm_np2(a.H);
  cudaError_t e = encode_bf16_rows(&p.map_x, a.x, a.R, a.dim, kCmM);
  if (e == cudaSuccess) e = encode_bf16_rows(&p.map_kv, a.wkv, kCmD, a.dim, kCmD);
  if (e == cudaSuccess) e = encode_bf16_rows(&p.map_gate, a.wgate, kCmD, a.dim, kCmD);
  if (e == cudaSuccess) e = encode_bf16_rows(&p.map_proj, a.wproj, a.H, a.dim, NP2);
  if (e != cudaSuccess) return e;
  switch (a.ratio) {
    case 1: return launch_ratio<1>(p, stream);
    case 2: return launch_ratio<2>(p, stream);
    case 4: return launch_ratio<4>(p, stream);
    case 8: return launch_ratio<8>(p, stream);
    case 16: return launch_ratio<16>(p, stream);
    case 32: return launch_ratio<32>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace indexer
