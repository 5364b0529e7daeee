// Key publish, query prep and RoPE-table kernels of the indexer.
//
// Both the key and the query path end in the same quantiser: per 32-block an
// e8m0 scale 2^e (e the power-of-two ceiling of amax/6, amax floored at 6*2^-126)
// and e2m1 codes rounded to nearest, ties to the even code ("Module compress" page,
// fp4_quant_e8m0_inplace / to_e2m1_rne). The bf16 values fed to it are produced
// with rounding that does not depend on summation order (exact sums rounded once,
// or fixed f32 operation sequences), so the codes are reproducible bit for bit.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace indexer {

// ---------------------------------------------------------------------------- RoPE table
// table[pos][i] = (cos, sin) of angle f32(pos) * f'_i (f32 product), evaluated in f64
// and rounded to f32 ("Module compress" page, yarn_freqs_cis).
__global__ void rope_table_kernel(RopeFreqs freqs, int half, int max_pos, float2* table) {
  pdl_allow_next();
  pdl_wait();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)max_pos * half) return;
  const int pos = (int)(idx / half);
  const int i = (int)(idx % half);
  const float ang = __fmul_rn((float)pos, freqs.f[i]);
  double s, c;
  sincos((double)ang, &s, &c);
  table[idx] = make_float2(__double2float_rn(c), __double2float_rn(s));
}

cudaError_t launch_rope_table(const RopeFreqs& freqs, int half, int max_pos, float* table, cudaStream_t stream) {
  const long long n = (long long)max_pos * half;
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  return launch_overlapped(rope_table_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, freqs, half, max_pos,
                           reinterpret_cast<float2*>(table));
}

// ---------------------------------------------------------------------------- key publish
// Per key:
//  1. k_pre[o] = bf16( sum_i wk[o][i] * latent[i] ): bf16*bf16 products are exact in f32,
//     their sum is carried error-free (TwoSum) and rounded once to bf16 ("DeepSeek V4.1"
//     index-keys page, Indexer: wk bf16 Linear). Output o's products are split over TPO
//     consecutive threads (four accumulators each), whose parts are merged with TwoSum
//     across the lanes; every global read is issued before the first is used.
//  2. RMSNorm: y = bf16( (w[o] * k_pre[o]) * (1 / sqrt(sum(k_pre^2) / 128 + eps)) ) with the
//     sum of squares taken exactly in 64-bit fixed point and the rest in f64; the
//     reciprocal square root is formed once per key.
//  3. RoPE on the last rope_dim dims at the group position: interleaved pair (2i, 2i+1)
//     rotated by table entry i with the f32 sequence x0*c - x1*s, x0*s + x1*c, then bf16.
//  4. e2m1/e8m0 quantisation per 32-block (warp w owns block w); the 64 code bytes and
//     4 scale bytes go to the key's places in its 64-key page of the pool.
// Many keys (prefill): one CTA per key. Few keys (a decode step): a cluster of kPubCl
// CTAs per key, CTA r forming outputs [32r, 32r + 32) of step 1 and storing them into the
// shared memory of CTA 0 of the cluster, which runs steps 2-4; step 1 is most of a key's
// arithmetic, so a key takes four SMs' issue slots instead of one.
constexpr int kPubCl = 4;
constexpr int kPubClThreads = 256;   // 8 threads per output dim, kHeadDim / kPubCl dims per CTA

// Warms L2 with wk (CTAs 0..3 of a launch, 32 rows each) while the kernels before run.
__device__ __forceinline__ void prefetch_wk(const PublishArgs& a, int cta) {
  if (threadIdx.x == 0 && cta < 4) prefetch_l2_bulk(a.wk + (size_t)cta * 32 * a.Din, (uint32_t)(32 * a.Din * 2));
}

// The key's latent row (Din * 2 bytes: a multiple of 16 at a 16-byte aligned address).
__device__ __forceinline__ const uint16_t* key_latent(const PublishArgs& a, int key) {
  return a.latent + (size_t)key * a.Din;   // [B][G][Din]: key = b * G + j
}

// The key's slot in the page pool and its RoPE position. False for a padding entry, and for
// metadata outside the pool or the RoPE table (reported when `report`); the answer depends
// on the key alone, so every CTA of a key's cluster takes the same branch.
__device__ __forceinline__ bool key_target(const PublishArgs& a, int key, bool report, long long& slot, int& pos) {
  const int b = key / a.G, j = key % a.G;
  slot = (long long)b * a.T_cap + a.slot0 + j;
  pos = a.pos0 + j * a.pos_step;
  if (a.slots == nullptr) return true;
  slot = a.slots[key];
  pos = a.positions[key];
  if (slot < 0) return false;   // a padding entry: nothing to publish
  if (slot >= (long long)a.num_pages * kPageKeys || pos < 0 || pos >= a.max_pos) {
    if (report && threadIdx.x == 0) atomicOr(a.status, kStatusBadMeta);
    return false;
  }
  return true;
}

// Step 1 for output o by its part `part` of TPO threads (NT threads call it together: the
// latent row is staged in `lat` by all of them). Returns k_pre[o] (in every part).
template <int TPO, int NT>
__device__ __forceinline__ float linear_out(const PublishArgs& a, const uint16_t* src, int o, int part, float* lat) {
  const int tid = threadIdx.x;
  const int span = ((a.Din + 8 * TPO - 1) / (8 * TPO)) * 8;   // elements per part, a multiple of 8
  const int e_begin = part * span, e_end = min(a.Din, e_begin + span);
  const uint16_t* wrow = a.wk + (size_t)o * a.Din;
  constexpr int kPre = 128 / TPO / 8;   // 16-byte chunks fetched up front (the first 128 / TPO elements)
  uint4 wpre[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u)
    wpre[u] = (e_begin + 8 * u < e_end) ? *reinterpret_cast<const uint4*>(wrow + e_begin + 8 * u) : make_uint4(0, 0, 0, 0);
  for (int i = tid; i < a.Din; i += NT) lat[i] = bf16_to_f32(src[i]);
  __syncthreads();

  constexpr int kAcc = 4;
  float s[kAcc], c[kAcc];
#pragma unroll
  for (int k = 0; k < kAcc; ++k) s[k] = c[k] = 0.f;
  for (int e0 = e_begin; e0 < e_end; e0 += 8 * kPre) {
    uint4 w8[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u)
      w8[u] = e0 == e_begin ? wpre[u]
                            : ((e0 + 8 * u < e_end) ? *reinterpret_cast<const uint4*>(wrow + e0 + 8 * u)
                                                    : make_uint4(0, 0, 0, 0));
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const uint32_t ww[4] = {w8[u].x, w8[u].y, w8[u].z, w8[u].w};
      const int eu = e0 + 8 * u;
      if (eu < e_end) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float p0 = __fmul_rn(bf16_to_f32(ww[k] & 0xFFFFu), lat[eu + 2 * k]);
          const float p1 = __fmul_rn(bf16_to_f32(ww[k] >> 16), lat[eu + 2 * k + 1]);
          float t, e;
          two_sum(s[k], p0, t, e);
          s[k] = t;
          c[k] = __fadd_rn(c[k], e);
          two_sum(s[k], p1, t, e);
          s[k] = t;
          c[k] = __fadd_rn(c[k], e);
        }
      }
    }
  }
  float hi = s[0], lo = c[0];
#pragma unroll
  for (int k = 1; k < kAcc; ++k) {
    float t, e;
    two_sum(hi, s[k], t, e);
    hi = t;
    lo = __fadd_rn(__fadd_rn(lo, c[k]), e);
  }
#pragma unroll
  for (int off = 1; off < TPO; off <<= 1) {
    const float ohi = __shfl_xor_sync(0xffffffffu, hi, off), olo = __shfl_xor_sync(0xffffffffu, lo, off);
    float t, e;
    two_sum(hi, ohi, t, e);
    hi = t;
    lo = __fadd_rn(__fadd_rn(lo, olo), e);
  }
  float t, e;
  two_sum(hi, lo, t, e);   // normalise: |e| <= ulp(t) / 2
  return bf16_to_f32(f32pair_to_bf16_rne(t, e));
}

// y = bf16( (w x) * (1 / sqrt(ms + eps)) ) evaluated in f64 as the RMSNorm reading states it,
// ms = sum(k_pre^2) / 128 summed in f64 (exact when the values lie within 2^30 of each other
// in magnitude). Slow on this part (f64 is a narrow unit): taken only where the f32 route
// below cannot vouch for its rounding.
__device__ __noinline__ float rmsnorm_f64(const float* kx, float wx, float eps) {
  double ss = 0.0;
  for (int i = 0; i < kHeadDim; ++i) ss += (double)kx[i] * (double)kx[i];
  const double r = 1.0 / sqrt(ss / (double)kHeadDim + (double)eps);
  return bf16_to_f32(f64_to_bf16_rne((double)wx * r));
}

// (hi, lo) <- (a_hi, a_lo) + (b_hi, b_lo), unnormalised: the high parts exactly, the low
// parts with two roundings.
__device__ __forceinline__ void pair_add(float& hi, float& lo, float bhi, float blo) {
  float t, e;
  two_sum(hi, bhi, t, e);
  hi = t;
  lo = __fadd_rn(__fadd_rn(lo, blo), e);
}

// Steps 2-4 by the key's 128 threads (tid = output dim; named barrier 1). kx: the key's
// 128 k_pre values in shared memory.
__device__ __forceinline__ void finish_key(const PublishArgs& a, long long slot, const float* kx,
                                           uint32_t knorm_bits, float2 cs) {
  __shared__ float wsum[2][4];
  __shared__ int wfast[4];
  __shared__ float kv[kHeadDim];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rstart = kHeadDim - a.rope_dim;
  const float x = kx[tid];

  // 2. RMSNorm. The result must be bf16 of the f64 evaluation (rmsnorm_f64). The f32 route
  //    carries every quantity as an unevaluated pair hi + lo:
  //    - x^2 is exact in f32 when every nonzero |x| lies in [2^-40, 2^56); the 128 squares
  //      are summed with TwoSum (relative error below 2^-42),
  //    - v = ms + eps; r = 1 / sqrt(v) from the f32 estimate r0 and one correction
  //      r0 * (1 + d/2 + 3d^2/8), d = 1 - v r0^2 formed from exact products,
  //    - P = (w x) * r with an exact product of the high part,
  //    so P is within 2^-41 |P| of the exact value and the f64 evaluation within 2^-50 of it.
  //    Where P lies more than 2^-38 |P| from the bf16 rounding midpoint next to it, both round
  //    alike; otherwise (about 2^-29 of the values) and outside those ranges the f64 path runs.
  const uint32_t xb = __float_as_uint(x) >> 16;   // x is a bf16 value
  const uint32_t ef = (xb >> 7) & 0xFFu;
  const bool in_range = (xb & 0x7FFFu) == 0 || (ef >= 127 - 40 && ef < 127 + 56);
  float sh = __fmul_rn(x, x), sl = 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    pair_add(sh, sl, __shfl_xor_sync(0xffffffffu, sh, off), __shfl_xor_sync(0xffffffffu, sl, off));
  const bool warp_fast = __all_sync(0xffffffffu, in_range);
  if (lane == 0) {
    wsum[0][warp] = sh;
    wsum[1][warp] = sl;
    wfast[warp] = warp_fast;
  }
  const float wx = __fmul_rn(bf16_to_f32(knorm_bits), x);   // exact (bf16 * bf16)
  named_bar_sync(1, kHeadDim);
  bool slow = !(wfast[0] && wfast[1] && wfast[2] && wfast[3]);
  float y = 0.f;
  if (!slow) {
    float mh = wsum[0][0], ml = wsum[1][0];
    pair_add(mh, ml, wsum[0][1], wsum[1][1]);
    float nh = wsum[0][2], nl = wsum[1][2];
    pair_add(nh, nl, wsum[0][3], wsum[1][3]);
    pair_add(mh, ml, nh, nl);
    mh = __fmul_rn(mh, 1.f / kHeadDim);   // exact: a power of two, and ms >= 2^-87 or 0
    ml = __fmul_rn(ml, 1.f / kHeadDim);
    float vh, vl;
    two_sum(mh, a.eps, vh, vl);
    vl = __fadd_rn(vl, ml);
    {
      float t, e;
      two_sum(vh, vl, t, e);
      vh = t;
      vl = e;
    }
    slow = !(vh >= 0x1p-100f && vh < 0x1p100f);
    if (!slow && wx == 0.f) {
      y = wx;   // (w x) * r of a signed zero, r finite
    } else if (!slow) {
      const float awx = fabsf(wx);
      slow = !(awx >= 0x1p-80f && awx < 0x1p100f);
      const float r0 = rsqrtf(vh);
      const float p = __fmul_rn(r0, r0), pe = __fmaf_rn(r0, r0, -p);   // r0^2 = p + pe
      const float q = __fmul_rn(vh, p), qe = __fmaf_rn(vh, p, -q);     // vh p = q + qe
      const float d = __fsub_rn(__fsub_rn(1.f, q), __fadd_rn(qe, __fmaf_rn(vh, pe, __fmul_rn(vl, p))));
      const float rl = __fmul_rn(r0, __fmaf_rn(0.375f, __fmul_rn(d, d), __fmul_rn(0.5f, d)));
      const float ph = __fmul_rn(wx, r0);
      const float pl = __fmaf_rn(wx, rl, __fmaf_rn(wx, r0, -ph));
      float Ph, Pl;
      two_sum(ph, pl, Ph, Pl);
      const float aP = fabsf(Ph);
      const float mid = __uint_as_float((__float_as_uint(Ph) & 0xFFFF0000u) | 0x8000u);
      const float dist = __fadd_rn(__fsub_rn(Ph, mid), Pl);   // (Ph - mid is exact)
      slow = slow || !(aP >= 0x1p-90f && aP < 0x1p120f) || fabsf(dist) <= __fmul_rn(aP, 0x1p-38f);
      y = bf16_to_f32(f32pair_to_bf16_rne(Ph, Pl));
    }
  }
  if (slow) y = rmsnorm_f64(kx, wx, a.eps);

  // 3. RoPE
  kv[tid] = y;
  named_bar_sync(1, kHeadDim);
  if (tid >= rstart) {
    const int pair = (tid - rstart) >> 1;
    const float x0 = kv[rstart + 2 * pair], x1 = kv[rstart + 2 * pair + 1];
    const float r0 = ((tid - rstart) & 1) == 0 ? __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y))
                                              : __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
    y = bf16_to_f32(f32_to_bf16_rne(r0));
  }

  // 4. quantise: MXFP4 -- warp w holds block w, one value per lane; FP8 -- one block of
  //    128 values (amax over the four warps), one e4m3 byte per value
  uint32_t amax = (__float_as_uint(y) >> 16) & 0x7FFFu;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const int m = (int)(slot % kPageKeys);
  if (a.fp8) {
    __shared__ uint32_t wmax[4];
    if (lane == 0) wmax[warp] = amax;
    named_bar_sync(1, kHeadDim);
    const uint32_t am = max(max(wmax[0], wmax[1]), max(wmax[2], wmax[3]));
    const int e = fp8_exponent(am);
    const float yq = __fmul_rn(y, pow2(-e));
    const float partner = __shfl_down_sync(0xffffffffu, yq, 1);
    uint8_t* page = a.k_pool + (size_t)(slot / kPageKeys) * kPageBytesFp8;
    if ((lane & 1) == 0)   // elements tid, tid + 1: two adjacent bytes of one core-matrix row
      *reinterpret_cast<uint16_t*>(page + page_code_offset_fp8(m, tid)) = (uint16_t)e4m3x2(yq, partner);
    if (tid == 0) *reinterpret_cast<float*>(page + page_scale_offset_fp8(m)) = pow2(e);
    return;
  }
  const int e = e8m0_exponent(amax);
  const float yq = __fmul_rn(y, pow2_neg(e));
  const float partner = __shfl_down_sync(0xffffffffu, yq, 1);
  uint8_t* page = a.k_pool + (size_t)(slot / kPageKeys) * kPageBytes;
  if ((lane & 1) == 0) page[page_code_offset(m, (warp * 32 + lane) >> 1)] = (uint8_t)e2m1x2(yq, partner);
  if (lane == 0) page[page_scale_offset(m) + warp] = (uint8_t)(e + 127);
}

// The RoPE table entry and norm weight of output dim tid (< kHeadDim) at position pos.
__device__ __forceinline__ void key_tail_inputs(const PublishArgs& a, int pos, int tid, uint32_t& knorm_bits,
                                                float2& cs) {
  const int rstart = kHeadDim - a.rope_dim;
  knorm_bits = a.knorm[tid];
  cs = make_float2(1.f, 0.f);
  if (tid >= rstart) cs = reinterpret_cast<const float2*>(a.rope_cs)[(size_t)pos * (a.rope_dim / 2) + ((tid - rstart) >> 1)];
}

// The whole publish of key `key` by one CTA of kHeadDim * TPO threads.
template <int TPO>
__device__ __forceinline__ void publish_key(const PublishArgs& a, int key) {
  __shared__ float lat[1024];
  __shared__ float kx[kHeadDim];
  long long slot;
  int pos;
  if (!key_target(a, key, true, slot, pos)) return;
  const int tid = threadIdx.x;
  uint32_t knorm_bits = 0;
  float2 cs = make_float2(1.f, 0.f);
  if (tid < kHeadDim) key_tail_inputs(a, pos, tid, knorm_bits, cs);
  const float v = linear_out<TPO, kHeadDim * TPO>(a, key_latent(a, key), tid / TPO, tid % TPO, lat);
  if (tid % TPO == 0) kx[tid / TPO] = v;
  __syncthreads();
  if (tid >= kHeadDim) return;   // one thread per output dimension from here on
  finish_key(a, slot, kx, knorm_bits, cs);
}

// The publish of key `key` by CTA `rank` of its cluster (kPubClThreads threads).
__device__ __forceinline__ void publish_key_cluster(const PublishArgs& a, int key, int rank) {
  __shared__ float lat[1024];
  __shared__ float kx[kHeadDim];   // filled in CTA 0 by the whole cluster
  long long slot;
  int pos;
  if (!key_target(a, key, rank == 0, slot, pos)) return;   // the whole cluster leaves together
  cluster_arrive_relaxed();   // (CTA 0 must be running before its shared memory is written)
  const int tid = threadIdx.x;
  uint32_t knorm_bits = 0;
  float2 cs = make_float2(1.f, 0.f);
  if (rank == 0 && tid < kHeadDim) key_tail_inputs(a, pos, tid, knorm_bits, cs);
  constexpr int TPO = kPubClThreads / (kHeadDim / kPubCl);
  const int o = rank * (kHeadDim / kPubCl) + tid / TPO;
  const float v = linear_out<TPO, kPubClThreads>(a, key_latent(a, key), o, tid % TPO, lat);
  cluster_wait();
  if (tid % TPO == 0) st_shared_cluster_f32(map_shared_rank(smem_u32(&kx[o]), 0), v);
  cluster_arrive_release();
  cluster_wait_acquire();   // CTA 0 now holds all 128 outputs
  if (rank != 0 || tid >= kHeadDim) return;
  finish_key(a, slot, kx, knorm_bits, cs);
}

template <int TPO>   // threads per output dimension
__global__ void __launch_bounds__(kHeadDim * TPO) publish_kernel(PublishArgs a) {
  pdl_allow_next();
  prefetch_wk(a, blockIdx.x);
  pdl_wait();
  publish_key<TPO>(a, blockIdx.x);
}

__global__ void __cluster_dims__(kPubCl, 1, 1) __launch_bounds__(kPubClThreads) publish_cluster_kernel(PublishArgs a) {
  pdl_allow_next();
  const int key = (int)blockIdx.x / kPubCl, rank = (int)blockIdx.x % kPubCl;   // 1-D clusters
  prefetch_wk(a, blockIdx.x);
  if (threadIdx.x == 0 && rank == 0) prefetch_l2_bulk(key_latent(a, key), (uint32_t)(a.Din * 2));
  pdl_wait();
  publish_key_cluster(a, key, rank);
}

// Many keys of a latent of at most 128 elements (prefill): a CTA of 128 threads publishes KPC
// keys. Thread o keeps row o of wk in registers for all of them (one CTA per key would read
// the whole 32 KB of wk from L2 for every key) and the CTA stages the keys' latents with one
// load; each key's arithmetic is publish_key<1>'s, in the same order.
template <int KPC>
__global__ void __launch_bounds__(kHeadDim) publish_multi_kernel(PublishArgs a, int n_keys) {
  constexpr int kKeysPerCta = KPC;
  __shared__ float lat[kKeysPerCta][128];
  __shared__ float kx[kHeadDim];
  pdl_allow_next();
  prefetch_wk(a, blockIdx.x);
  pdl_wait();
  const int tid = threadIdx.x;
  const int key0 = (int)blockIdx.x * kKeysPerCta;
  const int nk = min(kKeysPerCta, n_keys - key0);
  uint4 w8[16];   // row tid of wk: elements 8u .. 8u + 7 (zero past Din)
  const uint16_t* wrow = a.wk + (size_t)tid * a.Din;
#pragma unroll
  for (int u = 0; u < 16; ++u)
    w8[u] = 8 * u < a.Din ? *reinterpret_cast<const uint4*>(wrow + 8 * u) : make_uint4(0, 0, 0, 0);
  for (int i = tid; i < nk * 128; i += kHeadDim) {
    const int kk = i >> 7, e = i & 127;
    if (e < a.Din) lat[kk][e] = bf16_to_f32(key_latent(a, key0 + kk)[e]);
  }
  __syncthreads();
  if constexpr (kKeysPerCta == 2) {
    // two keys at a time: their dot products interleaved (eight independent TwoSum chains in
    // flight instead of four, each key's own arithmetic and order unchanged), then each key's
    // norm, rotation and quantiser in turn. This pays for CTAs of two keys (2048 keys: 25.3 ->
    // 23.3 us) but not for CTAs of four or eight (16384 keys: 123 -> 136-147 us), which keep
    // one key at a time
    constexpr int NQ = 2;
    for (int kk = 0; kk < nk; kk += NQ) {
      const int nq = min(NQ, nk - kk);
      long long slot[NQ];
      int pos[NQ];
      bool live[NQ];   // the same in every thread
#pragma unroll
      for (int q = 0; q < NQ; ++q) live[q] = q < nq && key_target(a, key0 + kk + q, true, slot[q], pos[q]);
      // the norm weight and rotation entries, loaded ahead of the dot products
      uint32_t knorm_bits[NQ];
      float2 cs[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        knorm_bits[q] = 0u;
        cs[q] = make_float2(1.f, 0.f);
        if (live[q]) key_tail_inputs(a, pos[q], tid, knorm_bits[q], cs[q]);
      }
      // k_pre[tid] = sum_e wk[tid][e] * latent[e]: four TwoSum-carried partial sums per key over
      // the element pairs of each 8-element chunk, combined in order (linear_out<1, 128>'s order)
      float sacc[NQ][4], cacc[NQ][4];
#pragma unroll
      for (int q = 0; q < NQ; ++q)
#pragma unroll
        for (int k = 0; k < 4; ++k) sacc[q][k] = cacc[q][k] = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        if (8 * u < a.Din) {
          const uint32_t ww[4] = {w8[u].x, w8[u].y, w8[u].z, w8[u].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float w0 = bf16_to_f32(ww[k] & 0xFFFFu), w1 = bf16_to_f32(ww[k] >> 16);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
              const float p0 = __fmul_rn(w0, lat[kk + q][8 * u + 2 * k]);   // kk + q < KPC (KPC a multiple of NQ)
              const float p1 = __fmul_rn(w1, lat[kk + q][8 * u + 2 * k + 1]);
              float t, e;
              two_sum(sacc[q][k], p0, t, e);
              sacc[q][k] = t;
              cacc[q][k] = __fadd_rn(cacc[q][k], e);
              two_sum(sacc[q][k], p1, t, e);
              sacc[q][k] = t;
              cacc[q][k] = __fadd_rn(cacc[q][k], e);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!live[q]) continue;
        float hi = sacc[q][0], lo = cacc[q][0];
#pragma unroll
        for (int k = 1; k < 4; ++k) {
          float t, e;
          two_sum(hi, sacc[q][k], t, e);
          hi = t;
          lo = __fadd_rn(__fadd_rn(lo, cacc[q][k]), e);
        }
        float t, e;
        two_sum(hi, lo, t, e);
        __syncthreads();   // the previous key's outputs have been read
        kx[tid] = bf16_to_f32(f32pair_to_bf16_rne(t, e));
        __syncthreads();
        finish_key(a, slot[q], kx, knorm_bits[q], cs[q]);
      }
    }
  } else {
    for (int kk = 0; kk < nk; ++kk) {
      long long slot;
      int pos;
      if (!key_target(a, key0 + kk, true, slot, pos)) continue;   // the same for every thread
      uint32_t knorm_bits = 0;
      float2 cs = make_float2(1.f, 0.f);
      key_tail_inputs(a, pos, tid, knorm_bits, cs);
      // k_pre[tid] = sum_e wk[tid][e] * latent[e]: four TwoSum-carried partial sums over the
      // element pairs of each 8-element chunk, combined in order (linear_out<1, 128>'s order)
      float sacc[4], cacc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) sacc[k] = cacc[k] = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        if (8 * u < a.Din) {
          const uint32_t ww[4] = {w8[u].x, w8[u].y, w8[u].z, w8[u].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float p0 = __fmul_rn(bf16_to_f32(ww[k] & 0xFFFFu), lat[kk][8 * u + 2 * k]);
            const float p1 = __fmul_rn(bf16_to_f32(ww[k] >> 16), lat[kk][8 * u + 2 * k + 1]);
            float t, e;
            two_sum(sacc[k], p0, t, e);
            sacc[k] = t;
            cacc[k] = __fadd_rn(cacc[k], e);
            two_sum(sacc[k], p1, t, e);
            sacc[k] = t;
            cacc[k] = __fadd_rn(cacc[k], e);
          }
        }
      }
      float hi = sacc[0], lo = cacc[0];
#pragma unroll
      for (int k = 1; k < 4; ++k) {
        float t, e;
        two_sum(hi, sacc[k], t, e);
        hi = t;
        lo = __fadd_rn(__fadd_rn(lo, cacc[k]), e);
      }
      float t, e;
      two_sum(hi, lo, t, e);
      __syncthreads();   // the previous key's outputs have been read
      kx[tid] = bf16_to_f32(f32pair_to_bf16_rne(t, e));
      __syncthreads();
      finish_key(a, slot, kx, knorm_bits, cs);
    }
  }
}

cudaError_t launch_publish(const PublishArgs& a, cudaStream_t stream) {
  const long long keys = (long long)a.B * a.G;
  // few keys (a decode step): a cluster of four CTAs per key; a few hundred: four threads
  // per output dimension; many keys (prefill): one, for throughput
  if (keys <= 160)
    return launch_overlapped(publish_cluster_kernel, dim3((unsigned)(keys * kPubCl)), dim3(kPubClThreads), 0, stream, a);
  if (keys < 512) return launch_overlapped(publish_kernel<4>, dim3((unsigned)keys), dim3(4 * kHeadDim), 0, stream, a);
  if (a.Din <= 128) {   // wk in registers, several keys per CTA (more for more keys)
    if (keys >= 8192)
      return launch_overlapped(publish_multi_kernel<8>, dim3((unsigned)((keys + 7) / 8)), dim3(kHeadDim), 0, stream,
                               a, (int)keys);
    if (keys >= 4096)
      return launch_overlapped(publish_multi_kernel<4>, dim3((unsigned)((keys + 3) / 4)), dim3(kHeadDim), 0, stream,
                               a, (int)keys);
    return launch_overlapped(publish_multi_kernel<2>, dim3((unsigned)((keys + 1) / 2)), dim3(kHeadDim), 0, stream, a,
                             (int)keys);
  }
  return launch_overlapped(publish_kernel<1>, dim3((unsigned)keys), dim3(kHeadDim), 0, stream, a);
}

// ---------------------------------------------------------------------------- query prep
// 16 threads per query-head vector, 8 consecutive bf16 each (one 16-byte load); RoPE
// at the row's position (start_pos + s of its sequence) with the same f32 rotation as
// the keys; the 4 threads of a
// 32-block share its amax by shuffles; each thread writes 4 code bytes, the first
// thread of a block its scale byte. w' = f32(w) * head_dim^-0.5 * H^-0.5.
// Warms L2 with the 16 query-head vectors from v0 (thread t == 0 of a 256-thread group).
__device__ __forceinline__ void prefetch_q16(const PrepArgs& a, long long v0, int t) {
  if (t == 0 && v0 < a.n_vec) {
    const long long nv = a.n_vec - v0 < 16 ? a.n_vec - v0 : 16;
    prefetch_l2_bulk(a.q + v0 * kHeadDim, (uint32_t)(nv * kHeadDim * 2));
  }
}

// Query prep of the 16 vectors from v0 by a group of 256 threads (t = 0..255).
__device__ __forceinline__ void prep_q16(const PrepArgs& a, long long v0, int t) {
  const int tid = t;
  const long long v = v0 + (tid >> 4);
  const int j = tid & 15;
  if (v >= a.n_vec) return;   // whole 16-lane groups leave together
  const int lane = tid & 31;
  const unsigned gmask = 0xFFFFu << (lane & 16);
  const int qrow = (int)(v >> a.h_shift);   // H is a power of two
  const int pos = a.rows ? a.rows[qrow].pos : a.start_pos + (a.S == 1 ? 0 : qrow % a.S);
  const uint4 raw = *reinterpret_cast<const uint4*>(a.q + v * kHeadDim + j * 8);
  float2 c[4];
  load_rope_slice(reinterpret_cast<const float2*>(a.rope_cs) + (size_t)pos * (a.rope_dim / 2), j, a.rope_dim, c);
  int e;
  if (a.fp8) {
    const uint2 codes = quant_q_slice_fp8(raw, j, c, a.rope_dim, gmask, &e);
    uint8_t* row = a.q_rows + v * kRowBytesFp8;   // 132-byte rows: 4-byte aligned only
    *reinterpret_cast<uint32_t*>(row + 8 * j) = codes.x;
    *reinterpret_cast<uint32_t*>(row + 8 * j + 4) = codes.y;
    if (j == 0) *reinterpret_cast<float*>(row + kCodeBytesFp8) = pow2(e);
  } else {
    const uint32_t word = quant_q_slice(raw, j, c, a.rope_dim, gmask, &e);
    uint8_t* row = a.q_rows + v * kRowBytes;
    *reinterpret_cast<uint32_t*>(row + 4 * j) = word;
    if ((j & 3) == 0) row[kCodeBytes + (j >> 2)] = (uint8_t)(e + 127);
  }
  if (j == 0) a.w_prime[v] = bf16_to_f32(a.w[v]) * a.w_scale;
}

__global__ void __launch_bounds__(256) prep_q_kernel(PrepArgs a) {
  pdl_allow_next();
  const long long v0 = (long long)blockIdx.x * 16;
  prefetch_q16(a, v0, threadIdx.x);
  pdl_wait();
  prep_q16(a, v0, threadIdx.x);
}

// A decode step's key publish and query prep in one launch (the two are independent):
// CTAs 0 .. kPubCl * n_keys - 1 publish the keys (a cluster per key), the others prepare
// 16 query-head vectors each (256 threads).
__global__ void __cluster_dims__(kPubCl, 1, 1) __launch_bounds__(kPubClThreads)
    publish_prep_kernel(PublishArgs pa, PrepArgs qa, int n_keys) {
  static_assert(kPubClThreads == 256, "query prep takes 16 vectors per 256 threads");
  pdl_allow_next();
  const int cta = (int)blockIdx.x;
  if (cta < n_keys * kPubCl) {   // whole clusters: n_keys * kPubCl is a multiple of the cluster size
    const int key = cta / kPubCl, rank = cta % kPubCl;
    prefetch_wk(pa, cta);
    if (threadIdx.x == 0 && rank == 0) prefetch_l2_bulk(key_latent(pa, key), (uint32_t)(pa.Din * 2));
    pdl_wait();
    publish_key_cluster(pa, key, rank);
  } else {
    const long long v0 = (long long)(cta - n_keys * kPubCl) * 16;
    prefetch_q16(qa, v0, threadIdx.x);
    pdl_wait();
    prep_q16(qa, v0, threadIdx.x);
  }
}

cudaError_t launch_publish_prep(const PublishArgs& pa, const PrepArgs& qa, cudaStream_t stream) {
  const long long keys = (long long)pa.B * pa.G;
  if (keys > 160 || qa.n_vec > 16384) {   // larger: the separate kernels
    cudaError_t e = launch_publish(pa, stream);
    return e != cudaSuccess ? e : launch_prep_q(qa, stream);
  }
  const long long prep_ctas = (qa.n_vec + 15) / 16;
  const long long blocks = keys * kPubCl + (prep_ctas + kPubCl - 1) / kPubCl * kPubCl;   // whole clusters
  return launch_overlapped(publish_prep_kernel, dim3((unsigned)blocks), dim3(kPubClThreads), 0, stream, pa, qa,
                           (int)keys);
}

// Many vectors (prefill): a CTA takes 64 vectors; each thread loads its four 16-byte slices
// straight into registers up front (the eight lanes of a vector half read 128 contiguous
// bytes), quantises them with the same per-slice arithmetic, and the CTA stages the 68-byte
// rows and w' in shared memory and writes them out as whole 16-byte chunks. Against one bulk
// copy of the CTA's 16 KB into shared memory under an mbarrier: 0.317 against 0.325 ms at
// the large prefill, 42.8 against 44.6 us at the 2048-key prefill (no barrier set-up, no
// polling, no shared-memory reads of q).
constexpr int kPrepBulkVecs = 64;

__global__ void __launch_bounds__(256) prep_q_bulk_kernel(PrepArgs a) {
  constexpr int NV = kPrepBulkVecs;
  __shared__ __align__(16) uint8_t srow[NV * kRowBytesFp8];   // MXFP4 rows use the first NV * 68 bytes
  __shared__ __align__(16) float sw[NV];
  pdl_allow_next();
  const int tid = threadIdx.x;
  const long long v0 = (long long)blockIdx.x * NV;
  const int nv = (int)(a.n_vec - v0 < NV ? a.n_vec - v0 : NV);
  pdl_wait();
  uint32_t wbits = 0u;
  if (tid < nv) wbits = a.w[v0 + tid];
  // MXFP4 lanes: 8 per vector (4 vectors a warp), the 4 lanes of a 32-block adjacent; a warp
  // takes one half of its vectors' slices (j < 8 or j >= 8), so that with the model's
  // 64-element RoPE tail a warp either rotates all its slices or none (no divergent
  // rotation). FP8 lanes: the 16 of a half-warp per vector (its scale spans the vector).
  const int lane = tid & 31, warp = tid >> 5;
  const int j = a.fp8 ? (tid & 15) : 8 * (warp & 1) + (lane & 7);
  const int g = a.fp8 ? (tid >> 4) : 4 * (warp >> 1) + (lane >> 3);   // vector within each round of 16
  const unsigned gmask = a.fp8 ? 0xFFFFu << (lane & 16) : 0xFFu << (lane & 24);
  uint4 rawv[NV / 16];
#pragma unroll
  for (int p = 0; p < NV / 16; ++p) {
    const int vi = 16 * p + g;
    rawv[p] = vi < nv ? __ldg(reinterpret_cast<const uint4*>(a.q + (v0 + vi) * kHeadDim) + j)
                      : make_uint4(0u, 0u, 0u, 0u);   // 16-byte aligned: q rows are 256 bytes
  }
  // the batch's first query row and its index in its sequence (one division per CTA; the
  // batch's rows follow it, wrapping at S)
  const int qrow0 = (int)(v0 >> a.h_shift);   // H is a power of two
  const int s0 = a.rows ? 0 : qrow0 % a.S;
  // the slice's RoPE entries, reloaded only when the position changes; with H >= NV the
  // CTA's vectors are all heads of row qrow0 (v0 is a multiple of NV and NV divides H), so
  // the position and the slice are taken once, ahead of the loop
  auto row_pos = [&](int qrow) {
    const int srow_ = s0 + (qrow - qrow0);
    return a.rows ? a.rows[qrow].pos : a.start_pos + (srow_ < a.S ? srow_ : srow_ % a.S);
  };
  const bool one_row = (1 << a.h_shift) >= NV;
  int cpos = -1;
  float2 c[4];
  if (one_row) {
    cpos = row_pos(qrow0);
    load_rope_slice(reinterpret_cast<const float2*>(a.rope_cs) + (size_t)cpos * (a.rope_dim / 2), j, a.rope_dim, c);
  }
#pragma unroll
  for (int p = 0; p < NV / 16; ++p) {
    const int vi = 16 * p + g;
    if (vi < nv) {   // the lanes of a vector agree
      if (!one_row) {
        const int pos = row_pos((int)((v0 + vi) >> a.h_shift));
        if (pos != cpos) {
          load_rope_slice(reinterpret_cast<const float2*>(a.rope_cs) + (size_t)pos * (a.rope_dim / 2), j,
                          a.rope_dim, c);
          cpos = pos;
        }
      }
      const uint4 raw = rawv[p];
      int e;
      if (a.fp8) {
        const uint2 codes = quant_q_slice_fp8(raw, j, c, a.rope_dim, gmask, &e);
        *reinterpret_cast<uint32_t*>(srow + vi * kRowBytesFp8 + 8 * j) = codes.x;   // 4-byte aligned rows
        *reinterpret_cast<uint32_t*>(srow + vi * kRowBytesFp8 + 8 * j + 4) = codes.y;
        if (j == 0) *reinterpret_cast<float*>(srow + vi * kRowBytesFp8 + kCodeBytesFp8) = pow2(e);
      } else {
        const uint32_t word = quant_q_slice(raw, j, c, a.rope_dim, gmask, &e);
        *reinterpret_cast<uint32_t*>(srow + vi * kRowBytes + 4 * j) = word;
        if ((j & 3) == 0) srow[vi * kRowBytes + kCodeBytes + (j >> 2)] = (uint8_t)(e + 127);
      }
    }
  }
  if (tid < nv) sw[tid] = bf16_to_f32(wbits) * a.w_scale;
  __syncthreads();
  const int rb = a.fp8 ? kRowBytesFp8 : kRowBytes;
  uint8_t* dst = a.q_rows + v0 * rb;   // 16-byte aligned: 64 * 68 and 64 * 132 are multiples of 16
  const int bytes = nv * rb, whole = bytes & ~15;
  for (int o = tid * 16; o < whole; o += 256 * 16)
    *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(srow + o);
  for (int o = whole + tid * 4; o < bytes; o += 256 * 4)
    *reinterpret_cast<uint32_t*>(dst + o) = *reinterpret_cast<const uint32_t*>(srow + o);
  for (int i = tid; i < nv; i += 256) a.w_prime[v0 + i] = sw[i];
}

cudaError_t launch_prep_q(const PrepArgs& a, cudaStream_t stream) {
  // few vectors (decode): one per 16-thread group, for the shortest chain; many: bulk copies
  if (a.n_vec <= 16384) {
    const long long blocks = (a.n_vec + 15) / 16;
    return launch_overlapped(prep_q_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, a);
  }
  const long long blocks = (a.n_vec + kPrepBulkVecs - 1) / kPrepBulkVecs;
  return launch_overlapped(prep_q_bulk_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, a);
}

// ---------------------------------------------------------------------------- batch plan
// A batch of n_seq sequences; sequence b owns rows q_start[b] .. q_start[b+1]-1, row s of
// it at position seq_pos[b] + s, and sees (seq_pos[b] + S_b) / ratio keys. The plan writes
// each row's metadata (position, visible keys, keys of its sequence) and the row groups
// of up to qg consecutive rows of one sequence that the score kernel's CTAs take. Every
// CTA loads the sequence table into shared memory and prefix-sums the group counts;
// thread i then describes row i and group i by binary search. A sequence whose rows or
// positions are inconsistent (rows outside [0, n_rows) or in decreasing order, a negative
// position, positions past the RoPE table, more keys than T_max) is reported in the status
// word and has no rows; rows no sequence owns see no keys.
constexpr int kPlanThreads = 1024;
constexpr int kPlanPerThread = kPlanMaxSeq / kPlanThreads;

__device__ __forceinline__ int last_le(const int* v, int n, int x) {   // largest i < n with v[i] <= x, or -1
  int lo = 0, hi = n;   // answer in [lo - 1, hi - 1]
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] <= x) lo = mid + 1;
    else hi = mid;
  }
  return lo - 1;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  __shared__ int qs[kPlanMaxSeq + 1];   // first row of each sequence
  __shared__ int gs[kPlanMaxSeq + 1];   // first group of each sequence
  __shared__ uint32_t ok[kPlanMaxSeq / 32];
  __shared__ int wsum[kPlanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_allow_next();
  pdl_wait();
  // 1. per sequence: validity and group count (kPlanPerThread consecutive sequences a
  //    thread). Rows must be ascending across the whole table, else no sequence has rows.
  int q0v[kPlanPerThread], q1v[kPlanPerThread], spv[kPlanPerThread];
  bool rows_bad = false;
  for (int i = tid; i < kPlanMaxSeq / 32; i += kPlanThreads) ok[i] = 0u;
#pragma unroll
  for (int u = 0; u < kPlanPerThread; ++u) {
    const int b = tid * kPlanPerThread + u;
    q0v[u] = q1v[u] = spv[u] = 0;
    if (b < a.n_seq) {
      q0v[u] = a.q_start[b];
      q1v[u] = a.q_start[b + 1];
      spv[u] = a.seq_pos[b];
      rows_bad = rows_bad || q0v[u] < 0 || q1v[u] < q0v[u] || q1v[u] > a.n_rows;
    }
  }
  rows_bad = __syncthreads_or(rows_bad) != 0;
  int cnt[kPlanPerThread];
  int tsum = 0;
#pragma unroll
  for (int u = 0; u < kPlanPerThread; ++u) {
    const int b = tid * kPlanPerThread + u;
    cnt[u] = 0;
    if (b < a.n_seq) {
      const long long last = (long long)spv[u] + (q1v[u] - q0v[u]);   // one past the last row's position
      const bool valid = !rows_bad && spv[u] >= 0 && last <= (long long)a.max_pos &&
                         last / a.ratio <= (long long)a.T_max;
      qs[b] = q0v[u];
      if (valid) {
        atomicOr(&ok[b >> 5], 1u << (b & 31));
        cnt[u] = (q1v[u] - q0v[u] + a.qg - 1) / a.qg;
      } else if (blockIdx.x == 0) {
        atomicOr(a.status, kStatusBadMeta);
      }
    }
    tsum += cnt[u];
  }
  // 2. exclusive prefix of the group counts
  int incl = tsum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    wsum[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  int run = (warp > 0 ? wsum[warp - 1] : 0) + incl - tsum;
#pragma unroll
  for (int u = 0; u < kPlanPerThread; ++u) {
    const int b = tid * kPlanPerThread + u;
    if (b < a.n_seq) gs[b] = run;
    run += cnt[u];
  }
  if (tid == 0) {
    gs[a.n_seq] = wsum[kPlanThreads / 32 - 1];
    qs[a.n_seq] = a.n_rows;
  }
  __syncthreads();
  const int i = blockIdx.x * kPlanThreads + tid;
  // 3. row i
  if (i < a.n_rows) {
    RowInfo r = {0, 0, 0, -1};
    const int b = last_le(qs, a.n_seq, i);
    if (b >= 0 && ((ok[b >> 5] >> (b & 31)) & 1u) && i < a.q_start[b + 1]) {
      const int sp = a.seq_pos[b], S_b = a.q_start[b + 1] - qs[b];
      r.pos = sp + (i - qs[b]);
      r.T = (sp + S_b) / a.ratio;
      r.vis = min(r.T, (r.pos + 1) / a.ratio);
      r.b = b;
    }
    a.rows[i] = r;
  }
  // 4. group i
  if (i < a.n_groups) {
    RowGroup g = {0, 0, 0, 0, 0, 0, 0, 0};
    if (i < gs[a.n_seq]) {
      const int b = last_le(gs, a.n_seq, i);
      const int k = i - gs[b];
      const int sp = a.seq_pos[b], S_b = a.q_start[b + 1] - qs[b];
      g.b = b;
      g.row0 = qs[b] + k * a.qg;
      g.nq = min(a.qg, S_b - k * a.qg);
      g.pos0 = sp + k * a.qg;
      g.T = (sp + S_b) / a.ratio;
    }
    a.groups[i] = g;
  }
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
  const int n = a.n_rows > a.n_groups ? a.n_rows : a.n_groups;
  if (n <= 0) return cudaSuccess;
  return launch_overlapped(plan_kernel, dim3((unsigned)((n + kPlanThreads - 1) / kPlanThreads)), dim3(kPlanThreads),
                           0, stream, a);
}

}  // namespace indexer
