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
// One CTA of 128 threads per key; thread o owns output dim o.
//  1. k_pre[o] = bf16( sum_i wk[o][i] * latent[i] ): bf16*bf16 products are exact in f32,
//     their sum is carried error-free (TwoSum) in eight interleaved accumulators and
//     rounded once to bf16 ("DeepSeek V4.1" index-keys page, Indexer: wk bf16 Linear).
//     The thread's wk row is fetched 128 elements at a time with all loads issued
//     before any is used, so a 128-wide row costs one memory round trip.
//  2. RMSNorm in f64: y = bf16( (w[o] * k_pre[o]) * (1 / sqrt(sum(k_pre^2) / 128 + eps)) );
//     the reciprocal square root is formed once per key.
//  3. RoPE on the last rope_dim dims at the group position: interleaved pair (2i, 2i+1)
//     rotated by table entry i with the f32 sequence x0*c - x1*s, x0*s + x1*c, then bf16.
//  4. e2m1/e8m0 quantisation per 32-block (warp w owns block w); the 64 code bytes and
//     4 scale bytes go to the key's places in its 128-key page.
__global__ void __launch_bounds__(128) publish_kernel(PublishArgs a) {
  __shared__ float lat[1024];
  __shared__ float kv[kHeadDim];
  __shared__ double wsum[4];
  __shared__ double rinv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_allow_next();
  pdl_wait();
  const int key = blockIdx.x;
  const int b = key / a.G, j = key % a.G;
  const uint16_t* src = a.latent + ((size_t)b * a.G + j) * a.Din;
  for (int i = tid; i < a.Din; i += 128) lat[i] = bf16_to_f32(src[i]);
  __syncthreads();

  // 1. exact dot product, rounded once
  const uint16_t* wrow = a.wk + (size_t)tid * a.Din;
  constexpr int kAcc = 8;
  float s[kAcc], c[kAcc];
#pragma unroll
  for (int k = 0; k < kAcc; ++k) s[k] = c[k] = 0.f;
  for (int i0 = 0; i0 < a.Din; i0 += 128) {
    uint4 w8[16];
#pragma unroll
    for (int u = 0; u < 16; ++u)
      w8[u] = (i0 + 8 * u < a.Din) ? *reinterpret_cast<const uint4*>(wrow + i0 + 8 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const uint32_t ww[4] = {w8[u].x, w8[u].y, w8[u].z, w8[u].w};
      const int e0 = i0 + 8 * u;
      if (e0 < a.Din) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int acc = (2 * k) & (kAcc - 1), acc2 = (2 * k + 1) & (kAcc - 1);
          const float p0 = __fmul_rn(bf16_to_f32(ww[k] & 0xFFFFu), lat[e0 + 2 * k]);
          const float p1 = __fmul_rn(bf16_to_f32(ww[k] >> 16), lat[e0 + 2 * k + 1]);
          float t, e;
          two_sum(s[acc], p0, t, e);
          s[acc] = t;
          c[acc] = __fadd_rn(c[acc], e);
          two_sum(s[acc2], p1, t, e);
          s[acc2] = t;
          c[acc2] = __fadd_rn(c[acc2], e);
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
  {
    float t, e;
    two_sum(hi, lo, t, e);   // normalise: |e| <= ulp(t) / 2
    hi = t;
    lo = e;
  }
  const float x = bf16_to_f32(f32pair_to_bf16_rne(hi, lo));

  // 2. RMSNorm in f64 (the squares of bf16 values are exact; the sum is exact for any
  //    realistic dynamic range, so its order does not matter)
  double ss = (double)x * (double)x;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if (lane == 0) wsum[warp] = ss;
  __syncthreads();
  if (tid == 0) {
    const double ms = ((wsum[0] + wsum[1]) + (wsum[2] + wsum[3])) / (double)kHeadDim;
    rinv = 1.0 / sqrt(ms + (double)a.eps);
  }
  __syncthreads();
  const float wx = __fmul_rn(bf16_to_f32(a.knorm[tid]), x);   // exact (bf16 * bf16)
  float y = bf16_to_f32(f64_to_bf16_rne((double)wx * rinv));

  // 3. RoPE
  kv[tid] = y;
  __syncthreads();
  const int rstart = kHeadDim - a.rope_dim;
  if (tid >= rstart) {
    const int rel = tid - rstart;
    const int pair = rel >> 1;
    const int pos = a.pos0 + j * a.pos_step;
    const float2 cs = reinterpret_cast<const float2*>(a.rope_cs)[(size_t)pos * (a.rope_dim / 2) + pair];
    const float x0 = kv[rstart + 2 * pair], x1 = kv[rstart + 2 * pair + 1];
    const float r0 = (rel & 1) == 0 ? __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y))
                                    : __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
    y = bf16_to_f32(f32_to_bf16_rne(r0));
  }

  // 4. quantise: warp w holds block w, one value per lane
  uint32_t amax = (__float_as_uint(y) >> 16) & 0x7FFFu;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const int e = e8m0_exponent(amax);
  const float yq = __fmul_rn(y, pow2_neg(e));
  const float partner = __shfl_down_sync(0xffffffffu, yq, 1);
  const int slot = a.slot0 + j;
  const int m = slot % kPageKeys;
  uint8_t* page = a.k_cache + ((size_t)b * (a.T_cap / kPageKeys) + slot / kPageKeys) * kPageBytes;
  if ((lane & 1) == 0) page[page_code_offset(m, (warp * 32 + lane) >> 1)] = (uint8_t)e2m1x2(yq, partner);
  if (lane == 0) page[page_scale_offset(m) + warp] = (uint8_t)(e + 127);
}

cudaError_t launch_publish(const PublishArgs& a, cudaStream_t stream) {
  const long long keys = (long long)a.B * a.G;
  return launch_overlapped(publish_kernel, dim3((unsigned)keys), dim3(128), 0, stream, a);
}

// ---------------------------------------------------------------------------- query prep
// 16 threads per query-head vector, 8 consecutive bf16 each (one 16-byte load); RoPE
// at position start_pos + s with the same f32 rotation as the keys; the 4 threads of a
// 32-block share its amax by shuffles; each thread writes 4 code bytes, the first
// thread of a block its scale byte. w' = f32(w) * head_dim^-0.5 * H^-0.5.
__global__ void __launch_bounds__(256) prep_q_kernel(PrepArgs a) {
  pdl_allow_next();
  pdl_wait();
  const int tid = threadIdx.x;
  const long long v = (long long)blockIdx.x * 16 + (tid >> 4);
  const int j = tid & 15;
  if (v >= a.n_vec) return;   // whole 16-lane groups leave together
  const int lane = tid & 31;
  const unsigned gmask = 0xFFFFu << (lane & 16);
  const int s = (int)((v / a.H) % a.S);
  const int pos = a.start_pos + s;
  const uint4 raw = *reinterpret_cast<const uint4*>(a.q + v * kHeadDim + j * 8);
  float2 c[4];
  load_rope_slice(reinterpret_cast<const float2*>(a.rope_cs) + (size_t)pos * (a.rope_dim / 2), j, a.rope_dim, c);
  int e;
  const uint32_t word = quant_q_slice(raw, j, c, a.rope_dim, gmask, &e);
  uint8_t* row = a.q_rows + v * kRowBytes;
  *reinterpret_cast<uint32_t*>(row + 4 * j) = word;
  if ((j & 3) == 0) row[kCodeBytes + (j >> 2)] = (uint8_t)(e + 127);
  if (j == 0) a.w_prime[v] = bf16_to_f32(a.w[v]) * a.w_scale;
}

cudaError_t launch_prep_q(const PrepArgs& a, cudaStream_t stream) {
  const long long blocks = (a.n_vec + 15) / 16;
  return launch_overlapped(prep_q_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, a);
}

}  // namespace indexer
