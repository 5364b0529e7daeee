// Device helpers shared by the indexer kernels (sm_103a): exact rounding helpers
// for the bf16 steps of the key/query path, and thin inline-PTX wrappers for
// mbarriers, bulk (TMA) copies and the tcgen05 tensor-core / tensor-memory ops.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace indexer {

constexpr int kHeadDim = 128;           // index_head_dim supported by the kernels
constexpr int kRowBytes = 68;           // 64 packed e2m1 bytes + 4 UE8M0 scale bytes
constexpr int kCodeBytes = 64;
constexpr int kFp4Block = 32;
constexpr int kPageKeys = 64;           // keys per page of the key cache (a page pool)
constexpr int kGroupBytes = 544;        // 8 keys: 512 code bytes + 32 scale bytes
constexpr int kPageBytes = kPageKeys * kRowBytes;   // 4352 = 8 groups of 544 bytes

// Byte offset, within its page, of code byte j (0..63) of key m: 8-key groups of 544
// bytes; in a group, the keys' codes in the K-major core-matrix order of the tensor cores
// (8 rows x 16 bytes per core matrix, 128 bytes between core matrices along K), then
// the keys' 4-byte scale words. Two pages side by side are one 128-row MMA operand
// (544 bytes between 8-row groups), so both formulas also hold for m in 64..127 counted
// from the first of two adjacent pages.
__host__ __device__ __forceinline__ int page_code_offset(int m, int j) {
  return (m >> 3) * kGroupBytes + (j >> 4) * 128 + (m & 7) * 16 + (j & 15);
}
// Byte offset, within its page, of the 32-bit scale word of key m (scale of block i in
// byte i).
__host__ __device__ __forceinline__ int page_scale_offset(int m) { return (m >> 3) * kGroupBytes + 512 + (m & 7) * 4; }

// FP8 rows (the FP8 indexer cache of the attention.py page: 128 fp8 values + a 4-byte
// f32 scale = 132 bytes): 128 e4m3 codes (element i in byte i), then the f32 scale, a
// power of two. FP8 pages hold 64 keys as 8 groups of 1056 bytes: the group's 1024 code
// bytes in the same core-matrix order (8 core matrices of 128 bytes along K), then its
// keys' f32 scales; two pages side by side are again one 128-row MMA operand.
constexpr int kRowBytesFp8 = 132;
constexpr int kCodeBytesFp8 = 128;
constexpr int kGroupBytesFp8 = 1056;
constexpr int kPageBytesFp8 = kPageKeys * kRowBytesFp8;   // 8448 = 8 groups of 1056 bytes
__host__ __device__ __forceinline__ int page_code_offset_fp8(int m, int j) {
  return (m >> 3) * kGroupBytesFp8 + (j >> 4) * 128 + (m & 7) * 16 + (j & 15);
}
__host__ __device__ __forceinline__ int page_scale_offset_fp8(int m) {
  return (m >> 3) * kGroupBytesFp8 + 1024 + (m & 7) * 4;
}

// Status bits OR-ed into the workspace status word by kernels whose bounded waits ran out.
constexpr uint32_t kStatusLoadTimeout = 1u;
constexpr uint32_t kStatusMmaTimeout = 2u;
// Status bit of invalid device-side metadata (a block-table entry outside the page pool, a
// slot or position out of range, inconsistent per-sequence rows): the affected keys or
// rows are skipped.
constexpr uint32_t kStatusBadMeta = 4u;
// One second: a bounded wait gives up after this long and reports through the status word.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ----------------------------------------------------------------------------- bf16 / rounding
__device__ __forceinline__ float bf16_to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }

// Round an f32 to bf16 to nearest, ties to even (finite inputs).
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b + 0x7FFFu + ((b >> 16) & 1u)) >> 16;
}

// Two f32 rounded to bf16 to nearest, ties to even, in one conversion: lo in bits 0-15,
// hi in bits 16-31 (for finite inputs the same as f32_to_bf16_rne of each).
__device__ __forceinline__ uint32_t bf16x2_rne(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// RoPE of one interleaved pair: (x0*c - x1*s, x0*s + x1*c) with f32 products and sums,
// each rounded to bf16 (returned as f32 values).
__device__ __forceinline__ void rope_pair_bf16(float& x0, float& x1, float2 cs) {
  const uint32_t r = bf16x2_rne(__fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y)),
                                __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x)));
  x0 = __uint_as_float(r << 16);
  x1 = __uint_as_float(r & 0xFFFF0000u);
}

// Round an f64 to bf16 once (no intermediate f32), to nearest with ties to even.
// bf16 keeps 7 explicit mantissa bits; below 2^-126 the spacing is fixed at 2^-133.
__device__ __forceinline__ uint32_t f64_to_bf16_rne(double x) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(x);
  const uint32_t sign = (uint32_t)(b >> 48) & 0x8000u;
  const unsigned long long a = b & 0x7FFFFFFFFFFFFFFFull;
  if (a == 0) return sign;
  const int e = (int)(a >> 52) - 1023;
  if (e >= -126) {
    const unsigned long long m = a & ((1ull << 52) - 1);
    uint32_t keep = (uint32_t)(m >> 45);
    const unsigned long long rest = m & ((1ull << 45) - 1);
    const unsigned long long half = 1ull << 44;
    int ee = e;
    if (rest > half || (rest == half && (keep & 1u))) {
      if (++keep == 128u) { keep = 0; ++ee; }
    }
    if (ee > 127) return sign | 0x7F80u;
    return sign | ((uint32_t)(ee + 127) << 7) | keep;
  }
  // bf16 subnormal range: value = n * 2^-133 with n in [0, 128]; n = 128 is the
  // smallest normal, whose bit pattern is exactly 128 as well.
  const double scaled = __longlong_as_double((long long)a) * 0x1p133;
  return sign | (uint32_t)__double2int_rn(scaled);
}

// Round (hi + lo) to bf16 correctly, where hi = fl32(hi + lo) (|lo| <= ulp(hi) / 2).
// Only when hi sits exactly on a bf16 midpoint can lo change the result.
__device__ __forceinline__ uint32_t f32pair_to_bf16_rne(float hi, float lo) {
  const uint32_t hb = __float_as_uint(hi);
  if ((hb & 0xFFFFu) == 0x8000u && lo != 0.0f) {
    const bool away = (lo > 0.0f) == (hi > 0.0f);
    return (hb >> 16) + (away ? 1u : 0u);
  }
  return f32_to_bf16_rne(hi);
}

// Error-free sum: s + e == a + b exactly (Knuth's TwoSum), no contraction.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float z = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
}

// ----------------------------------------------------------------------------- e2m1 / e8m0
// e8m0 exponent of a 32-block from its amax bit pattern (non-negative bf16): the
// smallest e with 6 * 2^e >= max(amax, 6 * 2^-126). Writing amax = (1 + m/128) * 2^E,
// 6 * 2^(E-2) = 1.5 * 2^E covers it iff m <= 64, else 6 * 2^(E-1) = 3 * 2^E does.
__device__ __forceinline__ int e8m0_exponent(uint32_t amax_bits) {
  const uint32_t a = amax_bits < 0x01C0u ? 0x01C0u : amax_bits;   // 0x01C0 = bf16 6 * 2^-126
  const int E = (int)(a >> 7) - 127;
  return E - ((a & 0x7Fu) <= 64u ? 2 : 1);
}

// 2^-e as an f32 (e in [-126, 126], so the result is a normal number).
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// FP8 rows: smallest e with 448 * 2^e >= max(amax, 448 * 2^-126), from the bf16 bits of
// amax (sign cleared). 448 = 1.75 * 2^8, so with amax = (1 + m/128) * 2^E, e = E - 8
// when 1 + m/128 <= 1.75 (m <= 96), else E - 7; 0x04E0 is the bf16 pattern of the floor.
__device__ __forceinline__ int fp8_exponent(uint32_t amax_bits) {
  const uint32_t a = amax_bits < 0x04E0u ? 0x04E0u : amax_bits;
  const int E = (int)(a >> 7) - 127;
  return E - ((a & 0x7Fu) <= 96u ? 8 : 7);
}
__device__ __forceinline__ float pow2(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Two e4m3 codes: x0 -> low byte, x1 -> high byte; round to nearest even (hardware
// conversion; the scaled values never exceed 448, so nothing saturates); the sign bits
// are forced to the signs of the inputs so that negative values rounding to zero keep it.
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; cvt.u32.u16 %0, t; }" : "=r"(r) : "f"(x1), "f"(x0));
  r |= (__float_as_uint(x0) >> 24) & 0x80u;
  r |= (__float_as_uint(x1) >> 16) & 0x8000u;
  return r;
}

// Two e2m1 codes in one byte: x0 -> low nibble, x1 -> high nibble; round to nearest
// even on the e2m1 grid (hardware conversion). The conversion keeps the sign of a
// negative value that rounds to zero (code 0x8; checked on the GPU for -0, -1e-30, -0.1
// and the tie -0.25), as the quantiser's sign rule asks.
__device__ __forceinline__ uint32_t e2m1x2(float x0, float x1) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(x1), "f"(x0));
  return r;
}

// Eight e2m1 codes in one word: byte k holds the codes of x[2k] (low nibble) and x[2k+1],
// each converted as e2m1x2 does; the four bytes are packed by the conversion's register moves.
__device__ __forceinline__ uint32_t e2m1x8(const float (&x)[8]) {
  uint32_t r;
  asm("{ .reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3}; }"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return r;
}

// max |x[k]| over eight values with three-input maxima (finite inputs; -0 counts as +0).
__device__ __forceinline__ float amax_abs8(const float (&x)[8]) {
  float a, b, c;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(a) : "f"(x[0]), "f"(x[1]), "f"(x[2]));
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(b) : "f"(x[3]), "f"(x[4]), "f"(x[5]));
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(c) : "f"(x[6]), "f"(x[7]), "f"(a));
  return fmaxf(b, c);
}

// ----------------------------------------------------------------------------- PTX: mbarrier / bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0u;
}
// ----------------------------------------------------------------------------- query prep
// RoPE table entries (cos, sin) of the 4 element pairs of slice j (0..15) of a
// 128-element head vector; pairs outside the last rope_dim elements get (1, 0), which
// the rotation below never reads.
__device__ __forceinline__ void load_rope_slice(const float2* cs_row, int j, int rope_dim, float2 (&c)[4]) {
  const int rstart = kHeadDim - rope_dim;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e0 = j * 8 + 2 * k;
    c[k] = e0 >= rstart ? cs_row[(e0 - rstart) >> 1] : make_float2(1.f, 0.f);
  }
}

// One 8-element slice j (0..15) of a 128-element query-head vector, given as 8 bf16 in
// `raw`: RoPE on the last rope_dim elements with the slice's table entries c (from
// load_rope_slice; interleaved pairs rotated with the f32 sequence x0*c - x1*s,
// x0*s + x1*c, each rounded to bf16), then e2m1 with the 32-block's e8m0 scale. Returns
// the 4 code bytes (element 2i in the low nibble of byte i) and the block's scale
// exponent in *e. The 4 threads of a 32-block (lanes 4i..4i+3 of a 16-lane half named by
// gmask) must call it together: they share the block amax.
__device__ __forceinline__ uint32_t quant_q_slice(uint4 raw, int j, const float2 (&c)[4], int rope_dim,
                                                  unsigned gmask, int* e) {
  const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = bf16_to_f32(wds[k] & 0xFFFFu);
    x[2 * k + 1] = bf16_to_f32(wds[k] >> 16);
  }
  const int rstart = kHeadDim - rope_dim;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e0 = j * 8 + 2 * k;   // even element; rstart is even so pairs never straddle
    if (e0 >= rstart) rope_pair_bf16(x[2 * k], x[2 * k + 1], c[k]);
  }
  // the largest |x| (bf16 values), as bf16 bits
  uint32_t amax = __float_as_uint(amax_abs8(x)) >> 16;
  amax = max(amax, __shfl_xor_sync(gmask, amax, 1));
  amax = max(amax, __shfl_xor_sync(gmask, amax, 2));
  const int ex = e8m0_exponent(amax);
  const float sc = pow2_neg(ex);
  float y[8];   // x * 2^-ex, exact (a power of two), two at a time
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 r = __fmul2_rn(make_float2(x[2 * k], x[2 * k + 1]), make_float2(sc, sc));
    y[2 * k] = r.x;
    y[2 * k + 1] = r.y;
  }
  *e = ex;
  return e2m1x8(y);
}

// FP8 query slice: the same RoPE as quant_q_slice, then the row's 128-value amax over the
// 16 lanes of the group, the power-of-two scale and eight e4m3 codes (returned as two
// words, element j*8 in the lowest byte); *e receives the scale exponent.
__device__ __forceinline__ uint2 quant_q_slice_fp8(uint4 raw, int j, const float2 (&c)[4], int rope_dim,
                                                   unsigned gmask, int* e) {
  const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = bf16_to_f32(wds[k] & 0xFFFFu);
    x[2 * k + 1] = bf16_to_f32(wds[k] >> 16);
  }
  const int rstart = kHeadDim - rope_dim;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e0 = j * 8 + 2 * k;
    if (e0 >= rstart) rope_pair_bf16(x[2 * k], x[2 * k + 1], c[k]);
  }
  float am = 0.f;   // the largest |x| (bf16 values), as bf16 bits
#pragma unroll
  for (int k = 0; k < 8; ++k) am = fmaxf(am, fabsf(x[k]));
  uint32_t amax = __float_as_uint(am) >> 16;
#pragma unroll
  for (int off = 1; off < 16; off <<= 1) amax = max(amax, __shfl_xor_sync(gmask, amax, off));
  const int ex = fp8_exponent(amax);
  const float sc = pow2(-ex);
  uint2 out;
  out.x = e4m3x2(__fmul_rn(x[0], sc), __fmul_rn(x[1], sc)) | (e4m3x2(__fmul_rn(x[2], sc), __fmul_rn(x[3], sc)) << 16);
  out.y = e4m3x2(__fmul_rn(x[4], sc), __fmul_rn(x[5], sc)) | (e4m3x2(__fmul_rn(x[6], sc), __fmul_rn(x[7], sc)) << 16);
  *e = ex;
  return out;
}

// ----------------------------------------------------------------------------- launch overlap
// The library's small, latency-bound grids are launched with programmatic stream
// serialisation (launch.h): such a kernel may start while the kernel before it on the stream
// is still running. pdl_allow_next() lets the next kernel start in turn; pdl_wait() blocks
// until every earlier kernel on the stream has completed and its memory is visible, and each
// kernel calls it before its first global-memory access (read or write), so only
// shared-memory set-up overlaps. Both are no-ops for a kernel launched without that
// attribute (the long grids), which starts once the kernel before it is done.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// The whole warp waits (bounded) for the phase, converged; warp-uniform result.
__device__ __forceinline__ bool warp_wait_bounded(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}
// Bulk (non-tensor TMA) copy global -> shared; dst, src and bytes multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barrier over `n` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier that also returns the AND of `v` over its `n` threads, so that every
// thread of a warpgroup takes the same branch after a bounded wait.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r) : "r"((uint32_t)v), "r"(id), "r"(n) : "memory");
  return r != 0u;
}

// ----------------------------------------------------------------------------- PTX: tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with block-32 UE8M0 scales from tensor memory,
// both operands e2m1 packed two per byte (kind::mxf4, K = 64 per instruction).
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p; }"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Instruction descriptor of kind::mxf4: A and B e2m1 (format 1, bits 7-9 / 10-12),
// both K-major, N >> 3 in bits 17-22, UE8M0 scales (bit 23), M >> 7 in bits 27-28,
// scale-factor data ids 0 (bytes 0 and 1 of each scale column), K = 64.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 7) << 27);
}

// Warms L2 with [gptr, gptr + bytes) (16-byte aligned, a multiple of 16 bytes). A hint
// only: the data is not delivered anywhere and a later write to the lines by another
// kernel keeps L2 coherent, so it may be issued before pdl_wait().
__device__ __forceinline__ void prefetch_l2_bulk(const void* gptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gptr), "r"(bytes) : "memory");
}

// ----------------------------------------------------------------------------- clusters
// Cluster-wide barrier halves (every thread of every CTA of the cluster takes part, in
// converged warps). The relaxed arrive orders nothing; the release arrive / acquire wait
// pair makes each CTA's earlier shared-memory stores (including remote ones) visible to
// the whole cluster.
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait_acquire() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// The shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_shared_cluster_f32(uint32_t caddr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(caddr), "f"(v) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both e4m3 (kind::f8f6f4, K = 32 per instruction).
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor of kind::f8f6f4: f32 accumulator (bits 4-5 = 1), A and B e4m3
// (bits 7-9 and 10-12 = 0), both K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f8(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, both bf16 (kind::f16, K = 16 per instruction).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor of kind::f16: f32 accumulator (bits 4-5 = 1), A and B bf16
// (bits 7-9 and 10-12 = 1), both K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, no swizzle, K-major: core matrices of 8 rows x 16 bytes
// (128 contiguous bytes); lbo = byte step between core matrices along K, sbo = byte step
// between 8-row groups along M/N; bits 46-48 hold the fixed value 0b001.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3,
                                           uint32_t v4, uint32_t v5, uint32_t v6, uint32_t v7) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               ::"r"(taddr), "r"(v0), "r"(v1), "r"(v2), "r"(v3), "r"(v4), "r"(v5), "r"(v6), "r"(v7)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Load 32 consecutive columns of this warp's 32 lanes and wait for them (one asm
// statement, so no use of the registers can be scheduled before the wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// A 32-column read in two steps, so that other work runs while it is in flight: the
// tcgen05.ld alone (the registers are not valid yet), then tcgen05.wait::ld, which names
// the registers as read-write operands so that no use of them moves above the wait.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld32_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Whole-accumulator reads: one tcgen05.ld of 64 or 128 columns and one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// Two f32 FMAs in one instruction (round to nearest each): (d0, d1) = (a0*b0 + c0, a1*b1 + c1),
// through the compiler's float2 builtin, so the register pairs are the allocator's choice.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  const float2 r = __ffma2_rn(make_float2(a0, a1), make_float2(b0, b1), make_float2(d0, d1));
  d0 = r.x;
  d1 = r.y;
}

}  // namespace indexer
