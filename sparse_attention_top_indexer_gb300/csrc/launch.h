// Internal launchers of the indexer kernels (host side). Arguments are validated by
// the C ABI (indexer_api.cu) before any of these is called; each returns the CUDA
// error of its launch.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

struct IndexerDims;   // include/indexer.h

namespace indexer {

// Launches `kernel` in stream order. With `overlap`, by programmatic stream serialisation: the
// kernel may start while the one before it still runs, and calls pdl_wait() before touching
// global memory (see device_common.cuh); without, it starts once the kernel before it is done
// (its pdl_wait() then returns at once).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool overlap, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The overlap pays for short, latency-bound grids (a decode step: 17.9 against 18.7 us with
// no overlap anywhere). A grid of more CTAs than this runs many waves, its start-up is a
// small share of its time, and the early start measured a loss (the large prefill's key
// publish, query prep and top-k launched without it: 3.029 -> 3.017 ms a step), so such
// grids launch in plain stream order.
constexpr long long kOverlapMaxCtas = 1024;

template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  const bool overlap = (long long)grid.x * grid.y * grid.z <= kOverlapMaxCtas;
  return launch_kernel(overlap, kernel, grid, block, smem, stream, static_cast<Args&&>(args)...);
}

constexpr int kMaxRopeHalf = 64;

struct RopeFreqs {
  float f[kMaxRopeHalf];   // f'_i, f32
};

cudaError_t launch_rope_table(const RopeFreqs& freqs, int half, int max_pos, float* table, cudaStream_t stream);

// Key slots: a key cache is a pool of 64-key pages ([num_pages][4352] bytes). Slot x is
// key x % 64 of pool page x / 64. A sequence-major cache k_cache[B][T_cap / 64][4352] is
// the pool whose sequence b owns pages b * T_cap / 64 onwards, so key t of sequence b sits
// in slot b * T_cap + t.
struct PublishArgs {
  const uint16_t* latent;   // [n_keys][Din] (sequence-major: [B][G][Din])
  const uint16_t* wk;       // [128][Din]
  const uint16_t* knorm;    // [128]
  const float* rope_cs;     // [max_pos][rd/2][2]
  uint8_t* k_pool;          // [num_pages][4352]
  uint32_t* status = nullptr;   // status word (paged publish) or nullptr
  int B, G, Din, rope_dim, T_cap;
  int slot0;                // sequence-major: slot of group 0 within its sequence
  int pos0, pos_step;       // sequence-major: RoPE position of group j is pos0 + j * pos_step
  // paged publish (slots != nullptr): key i goes to slot slots[i] (< 0: skipped) at RoPE
  // position positions[i]; B = 1, G = n_keys
  const int32_t* slots = nullptr;
  const int32_t* positions = nullptr;
  int num_pages, max_pos;
  int fp8;                  // FP8 rows (132 bytes, 8448-byte pages) instead of MXFP4
  float eps;
};
cudaError_t launch_publish(const PublishArgs& a, cudaStream_t stream);

// The query projection q = bf16(qr wq_b^T) with RoPE and the MXFP4 quantiser in its epilogue
// (the query prep of a uniform batch of R = B * S rows, row r at position start_pos + r % S).
struct QprojArgs {
  const uint16_t* qr;       // [R][Kq] bf16
  const uint16_t* wq_b;     // [H * 128][Kq] bf16 (row o produces feature o = head * 128 + dim)
  const uint16_t* w;        // [R][H] bf16
  const float* rope_cs;     // [max_pos][rd/2][2]
  uint8_t* q_rows;          // [R][H][68]
  float* w_prime;           // [R][H]
  uint16_t* q_out = nullptr;     // [R][H * 128] bf16 (the projection before RoPE), or nullptr
  uint32_t* status = nullptr;
  int R, Kq, H, S, start_pos, rope_dim;
  float w_scale;
};
cudaError_t launch_qproj(const QprojArgs& a, cudaStream_t stream);

// The producers upstream of the key publish and the query prep, from one pass over the
// hidden states x: the Compressor's latent (kv and gate projections, softmax pooling of
// `ratio` tokens per dim, RMSNorm to bf16), the latent through the fp4 quantiser with e4m3
// block-16 scales (dequantised to bf16), and the head weights w = weights_proj(x) (bf16).
struct CompressArgs {
  const uint16_t* x;        // [R][dim] bf16, R = B * S rows, S a multiple of ratio
  const uint16_t* wkv;      // [128][dim] bf16
  const uint16_t* wgate;    // [128][dim] bf16
  const uint16_t* norm_w;   // [128] bf16
  const uint16_t* wproj;    // [H][dim] bf16
  uint16_t* latent;         // [R / ratio][128] bf16
  uint16_t* latent_q = nullptr;   // [R / ratio][128] bf16 or nullptr
  uint16_t* w_out;          // [R][H] bf16
  uint32_t* status = nullptr;
  int R, dim, H, ratio;
  float eps;
};
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t stream);

// Per-row metadata of a batch of sequences with their own start positions and query-row
// counts, built on the device by the plan kernel.
struct alignas(16) RowInfo {
  int pos;   // RoPE position of the row (start_pos_b + s)
  int vis;   // keys it may see: min(T_b, (pos + 1) / ratio)
  int T;     // keys of its sequence: min(T_max, (start_pos_b + S_b) / ratio)
  int b;     // its sequence
};
// A group of up to QG consecutive rows of one sequence (one score CTA row).
struct alignas(16) RowGroup {
  int b, row0, nq, pos0;   // sequence, first row, rows, position of the first row
  int T, pad0, pad1, pad2;  // keys of the sequence
};

struct PlanArgs {
  const int32_t* seq_pos;   // [n_seq] start position of each sequence
  const int32_t* q_start;   // [n_seq + 1] first query row of each sequence
  RowInfo* rows;            // [n_rows]
  RowGroup* groups;         // [n_groups]
  uint32_t* status;
  int n_seq, n_rows, n_groups, qg, ratio, T_max, max_pos;
};
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream);
constexpr int kPlanMaxSeq = 4096;   // sequences one batch may hold

struct PrepArgs {
  const uint16_t* q;        // [rows][H][128]
  const uint16_t* w;        // [rows][H]
  const float* rope_cs;
  uint8_t* q_rows;          // [rows][H][68]
  float* w_prime;           // [rows][H]
  const RowInfo* rows = nullptr;   // per-row positions, or nullptr: row r is at start_pos + r % S
  uint32_t* status = nullptr;      // status word for a bounded wait that ran out, or nullptr
  long long n_vec;          // rows * H
  int S, H, rope_dim, start_pos;
  int h_shift;              // log2(H)
  int fp8;                  // FP8 rows ([rows][H][132]) instead of MXFP4 ([rows][H][68])
  float w_scale;            // head_dim^-0.5 * H^-0.5
};
cudaError_t launch_prep_q(const PrepArgs& a, cudaStream_t stream);
// A decode step's key publish and query prep in one launch (few keys and vectors), else
// the two launches in order.
cudaError_t launch_publish_prep(const PublishArgs& pa, const PrepArgs& qa, cudaStream_t stream);

struct ScoreArgs {
  const uint8_t* q_rows;    // [rows][H][68]
  const float* w_prime;     // [rows][H]
  const uint8_t* k_pool;    // [num_pages][4352]
  const int32_t* block_table = nullptr;   // [B][bt_stride] pool page of each logical page, or nullptr:
                                // sequence b owns pages b * pages_per_seq onwards
  int bt_stride, num_pages, pages_per_seq;
  const RowGroup* groups = nullptr;   // row groups of a batch with per-sequence positions, or nullptr:
                            // B sequences of S rows at start_pos
  float* scores;            // [rows][ld]
  int ld;
  const int32_t* cand = nullptr;   // [rows][cbk] or nullptr
  uint32_t* status;
  uint32_t* sched = nullptr;        // two words, zero between launches: the several-row kernel's
                                    // group counter and its count of finished CTAs
  int B, S, H, T, start_pos, ratio, cbk, cbs;   // with groups: T = T_max, S unused
  int n_groups;             // with groups
  int fill_masked;          // write -inf over key tiles no row of the group can see
  int sparse_pages;         // one query row per group: score only the pages of its kept
                            // blocks (cand); keys outside them are not written
  int tiles_per_cta;        // set by the launcher
  int fp8;                  // FP8 key and query rows (132 bytes, 8448-byte pages) instead of MXFP4
  // tests of the bounded waits (several-row kernel only): the waits' limit in ns (0: one
  // second), and a producer role that is held back so that every other role's wait runs out
  unsigned long long wait_ns = 0;
  int hold_producer = 0;
};
cudaError_t launch_scores(const ScoreArgs& a, cudaStream_t stream);
// Query rows per score CTA (QG) for n_heads H: 1 for single rows (decode), else 128 / H.
int score_group_rows(int H, bool single);

struct TopkArgs {
  const float* scores;      // [rows][ld]
  int32_t* out;             // [rows][topk]
  const int32_t* cand = nullptr;     // [rows][cbk] or nullptr
  const RowInfo* rinfo = nullptr;    // per-row vis / T, or nullptr (uniform S, T, start_pos)
  int rows, S, T, ld, start_pos, ratio, topk, offset, cbk, cbs;
  int sparse;               // consider only the positions of the kept blocks (cand), cbk * cbs <= 8192
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream);

struct CandArgs {
  const float* scores;      // [rows][ld]
  int32_t* blocks;          // [rows][cbk]
  const RowInfo* rinfo = nullptr;    // per-row vis / T, or nullptr
  int rows, S, T, ld, start_pos, ratio, cbk, cbs;
};
cudaError_t launch_candidates(const CandArgs& a, cudaStream_t stream);
// Candidate blocks and top-k of the same unfiltered rows in one launch (c and a describe the
// same rows); for level one with few rows.
cudaError_t launch_cand_topk(const CandArgs& c, const TopkArgs& a, cudaStream_t stream);

// Row-major key rows <-> 64-key pages (both directions use the same sizes).
struct LayoutArgs {
  const uint8_t* rows_in = nullptr;    // [n_seq][ld_rows][row bytes] (to pages)
  uint8_t* pages = nullptr;            // [n_seq][T_cap / 64][page bytes] (to pages)
  const uint8_t* pages_in = nullptr;   // (to rows)
  uint8_t* rows_out = nullptr;         // (to rows)
  int n_seq, n_keys, ld_rows, T_cap;
  int fp8;
};
cudaError_t launch_layout(const LayoutArgs& a, bool to_pages, cudaStream_t stream);

// Sets the thread-local message returned by indexer_last_error(); returns code.
int set_last_error(int code, const char* msg);

// Every argument check of indexer_forward (sets the error message and returns its code, or
// INDEXER_OK); enqueues nothing. dims is an IndexerDims of include/indexer.h.
int check_forward_args(const ::IndexerDims* dims, const uint16_t* q, const uint16_t* w, int B, int S,
                       int start_pos, const float* rope_cs, int max_pos, const uint8_t* k_cache, int T_cap,
                       const int32_t* cand_in, const int32_t* cand_out, const int32_t* topk_out,
                       const float* scores_out, const void* ws, size_t ws_bytes);

// Largest T the top-k kernel accepts (keys held in shared memory).
constexpr int kTopkMaxT = 32768;
constexpr int kCandMaxBlocks = 8192;

}  // namespace indexer
