// Internal launchers of the indexer kernels (host side). Arguments are validated by
// the C ABI (indexer_api.cu) before any of these is called; each returns the CUDA
// error of its launch.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace indexer {

// Launches `kernel` with programmatic stream serialisation (the kernel calls pdl_wait()
// before touching global memory; see device_common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

constexpr int kMaxRopeHalf = 64;

struct RopeFreqs {
  float f[kMaxRopeHalf];   // f'_i, f32
};

cudaError_t launch_rope_table(const RopeFreqs& freqs, int half, int max_pos, float* table, cudaStream_t stream);

struct PublishArgs {
  const uint16_t* latent;   // [B][G][Din]
  const uint16_t* wk;       // [128][Din]
  const uint16_t* knorm;    // [128]
  const float* rope_cs;     // [max_pos][rd/2][2]
  uint8_t* k_cache;         // [B][T_cap][68]
  int B, G, Din, rope_dim, T_cap;
  int slot0;                // cache slot of group 0
  int pos0, pos_step;       // RoPE position of group j: pos0 + j * pos_step
  float eps;
};
cudaError_t launch_publish(const PublishArgs& a, cudaStream_t stream);

struct PrepArgs {
  const uint16_t* q;        // [B][S][H][128]
  const uint16_t* w;        // [B][S][H]
  const float* rope_cs;
  uint8_t* q_rows;          // [B][S][H][68]
  float* w_prime;           // [B][S][H]
  long long n_vec;          // B * S * H
  int S, H, rope_dim, start_pos;
  float w_scale;            // head_dim^-0.5 * H^-0.5
};
cudaError_t launch_prep_q(const PrepArgs& a, cudaStream_t stream);

struct ScoreArgs {
  const uint8_t* q_rows;    // [B][S][H][68]
  const float* w_prime;     // [B][S][H]
  const uint8_t* k_cache;   // [B][T_cap / 128][8704] pages
  float* scores;            // [B][S][T]
  const int32_t* cand;      // [B][S][cbk] or nullptr
  uint32_t* status;
  int B, S, H, T, T_cap, start_pos, ratio, cbk, cbs;
  int fill_masked;          // write -inf over key tiles no row of the group can see
  int sparse_pages;         // one query row (S == 1): score only the pages of its kept blocks
                            // (cand); keys outside them are not written
  int tiles_per_cta;        // set by the launcher
};
cudaError_t launch_scores(const ScoreArgs& a, cudaStream_t stream);

struct TopkArgs {
  const float* scores;      // [rows][T]
  int32_t* out;             // [rows][topk]
  const int32_t* cand;      // [rows][cbk] or nullptr
  int rows, S, T, start_pos, ratio, topk, offset, cbk, cbs;
  int sparse;               // consider only the positions of the kept blocks (cand), cbk * cbs <= 8192
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream);

struct CandArgs {
  const float* scores;      // [rows][T]
  int32_t* blocks;          // [rows][cbk]
  int rows, S, T, start_pos, ratio, cbk, cbs;
};
cudaError_t launch_candidates(const CandArgs& a, cudaStream_t stream);

// Sets the thread-local message returned by indexer_last_error(); returns code.
int set_last_error(int code, const char* msg);

// Largest T the top-k kernel accepts (keys held in shared memory).
constexpr int kTopkMaxT = 32768;
constexpr int kCandMaxBlocks = 8192;

}  // namespace indexer
