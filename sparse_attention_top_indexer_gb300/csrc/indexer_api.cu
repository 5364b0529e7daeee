// C ABI of the indexer (declared in include/indexer.h): host-side validation, the
// workspace layout and kernel launches. Every entry point validates all arguments
// before it launches anything; the library holds no device memory of its own.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include <cuda_runtime.h>

#include "../../include/indexer.h"
#include "device_common.cuh"
#include "launch.h"

using namespace indexer;

namespace {

// Word of the workspace header holding the several-row score kernel's group counter (two
// words, zeroed by indexer_workspace_init and left zero by every launch).
constexpr int kSchedWord = 32;

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return INDEXER_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(INDEXER_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

// The kernels are built for sm_103a only.
int check_arch() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(INDEXER_ERR_ARCH, "device %d is sm_%d%d; the indexer kernels are built for sm_103a", dev, major, minor);
  return INDEXER_OK;
}

int check_dims(const IndexerDims* d) {
  if (!d) return fail(INDEXER_ERR_NULL, "dims is NULL");
  if (d->head_dim != 128) return fail(INDEXER_ERR_DIMS, "head_dim must be 128 (got %d)", d->head_dim);
  const int h = d->n_heads;
  if (h != 8 && h != 16 && h != 32 && h != 64 && h != 128)
    return fail(INDEXER_ERR_DIMS, "n_heads must be 8, 16, 32, 64 or 128 (got %d)", h);
  if (d->rope_dim < 2 || d->rope_dim > 128 || (d->rope_dim & 1))
    return fail(INDEXER_ERR_DIMS, "rope_dim must be even in [2, 128] (got %d)", d->rope_dim);
  if (d->ratio < 1) return fail(INDEXER_ERR_DIMS, "ratio must be >= 1 (got %d)", d->ratio);
  if (d->index_topk < 1) return fail(INDEXER_ERR_DIMS, "index_topk must be >= 1 (got %d)", d->index_topk);
  if (!(d->norm_eps >= 0.0f) || !std::isfinite(d->norm_eps))
    return fail(INDEXER_ERR_DIMS, "norm_eps must be finite and >= 0");
  if (d->key_format != INDEXER_KEY_MXFP4 && d->key_format != INDEXER_KEY_FP8)
    return fail(INDEXER_ERR_DIMS, "key_format must be INDEXER_KEY_MXFP4 or INDEXER_KEY_FP8 (got %d)", d->key_format);
  if (d->n_heads_total != 0 && (d->n_heads_total < h || d->n_heads_total > (1 << 16)))
    return fail(INDEXER_ERR_DIMS, "n_heads_total must be 0 or in [n_heads, 65536] (got %d)", d->n_heads_total);
  return INDEXER_OK;
}

// softmax_scale * index_n_heads^-0.5 with softmax_scale = index_head_dim^-0.5 ("DeepSeek V4.1"
// index-keys page, Indexer.__init__ and the weights line of Indexer.forward); a head shard
// keeps the model's head count.
float head_weight_scale(const IndexerDims* d) {
  const int h = d->n_heads_total ? d->n_heads_total : d->n_heads;
  return (float)(1.0 / std::sqrt((double)d->head_dim * (double)h));
}

// Bytes of one quantised row / one 64-key page in the dims' key format.
size_t row_bytes(const IndexerDims* d) {
  return d->key_format == INDEXER_KEY_FP8 ? INDEXER_KEY_ROW_BYTES_FP8 : INDEXER_KEY_ROW_BYTES;
}
bool is_fp8(const IndexerDims* d) { return d->key_format == INDEXER_KEY_FP8; }

int check_cand_dims(const IndexerDims* d, int T) {
  if (d->cand_topk_blocks < 1 || d->cand_block_size < 1)
    return fail(INDEXER_ERR_DIMS, "candidate filter needs cand_topk_blocks >= 1 and cand_block_size >= 1");
  const long long nblk = ((long long)T + d->cand_block_size - 1) / d->cand_block_size;
  if (nblk > kCandMaxBlocks)
    return fail(INDEXER_ERR_DIMS, "%lld candidate blocks exceed the limit of %d", nblk, kCandMaxBlocks);
  return INDEXER_OK;
}

int check_rows(int B, int S, int start_pos) {
  if (B < 1 || S < 1) return fail(INDEXER_ERR_DIMS, "B and S must be >= 1 (got %d, %d)", B, S);
  if (start_pos < 0) return fail(INDEXER_ERR_RANGE, "start_pos must be >= 0 (got %d)", start_pos);
  if ((long long)start_pos + S > (1LL << 30)) return fail(INDEXER_ERR_RANGE, "start_pos + S too large");
  return INDEXER_OK;
}

struct WsLayout {
  size_t q_rows, w_prime, scores, total;
};

// status header | query rows | w' | scores
WsLayout ws_layout(const IndexerDims* d, int B, int S, int start_pos) {
  WsLayout l;
  const size_t nvec = (size_t)B * S * d->n_heads;
  const size_t T = (size_t)((start_pos + S) / d->ratio);
  l.q_rows = INDEXER_STATUS_BYTES;
  l.w_prime = l.q_rows + round_up(nvec * row_bytes(d), 256);
  l.scores = l.w_prime + round_up(nvec * sizeof(float), 256);
  l.total = l.scores + round_up((size_t)B * S * T * sizeof(float), 256);
  return l;
}

struct PagedWsLayout {
  size_t q_rows, w_prime, scores, rows, groups, total;
  int qg, n_groups;
};

// status header | query rows | w' | scores [Q][T_max] | row metadata | row groups
PagedWsLayout paged_ws_layout(const IndexerDims* d, int Q, int n_seq, int T_max) {
  PagedWsLayout l;
  const size_t nvec = (size_t)Q * d->n_heads;
  l.qg = score_group_rows(d->n_heads, Q <= n_seq);
  const long long g = ((long long)Q + l.qg - 1) / l.qg + n_seq;
  l.n_groups = (int)(g < Q ? g : Q);
  l.q_rows = INDEXER_STATUS_BYTES;
  l.w_prime = l.q_rows + round_up(nvec * row_bytes(d), 256);
  l.scores = l.w_prime + round_up(nvec * sizeof(float), 256);
  l.rows = l.scores + round_up((size_t)Q * T_max * sizeof(float), 256);
  l.groups = l.rows + round_up((size_t)Q * sizeof(RowInfo), 256);
  l.total = l.groups + round_up((size_t)l.n_groups * sizeof(RowGroup), 256);
  return l;
}

#define RETURN_IF(x)        \
  do {                      \
    int _rc = (x);          \
    if (_rc != INDEXER_OK) return _rc; \
  } while (0)

}  // namespace

namespace indexer {
// Lets other translation units of the library report through indexer_last_error().
int set_last_error(int code, const char* msg) {
  g_last_error = msg;
  return code;
}
}  // namespace indexer

extern "C" {

const char* indexer_last_error(void) { return g_last_error.c_str(); }

int indexer_abi_version(void) { return 405; }

// ---------------------------------------------------------------------------- RoPE table
int indexer_rope_table(const IndexerYarn* y, int rope_dim, int max_pos, float* table, indexer_stream_t stream) {
  if (!y) return fail(INDEXER_ERR_NULL, "yarn is NULL");
  if (!table) return fail(INDEXER_ERR_NULL, "table is NULL");
  if (!aligned(table, 8)) return fail(INDEXER_ERR_ALIGN, "table must be 8-byte aligned");
  if (rope_dim < 2 || rope_dim > 128 || (rope_dim & 1))
    return fail(INDEXER_ERR_DIMS, "rope_dim must be even in [2, 128] (got %d)", rope_dim);
  if (max_pos < 1 || max_pos > (1 << 24)) return fail(INDEXER_ERR_RANGE, "max_pos must be in [1, 2^24]");
  if (!(y->theta > 1.0) || !(y->factor > 0.0)) return fail(INDEXER_ERR_DIMS, "theta must be > 1 and factor > 0");
  if (y->original_seq_len > 0 && (!(y->beta_fast > 0.0) || !(y->beta_slow > 0.0)))
    return fail(INDEXER_ERR_DIMS, "beta_fast and beta_slow must be > 0");
  RETURN_IF(check_arch());
  // f'_i on the host in f64, rounded to f32 (NTK-by-parts YaRN, "Module compress" page,
  // yarn_freqs_cis): ramp between the correction dims of beta_fast and beta_slow.
  const int half = rope_dim / 2;
  RopeFreqs f;
  double low = 0.0, high = 0.0;
  const bool yarn = y->original_seq_len > 0;
  if (yarn) {
    const double pi = 3.14159265358979323846;
    auto corr = [&](double rot) {
      return rope_dim * std::log((double)y->original_seq_len / (rot * 2.0 * pi)) / (2.0 * std::log(y->theta));
    };
    low = std::floor(corr(y->beta_fast));
    high = std::ceil(corr(y->beta_slow));
    if (low < 0.0) low = 0.0;
    if (high > rope_dim - 1) high = rope_dim - 1;
  }
  const double span = high != low ? high - low : 0.001;
  for (int i = 0; i < half; ++i) {
    double fi = std::pow(y->theta, -2.0 * i / rope_dim);
    if (yarn) {
      double ramp = (i - low) / span;
      ramp = ramp < 0.0 ? 0.0 : (ramp > 1.0 ? 1.0 : ramp);
      fi = fi / y->factor * ramp + fi * (1.0 - ramp);
    }
    f.f[i] = (float)fi;
  }
  const cudaError_t e = launch_rope_table(f, half, max_pos, table, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
  return ok();
}

// ---------------------------------------------------------------------------- key publish
// Validates a sequence-major key publish and fills its launch arguments (no launch).
static int build_publish(const IndexerDims* dims, const indexer_bf16* latent, int B, int G, int Din,
                         const indexer_bf16* wk, const indexer_bf16* k_norm_w, const float* rope_cs, int max_pos,
                         int start_pos, uint8_t* k_cache, int T_cap, PublishArgs* out) {
  RETURN_IF(check_dims(dims));
  if (!latent || !wk || !k_norm_w || !rope_cs || !k_cache) return fail(INDEXER_ERR_NULL, "a required pointer is NULL");
  if (B < 1 || G < 1) return fail(INDEXER_ERR_DIMS, "B and G must be >= 1 (got %d, %d)", B, G);
  if (Din < 8 || Din > 1024 || (Din % 8)) return fail(INDEXER_ERR_DIMS, "Din must be a multiple of 8 in [8, 1024]");
  if (!aligned(latent, 16) || !aligned(wk, 16)) return fail(INDEXER_ERR_ALIGN, "latent and wk must be 16-byte aligned");
  if (!aligned(rope_cs, 8)) return fail(INDEXER_ERR_ALIGN, "rope_cs must be 8-byte aligned");
  if (T_cap < INDEXER_PAGE_KEYS || (T_cap % INDEXER_PAGE_KEYS))
    return fail(INDEXER_ERR_ALIGN, "T_cap must be a positive multiple of %d (got %d)", INDEXER_PAGE_KEYS, T_cap);
  if (!aligned(k_cache, 16)) return fail(INDEXER_ERR_ALIGN, "k_cache must be 16-byte aligned");
  if (start_pos < 0) return fail(INDEXER_ERR_RANGE, "start_pos must be >= 0");
  const int r = dims->ratio;
  PublishArgs a{};
  if (start_pos == 0) {
    a.slot0 = 0;
    a.pos0 = 0;
    a.pos_step = r;
  } else {
    if (G != 1) return fail(INDEXER_ERR_RANGE, "decode publishes one key (G == 1), got G = %d", G);
    if ((start_pos + 1) % r != 0)
      return fail(INDEXER_ERR_RANGE, "start_pos %d does not complete a group of %d", start_pos, r);
    a.slot0 = start_pos / r;
    a.pos0 = start_pos + 1 - r;
    a.pos_step = r;
  }
  if ((long long)a.slot0 + G > T_cap) return fail(INDEXER_ERR_RANGE, "slots up to %lld exceed T_cap %d", (long long)a.slot0 + G, T_cap);
  if ((long long)a.pos0 + (long long)(G - 1) * a.pos_step >= max_pos)
    return fail(INDEXER_ERR_RANGE, "RoPE position beyond the table (max_pos %d)", max_pos);
  a.latent = latent;
  a.wk = wk;
  a.knorm = k_norm_w;
  a.rope_cs = rope_cs;
  a.k_pool = k_cache;
  a.status = nullptr;
  a.slots = nullptr;
  a.positions = nullptr;
  a.num_pages = 0;
  a.max_pos = max_pos;
  a.B = B;
  a.G = G;
  a.Din = Din;
  a.rope_dim = dims->rope_dim;
  a.T_cap = T_cap;
  a.fp8 = is_fp8(dims) ? 1 : 0;
  a.eps = dims->norm_eps;
  *out = a;
  return INDEXER_OK;
}

int indexer_publish_k(const IndexerDims* dims, const indexer_bf16* latent, int B, int G, int Din,
                      const indexer_bf16* wk, const indexer_bf16* k_norm_w, const float* rope_cs, int max_pos,
                      int start_pos, uint8_t* k_cache, int T_cap, indexer_stream_t stream) {
  PublishArgs a{};
  RETURN_IF(build_publish(dims, latent, B, G, Din, wk, k_norm_w, rope_cs, max_pos, start_pos, k_cache, T_cap, &a));
  RETURN_IF(check_arch());
  const cudaError_t e = launch_publish(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "publish launch");
  return ok();
}

// ---------------------------------------------------------------------------- query prep
static PrepArgs make_prep_args(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                               int start_pos, const float* rope_cs, uint8_t* q_rows, float* w_prime,
                               uint32_t* status) {
  PrepArgs a{};
  a.status = status;
  a.q = q;
  a.w = w;
  a.rope_cs = rope_cs;
  a.q_rows = q_rows;
  a.w_prime = w_prime;
  a.n_vec = (long long)B * S * dims->n_heads;
  a.S = S;
  a.H = dims->n_heads;
  a.h_shift = __builtin_ctz((unsigned)dims->n_heads);
  a.fp8 = is_fp8(dims) ? 1 : 0;
  a.rope_dim = dims->rope_dim;
  a.start_pos = start_pos;
  a.w_scale = head_weight_scale(dims);
  return a;
}

static int prep_q_checked(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                          int start_pos, const float* rope_cs, uint8_t* q_rows, float* w_prime,
                          cudaStream_t stream, uint32_t* status = nullptr) {
  const PrepArgs a = make_prep_args(dims, q, w, B, S, start_pos, rope_cs, q_rows, w_prime, status);
  const cudaError_t e = launch_prep_q(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prep_q launch");
  return INDEXER_OK;
}

static int check_prep_args(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                           int start_pos, const float* rope_cs, int max_pos) {
  RETURN_IF(check_dims(dims));
  RETURN_IF(check_rows(B, S, start_pos));
  if (!q || !w || !rope_cs) return fail(INDEXER_ERR_NULL, "q, w and rope_cs must not be NULL");
  if (!aligned(q, 16)) return fail(INDEXER_ERR_ALIGN, "q must be 16-byte aligned");
  if (!aligned(rope_cs, 8)) return fail(INDEXER_ERR_ALIGN, "rope_cs must be 8-byte aligned");
  if ((long long)start_pos + S > max_pos)
    return fail(INDEXER_ERR_RANGE, "query positions up to %lld exceed the RoPE table (max_pos %d)",
                (long long)start_pos + S - 1, max_pos);
  return INDEXER_OK;
}

int indexer_prep_q(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S, int start_pos,
                   const float* rope_cs, int max_pos, uint8_t* q_rows, float* w_prime, indexer_stream_t stream) {
  RETURN_IF(check_prep_args(dims, q, w, B, S, start_pos, rope_cs, max_pos));
  if (!q_rows || !w_prime) return fail(INDEXER_ERR_NULL, "q_rows and w_prime must not be NULL");
  if (!aligned(q_rows, 16) || !aligned(w_prime, 4))
    return fail(INDEXER_ERR_ALIGN, "q_rows must be 16-byte aligned and w_prime 4-byte aligned");
  RETURN_IF(check_arch());
  RETURN_IF(prep_q_checked(dims, q, w, B, S, start_pos, rope_cs, q_rows, w_prime, (cudaStream_t)stream));
  return ok();
}

// ---------------------------------------------------------------------------- fused query projection
int indexer_prep_q_proj(const IndexerDims* dims, const indexer_bf16* qr, int Kq, const indexer_bf16* wq_b,
                        const indexer_bf16* w, int B, int S, int start_pos, const float* rope_cs, int max_pos,
                        uint8_t* q_rows, float* w_prime, indexer_bf16* q_out, void* ws, size_t ws_bytes,
                        indexer_stream_t stream) {
  RETURN_IF(check_prep_args(dims, qr, w, B, S, start_pos, rope_cs, max_pos));
  if (is_fp8(dims)) return fail(INDEXER_ERR_DIMS, "the fused query projection writes MXFP4 query rows only");
  if (Kq < 64 || Kq > 16384 || (Kq % 64))
    return fail(INDEXER_ERR_DIMS, "Kq (q_lora_rank) must be a multiple of 64 in [64, 16384] (got %d)", Kq);
  if (dims->n_heads % 2) return fail(INDEXER_ERR_DIMS, "the fused query projection takes an even n_heads");
  if (!wq_b || !q_rows || !w_prime || !ws) return fail(INDEXER_ERR_NULL, "wq_b, q_rows, w_prime and ws must not be NULL");
  if (!aligned(wq_b, 16) || !aligned(q_rows, 16) || !aligned(w_prime, 4) || !aligned(ws, 16) ||
      (q_out && !aligned(q_out, 16)))
    return fail(INDEXER_ERR_ALIGN, "qr, wq_b, q_rows, q_out and ws must be 16-byte aligned, w_prime 4-byte aligned");
  if (ws_bytes < INDEXER_STATUS_BYTES) return fail(INDEXER_ERR_WORKSPACE, "ws needs %d bytes", INDEXER_STATUS_BYTES);
  if ((long long)B * S > (1ll << 30)) return fail(INDEXER_ERR_DIMS, "B * S is too large");
  RETURN_IF(check_arch());
  QprojArgs a{};
  a.qr = qr;
  a.wq_b = wq_b;
  a.w = w;
  a.rope_cs = rope_cs;
  a.q_rows = q_rows;
  a.w_prime = w_prime;
  a.q_out = q_out;
  a.status = static_cast<uint32_t*>(ws);
  a.R = B * S;
  a.Kq = Kq;
  a.H = dims->n_heads;
  a.S = S;
  a.start_pos = start_pos;
  a.rope_dim = dims->rope_dim;
  a.w_scale = make_prep_args(dims, qr, w, B, S, start_pos, rope_cs, q_rows, w_prime, nullptr).w_scale;
  const cudaError_t e = launch_qproj(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "query projection launch");
  return ok();
}

// ---------------------------------------------------------------------------- upstream producers
int indexer_compress_weights(const IndexerDims* dims, const indexer_bf16* x, int B, int S, int dim,
                             const indexer_bf16* wkv, const indexer_bf16* wgate, const indexer_bf16* norm_w,
                             const indexer_bf16* wproj, indexer_bf16* latent, indexer_bf16* latent_q,
                             indexer_bf16* w_out, void* ws, size_t ws_bytes, indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  if (!x || !wkv || !wgate || !norm_w || !wproj || !latent || !w_out || !ws)
    return fail(INDEXER_ERR_NULL, "a required pointer is NULL");
  if (B < 1 || S < 1) return fail(INDEXER_ERR_DIMS, "B and S must be >= 1 (got %d, %d)", B, S);
  const int r = dims->ratio;
  if (r != 1 && r != 2 && r != 4 && r != 8 && r != 16 && r != 32)
    return fail(INDEXER_ERR_DIMS, "the fused compressor takes ratio 1, 2, 4, 8, 16 or 32 (got %d)", r);
  if (S % r) return fail(INDEXER_ERR_DIMS, "S = %d is not a whole number of groups of %d tokens", S, r);
  if (dim < 64 || dim > 65536 || (dim % 64)) return fail(INDEXER_ERR_DIMS, "dim must be a multiple of 64 in [64, 65536]");
  if ((long long)B * S > (1ll << 30)) return fail(INDEXER_ERR_DIMS, "B * S is too large");
  if (!aligned(x, 16) || !aligned(wkv, 16) || !aligned(wgate, 16) || !aligned(wproj, 16) || !aligned(latent, 16) ||
      (latent_q && !aligned(latent_q, 16)) || !aligned(w_out, 4) || !aligned(ws, 16))
    return fail(INDEXER_ERR_ALIGN, "x, the weights, latent, latent_q and ws must be 16-byte aligned, w_out 4-byte");
  if (ws_bytes < INDEXER_STATUS_BYTES) return fail(INDEXER_ERR_WORKSPACE, "ws needs %d bytes", INDEXER_STATUS_BYTES);
  RETURN_IF(check_arch());
  CompressArgs a{};
  a.x = x;
  a.wkv = wkv;
  a.wgate = wgate;
  a.norm_w = norm_w;
  a.wproj = wproj;
  a.latent = latent;
  a.latent_q = latent_q;
  a.w_out = w_out;
  a.status = static_cast<uint32_t*>(ws);
  a.R = B * S;
  a.dim = dim;
  a.H = dims->n_heads;
  a.ratio = r;
  a.eps = dims->norm_eps;
  const cudaError_t e = launch_compress(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "compress launch");
  return ok();
}

// ---------------------------------------------------------------------------- scores
static int check_cache(const uint8_t* k_cache, int T_cap, int T) {
  if (!k_cache) return fail(INDEXER_ERR_NULL, "k_cache is NULL");
  if (!aligned(k_cache, 16)) return fail(INDEXER_ERR_ALIGN, "k_cache must be 16-byte aligned");
  if (T_cap < INDEXER_PAGE_KEYS || (T_cap % INDEXER_PAGE_KEYS))
    return fail(INDEXER_ERR_ALIGN, "T_cap must be a positive multiple of %d (got %d)", INDEXER_PAGE_KEYS, T_cap);
  if (T > T_cap) return fail(INDEXER_ERR_RANGE, "T = %d keys exceed T_cap = %d", T, T_cap);
  return INDEXER_OK;
}

int indexer_scores(const IndexerDims* dims, const uint8_t* q_rows, const float* w_prime, int B, int S, int start_pos,
                   const uint8_t* k_cache, int T_cap, const int32_t* cand_blocks, float* scores, void* ws,
                   size_t ws_bytes, indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  RETURN_IF(check_rows(B, S, start_pos));
  const int T = (start_pos + S) / dims->ratio;
  RETURN_IF(check_cache(k_cache, T_cap, T));
  if (!q_rows || !w_prime || !scores || !ws) return fail(INDEXER_ERR_NULL, "a required pointer is NULL");
  if (!aligned(q_rows, 16) || !aligned(w_prime, 16) || !aligned(scores, 4) || !aligned(ws, 16))
    return fail(INDEXER_ERR_ALIGN, "q_rows, w_prime and ws must be 16-byte aligned, scores 4-byte aligned");
  if (ws_bytes < INDEXER_STATUS_BYTES) return fail(INDEXER_ERR_WORKSPACE, "workspace smaller than %d bytes", INDEXER_STATUS_BYTES);
  if (cand_blocks) RETURN_IF(check_cand_dims(dims, T));
  RETURN_IF(check_arch());
  ScoreArgs a{};
  a.q_rows = q_rows;
  a.w_prime = w_prime;
  a.k_pool = k_cache;
  a.pages_per_seq = T_cap / INDEXER_PAGE_KEYS;
  a.scores = scores;
  a.ld = T;
  a.cand = cand_blocks;
  a.status = static_cast<uint32_t*>(ws);
  a.sched = static_cast<uint32_t*>(ws) + kSchedWord;
  a.B = B;
  a.S = S;
  a.H = dims->n_heads;
  a.T = T;
  a.start_pos = start_pos;
  a.ratio = dims->ratio;
  a.cbk = dims->cand_topk_blocks;
  a.cbs = dims->cand_block_size > 0 ? dims->cand_block_size : 1;
  a.fill_masked = 1;
  a.fp8 = is_fp8(dims) ? 1 : 0;
  const cudaError_t e = launch_scores(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "scores launch");
  return ok();
}

int indexer_scores_hold_test(const IndexerDims* dims, const uint8_t* q_rows, const float* w_prime, int B, int S,
                             int start_pos, const uint8_t* k_cache, int T_cap, float* scores, void* ws,
                             size_t ws_bytes, uint64_t wait_ns, indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  RETURN_IF(check_rows(B, S, start_pos));
  if (S < 2) return fail(INDEXER_ERR_DIMS, "the hold test runs the several-row kernel: S must be >= 2");
  if (wait_ns < 1000ull || wait_ns > 1000000000ull) return fail(INDEXER_ERR_RANGE, "wait_ns must be in [1e3, 1e9]");
  const int T = (start_pos + S) / dims->ratio;
  if (T < 1) return fail(INDEXER_ERR_RANGE, "no key is visible");
  RETURN_IF(check_cache(k_cache, T_cap, T));
  if (!q_rows || !w_prime || !scores || !ws) return fail(INDEXER_ERR_NULL, "a required pointer is NULL");
  if (!aligned(q_rows, 16) || !aligned(w_prime, 16) || !aligned(scores, 4) || !aligned(ws, 16))
    return fail(INDEXER_ERR_ALIGN, "q_rows, w_prime and ws must be 16-byte aligned, scores 4-byte aligned");
  if (ws_bytes < INDEXER_STATUS_BYTES) return fail(INDEXER_ERR_WORKSPACE, "workspace smaller than %d bytes", INDEXER_STATUS_BYTES);
  RETURN_IF(check_arch());
  ScoreArgs a{};
  a.q_rows = q_rows;
  a.w_prime = w_prime;
  a.k_pool = k_cache;
  a.pages_per_seq = T_cap / INDEXER_PAGE_KEYS;
  a.scores = scores;
  a.ld = T;
  a.status = static_cast<uint32_t*>(ws);
  a.sched = static_cast<uint32_t*>(ws) + kSchedWord;
  a.B = B;
  a.S = S;
  a.H = dims->n_heads;
  a.T = T;
  a.start_pos = start_pos;
  a.ratio = dims->ratio;
  a.cbk = dims->cand_topk_blocks;
  a.cbs = 1;
  a.fp8 = is_fp8(dims) ? 1 : 0;
  a.wait_ns = wait_ns;
  a.hold_producer = 1;
  const cudaError_t e = launch_scores(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "scores launch");
  return ok();
}

// ---------------------------------------------------------------------------- selection
int indexer_select_candidate_blocks(const IndexerDims* dims, const float* scores, int B, int S, int start_pos, int T,
                                    int32_t* blocks_out, indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  RETURN_IF(check_rows(B, S, start_pos));
  if (!scores || !blocks_out) return fail(INDEXER_ERR_NULL, "scores and blocks_out must not be NULL");
  if (!aligned(scores, 16)) return fail(INDEXER_ERR_ALIGN, "scores must be 16-byte aligned");
  if (T < 0 || T != (start_pos + S) / dims->ratio)
    return fail(INDEXER_ERR_RANGE, "T must equal (start_pos + S) / ratio");
  RETURN_IF(check_cand_dims(dims, T));
  RETURN_IF(check_arch());
  CandArgs a{};
  a.scores = scores;
  a.blocks = blocks_out;
  a.rows = B * S;
  a.S = S;
  a.T = T;
  a.ld = T;
  a.start_pos = start_pos;
  a.ratio = dims->ratio;
  a.cbk = dims->cand_topk_blocks;
  a.cbs = dims->cand_block_size;
  const cudaError_t e = launch_candidates(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "candidate launch");
  return ok();
}

static TopkArgs make_topk_args(const IndexerDims* dims, const float* scores, int B, int S, int start_pos, int T,
                               const int32_t* cand, int32_t* out, bool sparse) {
  TopkArgs a{};
  a.scores = scores;
  a.out = out;
  a.cand = cand;
  a.rows = B * S;
  a.S = S;
  a.T = T;
  a.ld = T;
  a.start_pos = start_pos;
  a.ratio = dims->ratio;
  a.topk = dims->index_topk;
  a.offset = dims->offset;
  a.cbk = dims->cand_topk_blocks;
  a.cbs = dims->cand_block_size > 0 ? dims->cand_block_size : 1;
  a.sparse = sparse ? 1 : 0;
  return a;
}

static int topk_checked(const IndexerDims* dims, const float* scores, int B, int S, int start_pos, int T,
                        const int32_t* cand, int32_t* out, cudaStream_t stream, bool sparse = false) {
  const TopkArgs a = make_topk_args(dims, scores, B, S, start_pos, T, cand, out, sparse);
  const cudaError_t e = launch_topk(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "topk launch");
  return INDEXER_OK;
}

// Level one with few rows and no filter of its own: candidate blocks and top-k in one launch.
static bool fuse_cand_topk(int rows, int T, const int32_t* cand_in, const int32_t* cand_out) {
  return cand_out != nullptr && cand_in == nullptr && rows < 4096 && T <= kTopkMaxT;
}

int indexer_topk(const IndexerDims* dims, const float* scores, int B, int S, int start_pos, int T, int32_t* out,
                 indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  RETURN_IF(check_rows(B, S, start_pos));
  if (!scores || !out) return fail(INDEXER_ERR_NULL, "scores and out must not be NULL");
  if (!aligned(scores, 16)) return fail(INDEXER_ERR_ALIGN, "scores must be 16-byte aligned");
  if (T < 0 || T != (start_pos + S) / dims->ratio)
    return fail(INDEXER_ERR_RANGE, "T must equal (start_pos + S) / ratio");
  if (T > kTopkMaxT) return fail(INDEXER_ERR_DIMS, "T = %d exceeds the top-k limit of %d", T, kTopkMaxT);
  RETURN_IF(check_arch());
  RETURN_IF(topk_checked(dims, scores, B, S, start_pos, T, nullptr, out, (cudaStream_t)stream));
  return ok();
}

// ---------------------------------------------------------------------------- forward
size_t indexer_workspace_size(const IndexerDims* dims, int B, int S, int start_pos) {
  if (check_dims(dims) != INDEXER_OK || check_rows(B, S, start_pos) != INDEXER_OK) return 0;
  return ws_layout(dims, B, S, start_pos).total;
}

// Every check of indexer_forward's arguments (no launch, nothing enqueued).
static int check_forward(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                         int start_pos, const float* rope_cs, int max_pos, const uint8_t* k_cache, int T_cap,
                         const int32_t* cand_in, const int32_t* cand_out, const int32_t* topk_out,
                         const float* scores_out, const void* ws, size_t ws_bytes) {
  RETURN_IF(check_prep_args(dims, q, w, B, S, start_pos, rope_cs, max_pos));
  const int T = (start_pos + S) / dims->ratio;
  RETURN_IF(check_cache(k_cache, T_cap, T));
  if (!topk_out || !ws) return fail(INDEXER_ERR_NULL, "topk_out and ws must not be NULL");
  if (!aligned(ws, 256)) return fail(INDEXER_ERR_ALIGN, "ws must be 256-byte aligned");
  if (scores_out && !aligned(scores_out, 16)) return fail(INDEXER_ERR_ALIGN, "scores_out must be 16-byte aligned");
  if (T > kTopkMaxT) return fail(INDEXER_ERR_DIMS, "T = %d exceeds the top-k limit of %d", T, kTopkMaxT);
  if (cand_in || cand_out) RETURN_IF(check_cand_dims(dims, T));
  const WsLayout l = ws_layout(dims, B, S, start_pos);
  if (ws_bytes < l.total) return fail(INDEXER_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, l.total);
  return check_arch();
}

// The forward of indexer_forward; with `pub`, the step's key publish runs first (in the same
// launch as the query prep when both are small).
static int forward_impl(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                        int start_pos, const float* rope_cs, int max_pos, const uint8_t* k_cache, int T_cap,
                        const int32_t* cand_in, int32_t* cand_out, int32_t* topk_out, float* scores_out, void* ws,
                        size_t ws_bytes, indexer_stream_t stream, const PublishArgs* pub) {
  RETURN_IF(check_forward(dims, q, w, B, S, start_pos, rope_cs, max_pos, k_cache, T_cap, cand_in, cand_out, topk_out,
                          scores_out, ws, ws_bytes));
  const int T = (start_pos + S) / dims->ratio;
  const WsLayout l = ws_layout(dims, B, S, start_pos);
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint8_t* q_rows = base + l.q_rows;
  float* w_prime = reinterpret_cast<float*>(base + l.w_prime);
  float* scores = scores_out ? scores_out : reinterpret_cast<float*>(base + l.scores);
  if (pub) {
    const PrepArgs pa = make_prep_args(dims, q, w, B, S, start_pos, rope_cs, q_rows, w_prime,
                                       reinterpret_cast<uint32_t*>(base));
    const cudaError_t e = launch_publish_prep(*pub, pa, st);
    if (e != cudaSuccess) return cuda_fail(e, "publish / prep_q launch");
  } else {
    RETURN_IF(prep_q_checked(dims, q, w, B, S, start_pos, rope_cs, q_rows, w_prime, st,
                             reinterpret_cast<uint32_t*>(base)));
  }
  // level two with one query row and no score output: only the kept blocks' keys are
  // scored and ranked (the other positions of the workspace scores are never read)
  const bool sparse2 = cand_in && !cand_out && !scores_out && S == 1 && T <= 32768 &&
                       (long long)dims->cand_topk_blocks * dims->cand_block_size <= 8192;
  if (T > 0) {
    ScoreArgs a{};
    a.q_rows = q_rows;
    a.w_prime = w_prime;
    a.k_pool = k_cache;
    a.pages_per_seq = T_cap / INDEXER_PAGE_KEYS;
    a.scores = scores;
    a.ld = T;
    // otherwise the candidate filter is applied by the top-k (cand_out sees unfiltered scores)
    a.cand = sparse2 ? cand_in : nullptr;
    a.sparse_pages = sparse2 ? 1 : 0;
    a.status = reinterpret_cast<uint32_t*>(base);
    a.sched = reinterpret_cast<uint32_t*>(base) + kSchedWord;
    a.B = B;
    a.S = S;
    a.H = dims->n_heads;
    a.T = T;
    a.start_pos = start_pos;
    a.ratio = dims->ratio;
    a.cbk = dims->cand_topk_blocks;
    a.cbs = dims->cand_block_size > 0 ? dims->cand_block_size : 1;
    a.fill_masked = scores_out ? 1 : 0;
    a.fp8 = is_fp8(dims) ? 1 : 0;
    const cudaError_t e = launch_scores(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "scores launch");
    if (cand_out) {
      CandArgs c{};
      c.scores = scores;
      c.blocks = cand_out;
      c.rows = B * S;
      c.S = S;
      c.T = T;
      c.ld = T;
      c.start_pos = start_pos;
      c.ratio = dims->ratio;
      c.cbk = dims->cand_topk_blocks;
      c.cbs = dims->cand_block_size;
      if (fuse_cand_topk(B * S, T, cand_in, cand_out)) {
        const TopkArgs ta = make_topk_args(dims, scores, B, S, start_pos, T, nullptr, topk_out, false);
        const cudaError_t e2 = launch_cand_topk(c, ta, st);
        if (e2 != cudaSuccess) return cuda_fail(e2, "candidate / topk launch");
        return ok();
      }
      const cudaError_t e2 = launch_candidates(c, st);
      if (e2 != cudaSuccess) return cuda_fail(e2, "candidate launch");
    }
  }
  RETURN_IF(topk_checked(dims, scores, B, S, start_pos, T, cand_in, topk_out, st, sparse2 && T > 0));
  return ok();
}

// ---------------------------------------------------------------------------- page pool
int indexer_publish_k_paged(const IndexerDims* dims, const indexer_bf16* latent, int N, int Din,
                            const indexer_bf16* wk, const indexer_bf16* k_norm_w, const float* rope_cs, int max_pos,
                            const int32_t* positions, const int32_t* slot_mapping, uint8_t* k_pool, int num_pages,
                            void* ws, size_t ws_bytes, indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  if (!latent || !wk || !k_norm_w || !rope_cs || !positions || !slot_mapping || !k_pool || !ws)
    return fail(INDEXER_ERR_NULL, "a required pointer is NULL");
  if (N < 0) return fail(INDEXER_ERR_DIMS, "N must be >= 0 (got %d)", N);
  if (Din < 8 || Din > 1024 || (Din % 8)) return fail(INDEXER_ERR_DIMS, "Din must be a multiple of 8 in [8, 1024]");
  if (!aligned(latent, 16) || !aligned(wk, 16)) return fail(INDEXER_ERR_ALIGN, "latent and wk must be 16-byte aligned");
  if (!aligned(rope_cs, 8)) return fail(INDEXER_ERR_ALIGN, "rope_cs must be 8-byte aligned");
  if (!aligned(positions, 4) || !aligned(slot_mapping, 4)) return fail(INDEXER_ERR_ALIGN, "positions and slot_mapping must be 4-byte aligned");
  if (!aligned(k_pool, 16)) return fail(INDEXER_ERR_ALIGN, "k_pool must be 16-byte aligned");
  if (num_pages < 1 || (long long)num_pages * INDEXER_PAGE_KEYS > (1LL << 31) - 1)
    return fail(INDEXER_ERR_DIMS, "num_pages must be in [1, 2^31 / %d)", INDEXER_PAGE_KEYS);
  if (max_pos < 1) return fail(INDEXER_ERR_RANGE, "max_pos must be >= 1");
  if (ws_bytes < INDEXER_STATUS_BYTES) return fail(INDEXER_ERR_WORKSPACE, "workspace smaller than %d bytes", INDEXER_STATUS_BYTES);
  if (!aligned(ws, 16)) return fail(INDEXER_ERR_ALIGN, "ws must be 16-byte aligned");
  RETURN_IF(check_arch());
  if (N == 0) return ok();
  PublishArgs a{};
  a.latent = latent;
  a.wk = wk;
  a.knorm = k_norm_w;
  a.rope_cs = rope_cs;
  a.k_pool = k_pool;
  a.status = static_cast<uint32_t*>(ws);
  a.B = 1;
  a.G = N;
  a.Din = Din;
  a.rope_dim = dims->rope_dim;
  a.slots = slot_mapping;
  a.positions = positions;
  a.num_pages = num_pages;
  a.max_pos = max_pos;
  a.fp8 = is_fp8(dims) ? 1 : 0;
  a.eps = dims->norm_eps;
  const cudaError_t e = launch_publish(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "publish launch");
  return ok();
}

static int check_batch(const IndexerDims* d, int Q, int n_seq, int T_max) {
  if (Q < 1 || n_seq < 1) return fail(INDEXER_ERR_DIMS, "Q and n_seq must be >= 1 (got %d, %d)", Q, n_seq);
  if (n_seq > kPlanMaxSeq) return fail(INDEXER_ERR_DIMS, "n_seq = %d exceeds the limit of %d", n_seq, kPlanMaxSeq);
  if (T_max < 1) return fail(INDEXER_ERR_DIMS, "T_max must be >= 1 (got %d)", T_max);
  if (T_max > kTopkMaxT) return fail(INDEXER_ERR_DIMS, "T_max = %d exceeds the top-k limit of %d", T_max, kTopkMaxT);
  if ((long long)Q * d->n_heads > (1LL << 31) / 128) return fail(INDEXER_ERR_DIMS, "Q * n_heads too large");
  return INDEXER_OK;
}

size_t indexer_workspace_size_paged(const IndexerDims* dims, int Q, int n_seq, int T_max) {
  if (check_dims(dims) != INDEXER_OK || check_batch(dims, Q, n_seq, T_max) != INDEXER_OK) return 0;
  return paged_ws_layout(dims, Q, n_seq, T_max).total;
}

int indexer_forward_paged(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int Q, int n_seq,
                          const int32_t* seq_pos, const int32_t* q_start, int T_max, const float* rope_cs,
                          int max_pos, const uint8_t* k_pool, int num_pages, const int32_t* block_table,
                          int bt_stride, const int32_t* cand_in, int32_t* cand_out, int32_t* topk_out,
                          float* scores_out, void* ws, size_t ws_bytes, indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  RETURN_IF(check_batch(dims, Q, n_seq, T_max));
  if (!q || !w || !seq_pos || !q_start || !rope_cs || !k_pool || !block_table || !topk_out || !ws)
    return fail(INDEXER_ERR_NULL, "a required pointer is NULL");
  if (!aligned(q, 16)) return fail(INDEXER_ERR_ALIGN, "q must be 16-byte aligned");
  if (!aligned(rope_cs, 8)) return fail(INDEXER_ERR_ALIGN, "rope_cs must be 8-byte aligned");
  if (!aligned(k_pool, 16)) return fail(INDEXER_ERR_ALIGN, "k_pool must be 16-byte aligned");
  if (!aligned(ws, 256)) return fail(INDEXER_ERR_ALIGN, "ws must be 256-byte aligned");
  if (!aligned(seq_pos, 4) || !aligned(q_start, 4) || !aligned(block_table, 4))
    return fail(INDEXER_ERR_ALIGN, "seq_pos, q_start and block_table must be 4-byte aligned");
  if (scores_out && !aligned(scores_out, 16)) return fail(INDEXER_ERR_ALIGN, "scores_out must be 16-byte aligned");
  if (max_pos < 1) return fail(INDEXER_ERR_RANGE, "max_pos must be >= 1");
  if (num_pages < 1) return fail(INDEXER_ERR_DIMS, "num_pages must be >= 1");
  const int pages_max = (T_max + INDEXER_PAGE_KEYS - 1) / INDEXER_PAGE_KEYS;
  if (bt_stride < pages_max)
    return fail(INDEXER_ERR_DIMS, "bt_stride %d < %d pages of T_max = %d keys", bt_stride, pages_max, T_max);
  if (cand_in || cand_out) RETURN_IF(check_cand_dims(dims, T_max));
  const PagedWsLayout l = paged_ws_layout(dims, Q, n_seq, T_max);
  if (ws_bytes < l.total) return fail(INDEXER_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, l.total);
  RETURN_IF(check_arch());
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(base);
  uint8_t* q_rows = base + l.q_rows;
  float* w_prime = reinterpret_cast<float*>(base + l.w_prime);
  // scores rows are T_max wide; a 16-byte row stride keeps the selection kernels' vector loads
  const int ld = T_max;
  float* scores = scores_out ? scores_out : reinterpret_cast<float*>(base + l.scores);
  RowInfo* rows = reinterpret_cast<RowInfo*>(base + l.rows);
  RowGroup* groups = reinterpret_cast<RowGroup*>(base + l.groups);
  {
    PlanArgs p{};
    p.seq_pos = seq_pos;
    p.q_start = q_start;
    p.rows = rows;
    p.groups = groups;
    p.status = status;
    p.n_seq = n_seq;
    p.n_rows = Q;
    p.n_groups = l.n_groups;
    p.qg = l.qg;
    p.ratio = dims->ratio;
    p.T_max = T_max;
    p.max_pos = max_pos;
    const cudaError_t e = launch_plan(p, st);
    if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  }
  {
    PrepArgs a{};
    a.q = q;
    a.w = w;
    a.rope_cs = rope_cs;
    a.q_rows = q_rows;
    a.w_prime = w_prime;
    a.rows = rows;
    a.status = status;
    a.n_vec = (long long)Q * dims->n_heads;
    a.S = 1;
    a.H = dims->n_heads;
    a.h_shift = __builtin_ctz((unsigned)dims->n_heads);
    a.fp8 = is_fp8(dims) ? 1 : 0;
    a.rope_dim = dims->rope_dim;
    a.w_scale = head_weight_scale(dims);
    const cudaError_t e = launch_prep_q(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "prep_q launch");
  }
  const bool single = l.qg == 1 && Q <= n_seq;
  const bool sparse2 = cand_in && !cand_out && !scores_out && single &&
                       (long long)dims->cand_topk_blocks * dims->cand_block_size <= 8192;
  {
    ScoreArgs a{};
    a.q_rows = q_rows;
    a.w_prime = w_prime;
    a.k_pool = k_pool;
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.num_pages = num_pages;
    a.groups = groups;
    a.n_groups = l.n_groups;
    a.scores = scores;
    a.ld = ld;
    a.cand = sparse2 ? cand_in : nullptr;
    a.sparse_pages = sparse2 ? 1 : 0;
    a.status = status;
    a.sched = status + kSchedWord;
    a.B = n_seq;
    a.S = single ? 1 : 2;   // selects the single-row (decode) kernel, matching l.qg
    a.H = dims->n_heads;
    a.T = T_max;
    a.ratio = dims->ratio;
    a.cbk = dims->cand_topk_blocks;
    a.cbs = dims->cand_block_size > 0 ? dims->cand_block_size : 1;
    a.fill_masked = scores_out ? 1 : 0;
    a.fp8 = is_fp8(dims) ? 1 : 0;
    const cudaError_t e = launch_scores(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "scores launch");
  }
  CandArgs cargs{};
  if (cand_out) {
    CandArgs& c = cargs;
    c.scores = scores;
    c.blocks = cand_out;
    c.rinfo = rows;
    c.rows = Q;
    c.S = 1;
    c.T = T_max;
    c.ld = ld;
    c.ratio = dims->ratio;
    c.cbk = dims->cand_topk_blocks;
    c.cbs = dims->cand_block_size;
    if (!fuse_cand_topk(Q, T_max, cand_in, cand_out)) {
      const cudaError_t e = launch_candidates(c, st);
      if (e != cudaSuccess) return cuda_fail(e, "candidate launch");
    }
  }
  {
    TopkArgs a{};
    a.scores = scores;
    a.out = topk_out;
    a.cand = cand_in;
    a.rinfo = rows;
    a.rows = Q;
    a.S = 1;
    a.T = T_max;
    a.ld = ld;
    a.ratio = dims->ratio;
    a.topk = dims->index_topk;
    a.offset = dims->offset;
    a.cbk = dims->cand_topk_blocks;
    a.cbs = dims->cand_block_size > 0 ? dims->cand_block_size : 1;
    a.sparse = sparse2 ? 1 : 0;
    const cudaError_t e = fuse_cand_topk(Q, T_max, cand_in, cand_out) ? launch_cand_topk(cargs, a, st)
                                                                       : launch_topk(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "topk launch");
  }
  return ok();
}

int indexer_forward(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                    int start_pos, const float* rope_cs, int max_pos, const uint8_t* k_cache, int T_cap,
                    const int32_t* cand_in, int32_t* cand_out, int32_t* topk_out, float* scores_out, void* ws,
                    size_t ws_bytes, indexer_stream_t stream) {
  return forward_impl(dims, q, w, B, S, start_pos, rope_cs, max_pos, k_cache, T_cap, cand_in, cand_out, topk_out,
                      scores_out, ws, ws_bytes, stream, nullptr);
}

int indexer_forward_publish(const IndexerDims* dims, const indexer_bf16* latent, int G, int Din,
                            const indexer_bf16* wk, const indexer_bf16* k_norm_w, const indexer_bf16* q,
                            const indexer_bf16* w, int B, int S, int start_pos, const float* rope_cs, int max_pos,
                            uint8_t* k_cache, int T_cap, const int32_t* cand_in, int32_t* cand_out,
                            int32_t* topk_out, float* scores_out, void* ws, size_t ws_bytes,
                            indexer_stream_t stream) {
  PublishArgs pa{};
  RETURN_IF(build_publish(dims, latent, B, G, Din, wk, k_norm_w, rope_cs, max_pos, start_pos, k_cache, T_cap, &pa));
  return forward_impl(dims, q, w, B, S, start_pos, rope_cs, max_pos, k_cache, T_cap, cand_in, cand_out, topk_out,
                      scores_out, ws, ws_bytes, stream, &pa);
}

// ---------------------------------------------------------------------------- host-buffer step
// Device staging for a step's host inputs and output, after the forward's own workspace.
struct HostStaging {
  size_t base, latent, q, w, top, total;
};
static size_t round256(size_t n) { return (n + 255) / 256 * 256; }
static HostStaging host_staging(const IndexerDims* dims, int B, int S, int start_pos, int G, int Din) {
  HostStaging h{};
  h.base = round256(indexer_workspace_size(dims, B, S, start_pos));
  h.latent = h.base;
  h.q = h.latent + round256((size_t)B * G * Din * 2);
  h.w = h.q + round256((size_t)B * S * dims->n_heads * dims->head_dim * 2);
  h.top = h.w + round256((size_t)B * S * dims->n_heads * 2);
  h.total = h.top + round256((size_t)B * S * dims->index_topk * 4);
  return h;
}

size_t indexer_workspace_size_host(const IndexerDims* dims, int B, int S, int start_pos, int G, int Din) {
  if (check_dims(dims) != INDEXER_OK || B <= 0 || S <= 0 || G < 0 || (G > 0 && Din <= 0)) return 0;
  return host_staging(dims, B, S, start_pos, G, G > 0 ? Din : 0).total;
}

int indexer_forward_publish_host(const IndexerDims* dims, const indexer_bf16* latent_h, int G, int Din,
                                 const indexer_bf16* wk, const indexer_bf16* k_norm_w, const indexer_bf16* q_h,
                                 const indexer_bf16* w_h, int B, int S, int start_pos, const float* rope_cs,
                                 int max_pos, uint8_t* k_cache, int T_cap, int32_t* topk_out_h, void* ws,
                                 size_t ws_bytes, indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  RETURN_IF(check_rows(B, S, start_pos));
  if ((G > 0 && !latent_h) || !q_h || !w_h || !topk_out_h || !ws)
    return fail(INDEXER_ERR_NULL, "a required pointer is NULL");
  if (G < 0 || (G > 0 && Din <= 0)) return fail(INDEXER_ERR_DIMS, "G must be >= 0, and Din > 0 when G > 0");
  if (G == 0) Din = 0;   // no key is published: the latent is not read
  const HostStaging h = host_staging(dims, B, S, start_pos, G, Din);
  if (ws_bytes < h.total)
    return fail(INDEXER_ERR_WORKSPACE, "ws has %zu bytes, indexer_workspace_size_host needs %zu", ws_bytes, h.total);
  if (!aligned(ws, 256)) return fail(INDEXER_ERR_ALIGN, "ws must be 256-byte aligned");
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto* lat_d = reinterpret_cast<indexer_bf16*>(base + h.latent);
  auto* q_d = reinterpret_cast<indexer_bf16*>(base + h.q);
  auto* w_d = reinterpret_cast<indexer_bf16*>(base + h.w);
  auto* top_d = reinterpret_cast<int32_t*>(base + h.top);
  // every check of the step (publish and forward, on the staging pointers) before any copy
  if (G > 0) {
    PublishArgs pa{};
    RETURN_IF(build_publish(dims, lat_d, B, G, Din, wk, k_norm_w, rope_cs, max_pos, start_pos, k_cache, T_cap, &pa));
  }
  RETURN_IF(check_forward(dims, q_d, w_d, B, S, start_pos, rope_cs, max_pos, k_cache, T_cap, nullptr, nullptr, top_d,
                          nullptr, ws, h.base));
  cudaStream_t st = (cudaStream_t)stream;
  const size_t qb = (size_t)B * S * dims->n_heads * dims->head_dim * 2, wb = (size_t)B * S * dims->n_heads * 2;
  const size_t lb = (size_t)B * G * Din * 2, tb = (size_t)B * S * dims->index_topk * 4;
  cudaError_t e = lb ? cudaMemcpyAsync(lat_d, latent_h, lb, cudaMemcpyHostToDevice, st) : cudaSuccess;
  if (e == cudaSuccess) e = cudaMemcpyAsync(q_d, q_h, qb, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(w_d, w_h, wb, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "input copies");
  if (G > 0)
    RETURN_IF(indexer_forward_publish(dims, lat_d, G, Din, wk, k_norm_w, q_d, w_d, B, S, start_pos, rope_cs, max_pos,
                                      k_cache, T_cap, nullptr, nullptr, top_d, nullptr, ws, h.base, stream));
  else   // no key completes this step: the forward alone
    RETURN_IF(indexer_forward(dims, q_d, w_d, B, S, start_pos, rope_cs, max_pos, k_cache, T_cap, nullptr, nullptr,
                              top_d, nullptr, ws, h.base, stream));
  e = cudaMemcpyAsync(topk_out_h, top_d, tb, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "output copy");
  return ok();
}

// ---------------------------------------------------------------------------- row-major caches
static int layout_call(const IndexerDims* dims, const uint8_t* rows_in, uint8_t* rows_out, int n_seq, int n_keys,
                       int ld_rows, const uint8_t* pages_in, uint8_t* pages_out, int T_cap, indexer_stream_t stream) {
  RETURN_IF(check_dims(dims));
  const bool to_pages = rows_in != nullptr;
  if ((to_pages ? (const void*)pages_out : (const void*)rows_out) == nullptr ||
      (to_pages ? (const void*)rows_in : (const void*)pages_in) == nullptr)
    return fail(INDEXER_ERR_NULL, "rows and k_cache must not be NULL");
  if (n_seq < 1 || n_keys < 0) return fail(INDEXER_ERR_DIMS, "n_seq must be >= 1 and n_keys >= 0");
  if (T_cap < INDEXER_PAGE_KEYS || (T_cap % INDEXER_PAGE_KEYS))
    return fail(INDEXER_ERR_ALIGN, "T_cap must be a positive multiple of %d (got %d)", INDEXER_PAGE_KEYS, T_cap);
  if (n_keys > T_cap || n_keys > ld_rows)
    return fail(INDEXER_ERR_RANGE, "n_keys %d exceeds T_cap %d or ld_rows %d", n_keys, T_cap, ld_rows);
  const void* rp = to_pages ? (const void*)rows_in : (const void*)rows_out;
  const void* pp = to_pages ? (const void*)pages_out : (const void*)pages_in;
  if (!aligned(rp, 4) || !aligned(pp, 16)) return fail(INDEXER_ERR_ALIGN, "rows must be 4-byte and k_cache 16-byte aligned");
  RETURN_IF(check_arch());
  LayoutArgs a{};
  a.rows_in = rows_in;
  a.pages = pages_out;
  a.pages_in = pages_in;
  a.rows_out = rows_out;
  a.n_seq = n_seq;
  a.n_keys = n_keys;
  a.ld_rows = ld_rows;
  a.T_cap = T_cap;
  a.fp8 = is_fp8(dims) ? 1 : 0;
  const cudaError_t e = launch_layout(a, to_pages, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "layout launch");
  return ok();
}

int indexer_cache_from_rows(const IndexerDims* dims, const uint8_t* rows, int n_seq, int n_keys, int ld_rows,
                            uint8_t* k_cache, int T_cap, indexer_stream_t stream) {
  return layout_call(dims, rows, nullptr, n_seq, n_keys, ld_rows, nullptr, k_cache, T_cap, stream);
}

int indexer_cache_to_rows(const IndexerDims* dims, const uint8_t* k_cache, int T_cap, int n_seq, int n_keys,
                          uint8_t* rows, int ld_rows, indexer_stream_t stream) {
  return layout_call(dims, nullptr, rows, n_seq, n_keys, ld_rows, k_cache, nullptr, T_cap, stream);
}

int indexer_workspace_init(void* ws, size_t ws_bytes, indexer_stream_t stream) {
  if (!ws) return fail(INDEXER_ERR_NULL, "ws is NULL");
  if (ws_bytes < INDEXER_STATUS_BYTES) return fail(INDEXER_ERR_WORKSPACE, "workspace smaller than %d bytes", INDEXER_STATUS_BYTES);
  const cudaError_t e = cudaMemsetAsync(ws, 0, INDEXER_STATUS_BYTES, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace init");
  return ok();
}

int indexer_status(void* ws, indexer_stream_t stream) {
  if (!ws) return fail(INDEXER_ERR_NULL, "ws is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word != 0u) {
    e = cudaMemsetAsync(ws, 0, sizeof(word), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    if (word & kStatusBadMeta)
      return fail(INDEXER_ERR_RANGE, "device-side metadata out of range: a block-table entry, slot, position or "
                  "row table was invalid and its keys or rows were skipped (status 0x%x)", word);
    return fail(INDEXER_ERR_DEVICE_TIMEOUT, "device wait ran out (status 0x%x)", word);
  }
  return ok();
}

}  // extern "C"

namespace indexer {
int check_forward_args(const IndexerDims* dims, const uint16_t* q, const uint16_t* w, int B, int S, int start_pos,
                       const float* rope_cs, int max_pos, const uint8_t* k_cache, int T_cap, const int32_t* cand_in,
                       const int32_t* cand_out, const int32_t* topk_out, const float* scores_out, const void* ws,
                       size_t ws_bytes) {
  return check_forward(dims, q, w, B, S, start_pos, rope_cs, max_pos, k_cache, T_cap, cand_in, cand_out, topk_out,
                       scores_out, ws, ws_bytes);
}
}  // namespace indexer
