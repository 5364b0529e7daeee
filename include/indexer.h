/*
 * indexer.h -- C ABI of the GB300 (sm_103a) DeepSeek-V4.1 compressed-attention
 * indexer: fp4 index-key publish, query prep, ReLU-weighted head-sum scoring with
 * the causal mask, the two-level candidate-block filter and the position-ordered
 * top-k.
 *
 * Sources (cited by page title and section):
 *   [index-keys]  DeepSeek V4.1 / ... / attention / indexer / index-keys page:
 *                 class Indexer (__init__, forward), SharedAttentionRuntime.
 *   [compress]    "Module compress" API page (spark_model deepseek_v41_ref):
 *                 fp4_quant_e8m0_inplace, to_e2m1_rne, yarn_freqs_cis,
 *                 select_candidate_blocks, precision policy.
 *   [attention.py] launcher/docker-images/dsv41-flash/patches/attention.py:
 *                 _indexer_k_cache_head_dim (68-byte MXFP4 row),
 *                 _fill_short_context_topk_indices, DeepseekV4Indexer.forward.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are caller-owned DEVICE memory unless stated otherwise.
 *     The library never allocates, frees or keeps device memory, and keeps no
 *     state between calls other than a thread-local error message.
 *   - bf16 tensors are passed as their 16-bit patterns (indexer_bf16).
 *   - Every call validates its arguments on the host before launching anything;
 *     on failure it returns a negative INDEXER_ERR_* code, launches nothing and
 *     sets indexer_last_error(). On success it returns INDEXER_OK after enqueuing
 *     its kernels on `stream` (asynchronous; no implicit synchronisation).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Sizes: B sequences, S query rows per sequence (all at the same start_pos),
 *     H = n_heads, D = head_dim = 128, rd = rope_dim, r = ratio,
 *     T = (start_pos + S) / r keys visible to the last row,
 *     vis(s) = (start_pos + s + 1) / r keys visible to row s (compress_lens).
 *   - Every quantised 128-vector (a key, or a query head) is 68 bytes: 64 bytes of
 *     packed e2m1 codes (element 2i in the low nibble of byte i, 2i+1 in the high
 *     nibble, sign in bit 3 of each nibble) and 4 UE8M0 scale bytes, one per block of
 *     32 values, block 0 in the lowest byte ([attention.py] _indexer_k_cache_head_dim:
 *     64 + 4 = 68). Query rows (q_rows) are stored as such 68-byte rows.
 *   - Keys live in pages of 64 keys (INDEXER_PAGE_KEYS), INDEXER_PAGE_BYTES = 4352
 *     bytes each, still 68 bytes per key. A page is 8 groups of 8 keys, 544 bytes per
 *     group: the group's 512 code bytes, then its keys' 4-byte scale words. Key m's
 *     code byte j sits at
 *         (m/8)*544 + (j/16)*128 + (m%8)*16 + (j%16)
 *     -- the tensor cores' K-major core-matrix order, so two pages side by side are one
 *     128-row MMA operand as they lie -- and its scale word at
 *         (m/8)*544 + 512 + (m%8)*4
 *     (the scale of block i in byte i). Two ways to hold them:
 *       * sequence-major: k_cache[B][T_cap/64][4352], sequence b's key t in page t/64
 *         of its own run (T_cap a multiple of 64, k_cache 16-byte aligned);
 *       * a page pool k_pool[num_pages][4352] shared by many sequences, with a block
 *         table giving each sequence's pages (the paged entry points below); slot x of
 *         the pool is key x % 64 of page x / 64.
 *   - FP8 rows (key_format = INDEXER_KEY_FP8; the attention.py page's FP8 indexer cache,
 *     "128 fp8 + 4 fp32 scale" = 132 bytes, scale_fmt ue8m0, block 128): 128 e4m3 codes
 *     (element i in byte i) then an f32 scale 2^e, e the power-of-two ceiling of
 *     amax / 448 with amax floored at 448 * 2^-126; codes round x / 2^e to nearest even,
 *     keeping the sign. Query heads use the same row. FP8 pages hold 64 keys in 8448
 *     bytes as 8 groups of 1056: the group's 1024 code bytes (key m's byte j at
 *     (m/8)*1056 + (j/16)*128 + (m%8)*16 + j%16), then its keys' f32 scales at
 *     (m/8)*1056 + 1024 + (m%8)*4. Every cache and q_rows buffer takes the row and page
 *     size of dims->key_format; the score is sum_h w' * relu(s_q * s_k * qcodes . kcodes).
 *   - Score buffers that the selection kernels read (scores of indexer_topk and
 *     indexer_select_candidate_blocks, scores_out of the forward calls) are 16-byte
 *     aligned.
 *   - Device-side waits are bounded: a kernel whose wait runs out sets a bit in
 *     the status word at the start of the workspace (indexer_status reads it).
 */
#ifndef INDEXER_H_
#define INDEXER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t indexer_bf16;          /* bf16 bit pattern */
typedef struct CUstream_st* indexer_stream_t;   /* == cudaStream_t */

#define INDEXER_OK                 0
#define INDEXER_ERR_NULL          -1   /* a required pointer is NULL */
#define INDEXER_ERR_ALIGN         -2   /* a pointer or stride breaks its alignment rule */
#define INDEXER_ERR_DIMS          -3   /* unsupported n_heads / head_dim / rope_dim / ratio / sizes */
#define INDEXER_ERR_RANGE         -4   /* positions, T > T_cap, table too short, bad start_pos */
#define INDEXER_ERR_WORKSPACE     -5   /* workspace smaller than indexer_workspace_size() */
#define INDEXER_ERR_ARCH          -6   /* current device is not sm_103 */
#define INDEXER_ERR_CUDA          -7   /* a CUDA runtime call or launch failed */
#define INDEXER_ERR_DEVICE_TIMEOUT -8  /* a bounded device-side wait ran out (indexer_status) */
/* indexer_status also returns INDEXER_ERR_RANGE when device-side metadata (a block table,
 * slot mapping, positions or row table) was out of range; the affected keys or rows were
 * skipped */

#define INDEXER_KEY_ROW_BYTES 68
#define INDEXER_PAGE_KEYS 64
#define INDEXER_PAGE_BYTES 4352        /* 64 keys x 68 bytes */
#define INDEXER_KEY_MXFP4 0
#define INDEXER_KEY_FP8 1
#define INDEXER_KEY_ROW_BYTES_FP8 132
#define INDEXER_PAGE_BYTES_FP8 8448    /* 64 keys x 132 bytes */
#define INDEXER_STATUS_BYTES 256       /* workspace header holding the status word */

/* Indexer shape and selection parameters ([index-keys] Indexer.__init__). */
typedef struct IndexerDims {
    int32_t n_heads;           /* H = index_n_heads: 8, 16, 32, 64 or 128 */
    int32_t head_dim;          /* D = index_head_dim: must be 128 */
    int32_t rope_dim;          /* rd = rope_head_dim: even, 2..128 (RoPE on the last rd dims) */
    int32_t ratio;             /* compress_ratio >= 1 */
    int32_t index_topk;        /* output width (columns beyond min(topk, T) are -1) */
    int32_t offset;            /* added to every emitted position */
    int32_t cand_topk_blocks;  /* level one: blocks kept (0: no two-level filter) */
    int32_t cand_block_size;   /* level one: compressed positions per block */
    float norm_eps;            /* k_norm RMSNorm epsilon */
    int32_t key_format;        /* INDEXER_KEY_MXFP4 (0) or INDEXER_KEY_FP8 (1): the row format of
                                  keys and quantised queries, see below */
    int32_t n_heads_total;     /* 0, or the model's index_n_heads when this call holds only a shard
                                  of n_heads of them (head-parallel scoring: [index-keys]
                                  Indexer.__init__ n_local_heads = index_n_heads // world_size, the
                                  head weights still scaled by index_n_heads^-0.5, and
                                  Indexer.forward all-reduces the partial scores); >= n_heads */
} IndexerDims;

/* YaRN parameters of the compressed layers ([compress] yarn_freqs_cis). */
typedef struct IndexerYarn {
    double theta;              /* compress_rope_theta */
    double factor;             /* YaRN scaling factor */
    int32_t original_seq_len;  /* YaRN applies when > 0 */
    double beta_fast;
    double beta_slow;
} IndexerYarn;

/* ---------------------------------------------------------------------------
 * indexer_rope_table -- the RoPE table freqs_cis as (cos, sin) pairs.
 * [compress] yarn_freqs_cis: precompute_freqs_cis WITH YaRN (original_seq_len > 0),
 * [seqlen][dim/2] of (cos, sin); the cos_sin_cache the fused ops of [attention.py]
 * take. NTK-by-parts YaRN: f_i = theta^(-2i/rd), ramp between the correction dims
 * of beta_fast and beta_slow, f'_i = f_i/factor*ramp + f_i*(1-ramp), rounded to f32;
 * angle = f32(pos) * f'_i in f32; cos/sin of that angle evaluated in f64 and
 * rounded to f32.
 *   table: device float[max_pos][rope_dim/2][2] (cos, sin), written.
 *   max_pos >= 1; rope_dim even in [2, 128].
 * ------------------------------------------------------------------------- */
int indexer_rope_table(const IndexerYarn* yarn, int rope_dim, int max_pos, float* table,
                       indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_publish_k -- index-key publish ([index-keys] Indexer.forward, the
 * owns_k branch; [attention.py] DeepseekV4Indexer._produce_k):
 *   k = wk(latent)           bf16 Linear, exact sum rounded once to bf16
 *   k = k_norm(k)            RMSNorm: bf16(w * k / sqrt(mean(k^2) + eps)), f64
 *   RoPE(k[..., -rd:])       interleaved pairs, f32 rotation, rounded to bf16
 *   fp4_act_quant(k, 32)     e2m1 (RNE, ties to even code) with e8m0 scales
 *   key slot s of sequence b: page s / 64, key s % 64 of k_cache[b]
 * Slots: start_pos == 0 (prefill) writes slots 0..G-1, group j at RoPE position
 * j*r; start_pos > 0 (decode) needs G == 1 and (start_pos + 1) % r == 0 and
 * writes slot start_pos / r at position start_pos + 1 - r.
 *   latent:   bf16 [B][G][Din], 16-byte aligned, Din a multiple of 8 in [8, 1024]
 *   wk:       bf16 [D][Din] (row o produces output dim o), 16-byte aligned
 *   k_norm_w: bf16 [D]
 *   rope_cs:  float [max_pos][rd/2][2]; every used position must be < max_pos
 *   k_cache:  uint8 [B][T_cap/64][4352] (sequence-major, see above); last slot < T_cap
 * ------------------------------------------------------------------------- */
int indexer_publish_k(const IndexerDims* dims, const indexer_bf16* latent, int B, int G, int Din,
                      const indexer_bf16* wk, const indexer_bf16* k_norm_w, const float* rope_cs,
                      int max_pos, int start_pos, uint8_t* k_cache, int T_cap, indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_prep_q -- query prep ([index-keys] Indexer.forward: RoPE at the query's
 * own position start_pos + s, fp4_act_quant; weights_proj(x) * softmax_scale *
 * n_heads^-0.5 with softmax_scale = head_dim^-0.5; [attention.py]
 * fused_indexer_q_rope_quant):
 *   q:       bf16 [B][S][H][128] (post wq_b, pre-RoPE), 16-byte aligned
 *   w:       bf16 [B][S][H] (weights_proj output)
 *   q_rows:  uint8 [B][S][H][68] quantised query rows (same row format as keys), 16-byte
 *            aligned
 *   w_prime: float [B][S][H] = w * 128^-0.5 * H^-0.5 (f32)
 * Head-parallel: with dims->n_heads_total set, q and w hold this call's n_heads heads and
 *   w' = w * 128^-0.5 * n_heads_total^-0.5, so the scores of indexer_scores are this
 *   shard's part of the head sum; the shards' scores add up (an all-reduce) to the full
 *   score, masked entries staying -inf, before indexer_topk.
 * ------------------------------------------------------------------------- */
int indexer_prep_q(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                   int start_pos, const float* rope_cs, int max_pos, uint8_t* q_rows, float* w_prime,
                   indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_prep_q_proj -- the query projection fused with query prep ([index-keys]
 * Indexer.forward: q = wq_b(qr) unflattened to [H][128], then the same RoPE and
 * fp4_act_quant as indexer_prep_q; weights_proj output scaled as there). Reading: wq_b
 * is a bf16 Linear (no bias); its output is the f32 tensor-core accumulation of the
 * exact bf16 products, rounded once to bf16 (the order of the f32 sums is the
 * hardware's, so a q value can differ from the exactly rounded sum by one bf16 unit where
 * the sum lies within f32 rounding of a bf16 midpoint); the quantised rows are those of
 * that q. The bf16 q never goes through global memory unless q_out is given.
 *   qr:      bf16 [B][S][Kq] (Kq = q_lora_rank, a multiple of 64 in [64, 16384]), 16-byte
 *            aligned
 *   wq_b:    bf16 [H * 128][Kq] (row o produces feature o = head * 128 + dim), 16-byte aligned
 *   w:       bf16 [B][S][H] (weights_proj output)
 *   q_rows:  uint8 [B][S][H][68], 16-byte aligned; w_prime: float [B][S][H]
 *   q_out:   bf16 [B][S][H][128] (the projection before RoPE, for checks) or NULL
 *   ws/ws_bytes: status word (INDEXER_STATUS_BYTES), initialised by indexer_workspace_init
 * MXFP4 query rows only (INDEXER_ERR_DIMS for key_format FP8); n_heads even.
 * ------------------------------------------------------------------------- */
int indexer_prep_q_proj(const IndexerDims* dims, const indexer_bf16* qr, int Kq, const indexer_bf16* wq_b,
                        const indexer_bf16* w, int B, int S, int start_pos, const float* rope_cs, int max_pos,
                        uint8_t* q_rows, float* w_prime, indexer_bf16* q_out, void* ws, size_t ws_bytes,
                        indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_compress_weights -- the producers upstream of the key publish and the query prep,
 * from one pass over the hidden states x (B sequences of S tokens, S a multiple of ratio):
 *   latent   = Compressor(x): kv = x Wkv^T and score = x Wgate^T per token (f32 tensor-core
 *              sums of bf16 products; [attention.py] compressor_kv_score, fused_wkv_wgate),
 *              per latent dim the softmax over each group's ratio tokens of score weighting kv
 *              ([compress] compressor: softmax pooling of ratio tokens, a plain projection at
 *              ratio 1), then RMSNorm(norm_w, dims->norm_eps) rounded to bf16 (the
 *              compressor is f32 until its RMSNorm casts to bf16); the pre-RoPE latent that
 *              indexer_publish_k takes;
 *   latent_q = the latent through [compress] fp4_quant_e4m3_inplace (LATENT_BLOCK 16, amax
 *              floored at 6 * 2^-9, scale amax / 6 rounded through e4m3, e2m1 values),
 *              dequantised back to bf16 (the compressed KV the attention layer keeps);
 *   w_out    = weights_proj(x) ([index-keys] Indexer.__init__, a bf16 Linear dim -> n_heads),
 *              the f32 accumulation rounded once to bf16; indexer_prep_q's w.
 *   x:        bf16 [B][S][dim], dim a multiple of 64 in [64, 65536], 16-byte aligned
 *   wkv, wgate: bf16 [128][dim] (the two halves of fused_wkv_wgate); norm_w: bf16 [128]
 *   wproj:    bf16 [n_heads][dim]
 *   latent, latent_q: bf16 [B][S / ratio][128] (latent_q may be NULL)
 *   w_out:    bf16 [B][S][n_heads]
 *   ws/ws_bytes: status word (INDEXER_STATUS_BYTES), initialised by indexer_workspace_init
 * ratio must be 1, 2, 4, 8, 16 or 32 (a group's tokens share one warp).
 * ------------------------------------------------------------------------- */
int indexer_compress_weights(const IndexerDims* dims, const indexer_bf16* x, int B, int S, int dim,
                             const indexer_bf16* wkv, const indexer_bf16* wgate, const indexer_bf16* norm_w,
                             const indexer_bf16* wproj, indexer_bf16* latent, indexer_bf16* latent_q,
                             indexer_bf16* w_out, void* ws, size_t ws_bytes, indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_scores -- index scores of prepared queries against the key cache
 * ([index-keys] Indexer.forward: einsum("bshd,btd->bsht"), relu, * weights,
 * sum over heads; causal mask t >= vis(s) -> -inf; level two: -inf outside the
 * candidate blocks):
 *   score[b][s][t] = sum_h w'[b,s,h] * relu(sum_d qhat[b,s,h,d] * khat[b,t,d])
 * over the dequantised fp4 values, products exact, f32 accumulation.
 *   q_rows/w_prime as written by indexer_prep_q (both 16-byte aligned)
 *   k_cache/T_cap: the sequence-major key cache (T_cap a multiple of 64)
 *   cand_blocks: int32 [B][S][cand_topk_blocks] kept block ids (-1 = none), or
 *                NULL for no candidate filter
 *   scores: float [B][S][T] written (T = (start_pos + S) / r)
 *   ws/ws_bytes: workspace of at least INDEXER_STATUS_BYTES (the status word and the
 *                scoring kernels' work counter), initialised once by indexer_workspace_init
 * ------------------------------------------------------------------------- */
int indexer_scores(const IndexerDims* dims, const uint8_t* q_rows, const float* w_prime, int B, int S,
                   int start_pos, const uint8_t* k_cache, int T_cap, const int32_t* cand_blocks,
                   float* scores, void* ws, size_t ws_bytes, indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_select_candidate_blocks -- level one of the two-level top-k
 * ([compress] select_candidate_blocks; [index-keys] Indexer.forward). The pages
 * give the signature only; this library's reading: blocks of cand_block_size
 * positions, a block is eligible when it holds a position t < vis(s) with a
 * finite score, its score is the max of those, the cand_topk_blocks best
 * eligible blocks are kept (ties to the lower block index).
 *   scores: float [B][S][T] as written by indexer_scores
 *   blocks_out: int32 [B][S][cand_topk_blocks], kept block ids ascending, -1 pad
 *   Needs T / cand_block_size + 1 <= 8192 blocks.
 * ------------------------------------------------------------------------- */
int indexer_select_candidate_blocks(const IndexerDims* dims, const float* scores, int B, int S,
                                    int start_pos, int T, int32_t* blocks_out, indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_topk -- top-k by score re-sorted into position order, offset added,
 * -1 where unreachable ([index-keys] Indexer.forward, last three lines;
 * [attention.py] topk_indices_buffer width and _fill_short_context_topk_indices).
 * k_eff = min(index_topk, T). Among the finite scores at t < vis(s) the k_eff
 * largest are kept (ties to the lower position) and written ascending as
 * t + offset, then -1 up to index_topk columns. Rows with vis(s) <= k_eff
 * and all scores finite reduce to [0 .. vis) + offset (short-context rule).
 *   scores: float [B][S][T]; out: int32 [B][S][index_topk]
 *   T <= 32768.
 * ------------------------------------------------------------------------- */
int indexer_topk(const IndexerDims* dims, const float* scores, int B, int S, int start_pos, int T,
                 int32_t* out, indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_forward -- the whole hot path after the key publish: query prep,
 * scores, causal mask, optional level-one candidate publication (cand_out,
 * the candidate source layer) or level-two filter (cand_in, a consumer layer),
 * and the top-k ([index-keys] Indexer.forward). Either candidate pointer may be
 * NULL; both non-NULL is allowed (filter by cand_in, publish from the
 * unfiltered scores).
 *   q, w, rope_cs, max_pos: as indexer_prep_q
 *   k_cache, T_cap:         as indexer_scores
 *   cand_in / cand_out:     int32 [B][S][cand_topk_blocks] or NULL
 *   topk_out:               int32 [B][S][index_topk]
 *   scores_out:             float [B][S][T] or NULL (the masked scores), 16-byte aligned
 *   ws / ws_bytes:          workspace, at least indexer_workspace_size(),
 *                           initialised once by indexer_workspace_init
 * ------------------------------------------------------------------------- */
int indexer_forward(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                    int start_pos, const float* rope_cs, int max_pos, const uint8_t* k_cache, int T_cap,
                    const int32_t* cand_in, int32_t* cand_out, int32_t* topk_out, float* scores_out,
                    void* ws, size_t ws_bytes, indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_forward_publish -- indexer_publish_k followed by indexer_forward, in one call
 * ([index-keys] Indexer.forward publishes the keys its tokens complete before scoring;
 * [attention.py] DeepseekV4Indexer.forward: _produce_k, then the query path). The step's
 * keys are written before any score is computed. The publish and the query prep are
 * independent, so for a decode step (at most 160 keys and 16384 query-head vectors)
 * they run in one launch. Arguments: those of indexer_publish_k (latent [B][G][Din], wk,
 * k_norm_w, the start_pos rule for G) and of indexer_forward; k_cache is written.
 * ------------------------------------------------------------------------- */
int indexer_forward_publish(const IndexerDims* dims, const indexer_bf16* latent, int G, int Din,
                            const indexer_bf16* wk, const indexer_bf16* k_norm_w, const indexer_bf16* q,
                            const indexer_bf16* w, int B, int S, int start_pos, const float* rope_cs, int max_pos,
                            uint8_t* k_cache, int T_cap, const int32_t* cand_in, int32_t* cand_out,
                            int32_t* topk_out, float* scores_out, void* ws, size_t ws_bytes,
                            indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_forward_publish_host -- indexer_forward_publish with the step's inputs and
 * its top-k in HOST memory: the call copies latent, q and w to device staging inside the
 * workspace, runs the step and copies the indices back, all on `stream` (pinned host
 * buffers let the copies run asynchronously; topk_out_h is valid once the stream has
 * reached the call's end). Arguments as indexer_forward_publish, with:
 *   latent_h: bf16 [B][G][Din], q_h: bf16 [B][S][H][128], w_h: bf16 [B][S][H] (host);
 *             G == 0 (a decode token that completes no group): no key is published, the
 *             step is indexer_forward, and latent_h may be NULL
 *   topk_out_h: int32 [B][S][index_topk] (host)
 *   ws/ws_bytes: at least indexer_workspace_size_host() bytes, 256-byte aligned,
 *                initialised once by indexer_workspace_init
 * No candidate filter and no score output (use indexer_forward_publish for those).
 * ------------------------------------------------------------------------- */
size_t indexer_workspace_size_host(const IndexerDims* dims, int B, int S, int start_pos, int G, int Din);
int indexer_forward_publish_host(const IndexerDims* dims, const indexer_bf16* latent_h, int G, int Din,
                                 const indexer_bf16* wk, const indexer_bf16* k_norm_w, const indexer_bf16* q_h,
                                 const indexer_bf16* w_h, int B, int S, int start_pos, const float* rope_cs,
                                 int max_pos, uint8_t* k_cache, int T_cap, int32_t* topk_out_h, void* ws,
                                 size_t ws_bytes, indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * indexer_forward_noalloc -- indexer_forward for callers that cannot allocate
 * device memory at call time. The pages have no counterpart: this is a deployment
 * convenience of the library. Some hosts own all of the device's memory -- a
 * plugin inside another runtime's memory pool, or a server whose memory budget is
 * fixed at start-up -- and cannot hand this library a workspace. This entry point
 * takes the same arguments as indexer_forward minus the workspace and uses a fixed
 * scratch array inside the library's device memory instead:
 *   - the scratch holds INDEXER_NOALLOC_SCRATCH_BYTES (8 MiB); sizes whose
 *     indexer_workspace_size() exceeds it are rejected with INDEXER_ERR_WORKSPACE
 *     and a message naming both sizes (nothing is launched);
 *   - every GPU that loads the library keeps that array until the process exits;
 *   - the first call on a device, with that device current, looks up the array's
 *     device address (cudaGetSymbolAddress); make that first call before any stream
 *     capture. The call allocates nothing and never calls cudaMalloc or cudaFree;
 *   - all calls share the one array: calls that may run at the same time on the GPU
 *     (different streams or host threads without ordering) race on it and must not
 *     be issued; each call clears the status word it starts from;
 *   - arguments are checked before anything is enqueued: a rejected call does not
 *     touch the array;
 *   - the array's address stays valid for the life of the process; after a
 *     cudaDeviceReset the module holding it is gone, so do not call this entry point
 *     on that device again;
 *   - device-wait timeouts set the status word at the start of the array; read it
 *     with indexer_noalloc_status.
 * ------------------------------------------------------------------------- */
#define INDEXER_NOALLOC_SCRATCH_BYTES (8 * 1024 * 1024)
int indexer_forward_noalloc(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int B, int S,
                            int start_pos, const float* rope_cs, int max_pos, const uint8_t* k_cache, int T_cap,
                            const int32_t* cand_in, int32_t* cand_out, int32_t* topk_out, float* scores_out,
                            indexer_stream_t stream);

/* indexer_noalloc_status -- the status word of indexer_forward_noalloc's static array on
 * the current device (no counterpart on the pages): synchronises `stream`, reads and clears
 * the word, and returns INDEXER_OK, INDEXER_ERR_DEVICE_TIMEOUT or INDEXER_ERR_RANGE as
 * indexer_status does for a workspace. Allocates nothing. */
int indexer_noalloc_status(indexer_stream_t stream);

/* ---------------------------------------------------------------------------
 * Page pool and mixed batches: a server's form of the same path ([attention.py]
 * DeepseekV4IndexerCache: paged indexer cache of 64-state pages through a slot
 * mapping; DeepseekV4Indexer.forward over batches that mix decode rows and prefill
 * chunks). All per-key and per-sequence metadata is DEVICE memory, read by the kernels,
 * so the calls can be captured in a CUDA graph; the host passes bounds only. Metadata
 * that is out of range is not dereferenced: the kernel skips the key or row and sets a
 * status bit that indexer_status reports as INDEXER_ERR_RANGE.
 * ------------------------------------------------------------------------- */

/* indexer_publish_k_paged -- the key publish of indexer_publish_k for N keys that each
 * name their own pool slot and RoPE position:
 *   latent:       bf16 [N][Din], 16-byte aligned (Din a multiple of 8 in [8, 1024])
 *   positions:    int32 [N], RoPE position of key i (in [0, max_pos))
 *   slot_mapping: int32 [N], pool slot of key i (page * 64 + key in page); < 0: skipped
 *   k_pool:       uint8 [num_pages][4352], 16-byte aligned
 *   ws/ws_bytes:  status word (INDEXER_STATUS_BYTES), initialised by indexer_workspace_init */
int indexer_publish_k_paged(const IndexerDims* dims, const indexer_bf16* latent, int N, int Din,
                            const indexer_bf16* wk, const indexer_bf16* k_norm_w, const float* rope_cs, int max_pos,
                            const int32_t* positions, const int32_t* slot_mapping, uint8_t* k_pool, int num_pages,
                            void* ws, size_t ws_bytes, indexer_stream_t stream);

/* indexer_forward_paged -- indexer_forward over a batch of n_seq sequences with their own
 * start positions and query-row counts, keys in a page pool:
 *   q:           bf16 [Q][H][128] query rows of all sequences, 16-byte aligned
 *   w:           bf16 [Q][H]
 *   seq_pos:     int32 [n_seq], start_pos of each sequence
 *   q_start:     int32 [n_seq + 1], ascending; sequence b owns rows q_start[b] ..
 *                q_start[b+1]-1, its row s at position seq_pos[b] + s, and sees
 *                T_b = (seq_pos[b] + S_b) / ratio keys, row s vis(s) of them
 *   T_max:       a bound on every T_b (the row width of scores_out), <= 32768
 *   k_pool:      uint8 [num_pages][4352]
 *   block_table: int32 [n_seq][bt_stride], pool page of each of a sequence's logical
 *                pages (key t in logical page t / 64); bt_stride >= ceil(T_max / 64)
 *   cand_in / cand_out: int32 [Q][cand_topk_blocks] or NULL (as indexer_forward)
 *   topk_out:    int32 [Q][index_topk]
 *   scores_out:  float [Q][T_max] or NULL; positions >= T_b of a row are not written
 *   ws/ws_bytes: workspace of at least indexer_workspace_size_paged(), initialised once
 * Rows that no sequence owns (q_start[0] > 0 or q_start[n_seq] < Q) get all -1. At most
 * 4096 sequences per call. */
int indexer_forward_paged(const IndexerDims* dims, const indexer_bf16* q, const indexer_bf16* w, int Q, int n_seq,
                          const int32_t* seq_pos, const int32_t* q_start, int T_max, const float* rope_cs,
                          int max_pos, const uint8_t* k_pool, int num_pages, const int32_t* block_table,
                          int bt_stride, const int32_t* cand_in, int32_t* cand_out, int32_t* topk_out,
                          float* scores_out, void* ws, size_t ws_bytes, indexer_stream_t stream);

/* Bytes of workspace indexer_forward_paged needs (0 on invalid sizes). Layout: status
 * header, quantised query rows, head weights, f32 scores [Q][T_max], row metadata, row
 * groups. */
size_t indexer_workspace_size_paged(const IndexerDims* dims, int Q, int n_seq, int T_max);

/* ---------------------------------------------------------------------------
 * Row-major caches. The pages hold the indexer cache one row per compressed position:
 * [index-keys] Indexer.__init__ registers k_cache [max_batch_size][max_seq_len / ratio]
 * [index_head_dim]; [attention.py] DeepseekV4IndexerCache binds a [num_blocks]
 * [block_size][68] (MXFP4) or [..][132] (FP8) tensor, _indexer_k_cache_head_dim giving
 * the row width. These two calls move keys between that row-major form and this
 * library's 64-key pages (a pure byte permutation, bit-exact both ways), so a caller
 * holding such a cache can use every other entry point:
 *   rows:    uint8 [n_seq][ld_rows][row bytes] (68 or 132 by dims->key_format), 4-byte
 *            aligned; key t of sequence b is row b * ld_rows + t
 *   k_cache: uint8 [n_seq][T_cap / 64][page bytes], 16-byte aligned (a page pool
 *            [num_pages][page bytes] is n_seq = num_pages, T_cap = ld_rows = 64)
 *   n_keys:  keys 0 .. n_keys-1 of every sequence are moved (n_keys <= T_cap, <= ld_rows);
 *            the other keys of the destination are left as they are.
 * ------------------------------------------------------------------------- */
int indexer_cache_from_rows(const IndexerDims* dims, const uint8_t* rows, int n_seq, int n_keys, int ld_rows,
                            uint8_t* k_cache, int T_cap, indexer_stream_t stream);
int indexer_cache_to_rows(const IndexerDims* dims, const uint8_t* k_cache, int T_cap, int n_seq, int n_keys,
                          uint8_t* rows, int ld_rows, indexer_stream_t stream);

/* Bytes of workspace indexer_forward needs for these sizes (0 on invalid dims).
 * Layout: status header, quantised query rows, head weights, f32 scores. */
size_t indexer_workspace_size(const IndexerDims* dims, int B, int S, int start_pos);

/* Zeroes the status word at the start of a workspace (enqueued on `stream`). A
 * workspace must be initialised once before its first use; kernels only ever OR
 * bits into the word, and indexer_status clears it when it reads it. */
int indexer_workspace_init(void* ws, size_t ws_bytes, indexer_stream_t stream);

/* Synchronises `stream`, reads and clears the status word of `ws` and returns
 * INDEXER_OK or INDEXER_ERR_DEVICE_TIMEOUT. For tests and diagnostics. */
int indexer_status(void* ws, indexer_stream_t stream);

/* indexer_scores_hold_test -- for tests of the bounded device waits only (no counterpart
 * on the pages). Launches the several-row score kernel of indexer_scores (S >= 2, no
 * candidate filter) with its producer role held back: no query row, key tile or MMA is
 * ever requested, so every other role's wait runs out after wait_ns nanoseconds (1e3 ..
 * 1e9). The kernel records the timeout in the status word of `ws` (indexer_status then
 * returns INDEXER_ERR_DEVICE_TIMEOUT), frees its tensor memory and returns with nothing in
 * flight; `scores` is not written. Arguments otherwise as indexer_scores. */
int indexer_scores_hold_test(const IndexerDims* dims, const uint8_t* q_rows, const float* w_prime, int B, int S,
                             int start_pos, const uint8_t* k_cache, int T_cap, float* scores, void* ws,
                             size_t ws_bytes, uint64_t wait_ns, indexer_stream_t stream);

/* Message of the last failure on this thread ("" if none). */
const char* indexer_last_error(void);

/* ABI version (major * 100 + minor). */
int indexer_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* INDEXER_H_ */
