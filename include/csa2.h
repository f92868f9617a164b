/*
 * csa2.h - C ABI of the CSA2 compressed-sparse-attention step on one GB300
 * (sm_103a) GPU.
 *
 * The step follows the method described in "Reading Notes of
 * DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
 * section 3f, component C2 (steps 1-4), together with "DeepSeek-V4.1-Flash
 * on WASTE", section "What is new", item 1, and the PocketLLM page
 * "DeepSeek-V4.1-Flash", section "The CSA2 attention layers". One layer step
 * of a query at position t is:
 *
 *   compress     m raw KV vectors of a closed group -> one stored entry
 *   index_score  sigma(j) = sum_h w_h * relu(q^I_h . k^I_j) over visible j
 *   topk         the K largest sigma, ties to the lower index
 *   attend       one softmax with a per-head sink over the window rows
 *                [max(lo, t-w+1), t] and the selected entries
 *
 * Conventions for every entry point:
 *   - Every array argument is a DEVICE pointer into memory the caller owns
 *     (PyTorch allocates it), unless the comment says "host".
 *   - Rows are row-major with the last axis contiguous. bf16 values travel as
 *     uint16_t bit patterns. The fp8 format (CSA2_KV_FP8_E4M3_B32) stores one
 *     e4m3 byte per channel plus one ue8m0 scale byte (value 2^(E-127)) per 32
 *     consecutive channels, in a separate [rows, dim/32] byte array. The fp4
 *     formats store E2M1 codes (grid 0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6)
 *     two per byte, the even channel in the low nibble ([rows, dim/2] bytes):
 *     CSA2_KV_FP4_E4M3_B16 with one e4m3 scale byte per 16 channels
 *     ([rows, dim/16]), the scale e4m3(max(amax, 6*2^-9) / 6); CSA2_KV_MXFP4_B32
 *     with one ue8m0 scale byte per 32 channels ([rows, dim/32]), the scale
 *     2^round(log2(max(amax, 6*2^-126) / 6)) ("Reading Notes ...", 3f C4;
 *     PocketLLM page, "The op layer"). Codes round to the nearest grid value,
 *     ties to the even code, saturating at +-6.
 *   - `stream` is a cudaStream_t passed as void*; every call only enqueues
 *     work on it (asynchronous, stream-ordered) and returns after host-side
 *     argument validation.
 *   - Nothing here aborts or traps. Host-side validation failures return
 *     CSA2_ERR_INVALID_ARG / CSA2_ERR_UNSUPPORTED without enqueuing anything.
 *     Bad values found on the device (an index outside its pool, a window
 *     position outside its buffer, n_vis larger than the pool, a segment not
 *     made of whole groups) are skipped by the kernels, which record a bit in
 *     a device error word; csa2_check() synchronises and reports it.
 *   - The library allocates device memory only inside csa2_create (two
 *     small buffers: the device error word and the index scan's two 64-bit
 *     work counters). Scratch space is the caller's `workspace`, whose size the
 *     *_workspace_size functions give; it must be 256-byte aligned. The one
 *     exception is csa2_attend_noalloc, whose scratch is a fixed device array
 *     owned by the library (see its comment).
 *   - Strings returned by the library are owned by it.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned buffer    */
  CSA2_ERR_UNSUPPORTED = 2,  /* a geometry the kernels were not built for     */
  CSA2_ERR_CUDA = 3,         /* a CUDA runtime call failed (see last_error)   */
  CSA2_ERR_DEVICE_FLAG = 4,  /* a kernel recorded bad input (csa2_check)      */
  CSA2_ERR_TIMEOUT = 5,      /* a bounded device wait gave up (csa2_check)    */
  CSA2_ERR_WORKSPACE = 6     /* workspace too small                           */
} csa2_status;

/* Layer modes: "Reading Notes ...", section 3f, C2 step 4 (mode table). */
typedef enum csa2_mode {
  CSA2_MODE_FULL = 0,    /* compress own entries, score, select, attend      */
  CSA2_MODE_REINDEX = 1, /* borrowed pool and keys; own score + selection    */
  CSA2_MODE_REUSE = 2    /* borrowed pool and selection; attend only         */
} csa2_mode;

typedef enum csa2_kv_format {
  CSA2_KV_BF16 = 0,
  CSA2_KV_FP8_E4M3_B32 = 1, /* e4m3 codes + one ue8m0 scale per 32 channels */
  /* attention KV (kv_format) only: compressed pool rows fp4 with an e4m3
     scale per 16 channels; window rows stay fp8 (CSA2_KV_FP8_E4M3_B32), as
     the pages keep the sliding-window cache in FP8 ("Reading Notes ...", 3f C4) */
  CSA2_KV_FP4_E4M3_B16 = 2,
  /* index keys (idx_key_format) only: fp4 with a ue8m0 scale per 32 channels */
  CSA2_KV_MXFP4_B32 = 3
} csa2_kv_format;

/* Device error word bits (csa2_check / csa2_device_flags). */
#define CSA2_FLAG_BAD_TOPK_INDEX   0x01u /* selected index outside [0, pool length) */
#define CSA2_FLAG_BAD_WINDOW       0x02u /* window position outside its buffer      */
#define CSA2_FLAG_BAD_SEGMENT      0x04u /* compress segment not whole groups, or
                                            its entries fall outside the pool       */
#define CSA2_FLAG_NVIS_TOO_LARGE   0x08u /* n_vis larger than the sequence's pool   */
#define CSA2_FLAG_WAIT_TIMEOUT     0x10u /* a bounded mbarrier wait gave up         */
#define CSA2_FLAG_BAD_QUERY        0x20u /* seq_of_q outside [0, n_seq)             */

/* Geometry and numerics of one CSA2 layer ("DeepSeek-V4.1-Flash on WASTE",
 * section "The shape"; PocketLLM page, geometry table). Supported values:
 *   n_heads 64, head_dim 512, rope_dim 0 or 64 (the last rope_dim channels
 *   are rotated, adjacent pairs), window 1..128, compress_ratio 1..16,
 *   idx_heads 8/16/32, idx_dim 128, topk 1..2048 (multiple of 1),
 *   kv_format bf16 / fp8 / fp4-e4m3-b16, idx_key_format bf16 / fp8 / mxfp4.
 * softmax_scale multiplies q.k (1/sqrt(512)); the sink is a logit on the
 * same scale. RoPE frequencies follow YaRN (DeepSeek-V3 ramp): rope_theta,
 * yarn_factor (<= 1 disables the ramp), yarn_orig_len, yarn_beta_fast/slow. */
typedef struct csa2_config {
  int32_t n_heads;
  int32_t head_dim;
  int32_t rope_dim;
  int32_t window;
  int32_t compress_ratio;
  int32_t idx_heads;
  int32_t idx_dim;
  int32_t topk;
  int32_t kv_format;
  int32_t idx_key_format;
  float softmax_scale;
  float norm_eps;
  double rope_theta;
  double yarn_factor;
  double yarn_orig_len;
  double yarn_beta_fast;
  double yarn_beta_slow;
  /* hierarchical indexer ("Reading Notes ...", 3f C3): blocks of cand_block
   * consecutive entries (a power of two, 1..64; 8), of which the candidate
   * source keeps cand_keep (1..2048; 2048) as the pool */
  int32_t cand_block;
  int32_t cand_keep;
} csa2_config;

typedef struct csa2_ctx csa2_ctx;

/* Fills `cfg` (host) with the DeepSeek-V4.1-Flash compressed-layer defaults:
 * 64 x 512, rope 64, window 128, ratio 4, 8 x 128 indexer, top-512, bf16,
 * scale 1/sqrt(512), eps 1e-20, theta 160000, YaRN 16 over 65536, beta 32/1,
 * candidate blocks of 8, 2048 kept. */
void csa2_default_config(csa2_config* cfg);

/* Validates `cfg` (host), computes the RoPE frequencies in double precision
 * and allocates, on the current CUDA device, the device error word and the
 * index scan's two 64-bit work counters; it also creates the context's side
 * and copy streams and its events. The context is bound to that device; use
 * it from one host thread at a time.
 * One context's calls must not overlap on the GPU: every index scan of a
 * context (csa2_index_score, csa2_index_score_pool, csa2_step) draws work
 * from the context's one pair of counters, and csa2_step also uses the
 * context's side stream and events. Calls enqueued on one stream are
 * ordered and safe; to run work on several streams at once, give each
 * stream its own context. */
csa2_status csa2_create(const csa2_config* cfg, csa2_ctx** out);
void csa2_destroy(csa2_ctx* ctx);

/* Message of the last failure on this context (never NULL). */
const char* csa2_last_error(const csa2_ctx* ctx);
const char* csa2_status_string(csa2_status s);
/* Writes the ctx's RoPE frequencies (rope_dim/2 doubles) to `out` (host). */
csa2_status csa2_rope_frequencies(const csa2_ctx* ctx, double* out, int32_t n);

/* Synchronises `stream`, reads and clears the device error word; returns
 * CSA2_ERR_DEVICE_FLAG / CSA2_ERR_TIMEOUT if a kernel recorded bad input. The
 * word's bits are written to *flags_out (host, nullable). */
csa2_status csa2_check(csa2_ctx* ctx, void* stream, uint32_t* flags_out);

/* Test aid for the bounded device waits (no counterpart in the method):
 * enqueues one kernel whose single thread waits, with the same bounded
 * mbarrier wait the attention kernels use, on a barrier that nothing ever
 * arrives at. After limit_ns nanoseconds (host, 1 .. 1e9) the wait gives up,
 * records CSA2_FLAG_WAIT_TIMEOUT and the kernel returns: the next csa2_check
 * on the stream reports CSA2_ERR_TIMEOUT, and the context stays usable. */
csa2_status csa2_debug_wait_timeout(csa2_ctx* ctx, void* stream, uint64_t limit_ns);

/* ------------------------------------------------------------------------
 * csa2_store_rows: store fp32 rows in a KV storage format, optionally rotated.
 * Used to append window rows ("DeepSeek-V4.1-Flash on WASTE", item 1: the
 * window stores each position's KV already rotated) and to put index keys or
 * pool rows into the fp8 format (PocketLLM page, "The CSA2 attention layers":
 * the window is quantised to FP8 over 32 elements).
 *   rows     [n_rows, dim] fp32
 *   pos      [n_rows] int64, nullable: when given and rope_dim > 0 the last
 *            rope_dim channels of row i are rotated by angle pos[i]*f_k first
 *   format   csa2_kv_format; out [n_rows, dim] bf16 or e4m3 bytes,
 *            out_scale [n_rows, dim/32] ue8m0 bytes (fp8 only, else NULL)
 * dim must be 128 (index keys) or 512 (attention rows). */
csa2_status csa2_store_rows(csa2_ctx* ctx, void* stream, const float* rows, int64_t n_rows,
                            int32_t dim, const int64_t* pos, int32_t format, void* out,
                            uint8_t* out_scale);

/* ------------------------------------------------------------------------
 * csa2_compress: step 1 ("Reading Notes ...", 3f C2 step 1; WASTE item 1;
 * PocketLLM "The CSA2 attention layers"). For every closed group of m =
 * compress_ratio tokens: per-channel softmax of the gate logits over the
 * group, weighted sum of the raw vectors (fp32), RMSNorm with norm_w; the
 * index key RMSNorm_{k_norm_w}(c_hat . w_idx^T) from the unrotated c_hat;
 * then RoPE of c_hat at the group's first token position j*m; store both.
 *   raw        [n_tokens, 512] bf16 tokens, sequences packed by tok_off
 *   gate       [n_tokens, 512] fp32 gate logits (ignored, may be NULL, at m=1)
 *   tok_off    [n_seq+1] int64 token offsets; each segment a multiple of m
 *   first_pos  [n_seq] int64 position of each segment's first token (a
 *              multiple of m); group j of sequence b is written to pool row
 *              pool_off[b] + j, j = position / m
 *   pool_off   [n_seq+1] int64 pool row offsets
 *   norm_w     [512] fp32; w_idx [idx_dim, 512] bf16 (NULL: no index keys);
 *   k_norm_w   [idx_dim] fp32
 *   pool_kv / pool_kv_scale   rows in kv_format (scale NULL for bf16)
 *   idx_keys / idx_key_scale  rows in idx_key_format (both NULL if w_idx NULL)
 * n_tokens (host) is the total token count; 0 enqueues nothing. */
csa2_status csa2_compress(csa2_ctx* ctx, void* stream, const uint16_t* raw, const float* gate,
                          int32_t n_seq, int64_t n_tokens, const int64_t* tok_off,
                          const int64_t* first_pos, const int64_t* pool_off, const float* norm_w,
                          const uint16_t* w_idx, const float* k_norm_w, void* pool_kv,
                          uint8_t* pool_kv_scale, void* idx_keys, uint8_t* idx_key_scale);

/* ------------------------------------------------------------------------
 * csa2_compress_append: the compressor with its partial group carried in
 * state ("Reading Notes of DeepSeek-V4.1-Flash", 3f "the compressor": during
 * decode an entry is emitted only every compress_ratio steps and the partial
 * group waits in state; "DeepSeek-V4.1-Flash" (PocketLLM), "The container":
 * the trailing group waits between calls and a step that closes no group
 * writes nothing). Tokens arrive in any number per call and sequence:
 *   raw, gate  [n_tokens, 512] new tokens (bf16) and gate logits (fp32; NULL
 *              at m = 1), sequences packed by tok_off [n_seq+1] (any counts)
 *   first_pos  [n_seq] int64 position of sequence b's first new token (any
 *              position >= 0); its tokens have positions first_pos[b] ..
 *              first_pos[b] + n_b - 1
 *   state_raw  [n_seq, m, 512] bf16 and state_gate [n_seq, m, 512] fp32,
 *              caller-owned: the token at position p of a group still open
 *              lives in slot p mod m of its sequence. The tokens of b's open
 *              group (positions floor(first_pos[b]/m) m .. first_pos[b] - 1)
 *              must be there from earlier calls; NULL is allowed at m = 1.
 * Every group that this call completes, j with first_pos[b] < (j+1) m <=
 * first_pos[b] + n_b, is compressed exactly as csa2_compress does (same
 * arithmetic, so the same bits whatever the chunking) into pool row
 * pool_off[b] + j and its index key; then the new tokens of b's group still
 * open are written to the state. Two launches (the compress, then the state
 * store) on `stream`. Other arguments as for csa2_compress. */
csa2_status csa2_compress_append(csa2_ctx* ctx, void* stream, const uint16_t* raw, const float* gate,
                                 int32_t n_seq, int64_t n_tokens, const int64_t* tok_off,
                                 const int64_t* first_pos, const int64_t* pool_off, const float* norm_w,
                                 const uint16_t* w_idx, const float* k_norm_w, void* pool_kv,
                                 uint8_t* pool_kv_scale, void* idx_keys, uint8_t* idx_key_scale,
                                 uint16_t* state_raw, float* state_gate);

/* ------------------------------------------------------------------------
 * csa2_index_score: step 2 ("Reading Notes ...", 3f C2 step 2, the lightning
 * indexer form). scores[q, j] = sum_h w_heads[q,h] * max(0, q_idx[q,h,:] .
 * key_j) for j < n_vis[q], key_j = row pool_off[seq_of_q[q]] + j of idx_keys.
 * Entries j >= n_vis[q] of the scores row are not written.
 *   q_idx     [n_query, idx_heads, idx_dim] bf16
 *   w_heads   [n_query, idx_heads] fp32
 *   idx_keys  [pool rows, idx_dim] in idx_key_format; idx_key_scale its
 *             [rows, idx_dim/32] scales (fp8 only)
 *   pool_off  [n_seq+1] int64; seq_of_q [n_query] int32; n_vis [n_query] int32
 *   max_vis   (host) an upper bound of every n_vis[q]
 *   scores    [n_query, scores_ld] fp32, scores_ld >= max_vis
 * Products are exact (bf16 x bf16, or e4m3 codes), sums in fp32.
 * The scan hands out work through the context's counters: two index scans
 * of one context must not run at the same time on different streams. */
csa2_status csa2_index_score(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query,
                             const uint16_t* q_idx, const float* w_heads, const void* idx_keys,
                             const uint8_t* idx_key_scale, const int64_t* pool_off,
                             const int32_t* seq_of_q, const int32_t* n_vis, int64_t max_vis,
                             float* scores, int64_t scores_ld);

/* ------------------------------------------------------------------------
 * csa2_topk: step 2's selection S_t = TopK sigma_t ("Reading Notes ...", 3f
 * C2 step 2; PocketLLM "The CSA2 attention layers", -1 padding). For each
 * query: the min(k, n_vis[q]) largest of scores[q, 0:n_vis[q]], ties broken
 * toward the lower index, -0.0 equal to +0.0; written in ascending index
 * order to out_idx[q, 0:k], the rest -1. Scores must not be NaN.
 *   scores  [n_query, scores_ld] fp32; n_vis [n_query] int32
 *   k       1..2048; out_idx [n_query, k] int32
 *   max_vis (host) upper bound of n_vis
 *   workspace of csa2_topk_workspace_size(ctx, n_query, max_vis) bytes */
size_t csa2_topk_workspace_size(const csa2_ctx* ctx, int32_t n_query, int64_t max_vis);
csa2_status csa2_topk(csa2_ctx* ctx, void* stream, int32_t n_query, const float* scores,
                      int64_t scores_ld, const int32_t* n_vis, int64_t max_vis, int32_t k,
                      int32_t* out_idx, void* workspace, size_t workspace_bytes);

/* ------------------------------------------------------------------------
 * The hierarchical sparse indexer ("Reading Notes ...", 3f C3; PocketLLM
 * "DeepSeek-V4.1-Flash", "The container", select_candidate_blocks).
 *
 * csa2_candidate_pool: the first level, on the candidate source's scores
 * (csa2_index_score output). The n_vis[q] entries of query q fall into
 * blocks of B = cand_block consecutive entries; a block scores the largest
 * score among its entries; the block holding entry n_vis[q]-1 (still
 * filling) is pinned; the cand_keep best blocks by (score, lower block index)
 * form the pool, written to cand [n_query, cand_keep] as ascending block
 * indices, -1 padded. Bit-exact on given fp32 scores.
 *   scores [n_query, ld] fp32, n_vis [n_query] int32, max_vis (host bound)
 *   workspace: csa2_candidate_pool_workspace_size bytes */
size_t csa2_candidate_pool_workspace_size(const csa2_ctx* ctx, int32_t n_query, int64_t max_vis);
csa2_status csa2_candidate_pool(csa2_ctx* ctx, void* stream, int32_t n_query, const float* scores,
                                int64_t scores_ld, const int32_t* n_vis, int64_t max_vis, int32_t* cand,
                                void* workspace, size_t workspace_bytes);

/* csa2_index_score_pool: csa2_index_score over the pool only. Pool entry p
 * of query q is entry j = B * cand[q, p / B] + p % B; its score goes to
 * scores_pool[q, p] (row length cand_keep * B). The pool's entries below
 * n_vis[q] are p < n_pool[q] = B (kept blocks - 1) + (n_vis - B (n_blocks - 1)),
 * written to n_pool [n_query] int32 (out); other entries are not written.
 * Keys, formats and the other arguments as for csa2_index_score. */
csa2_status csa2_index_score_pool(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query,
                                  const uint16_t* q_idx, const float* w_heads, const void* idx_keys,
                                  const uint8_t* idx_key_scale, const int64_t* pool_off, const int32_t* seq_of_q,
                                  const int32_t* n_vis, int64_t max_vis, const int32_t* cand, float* scores_pool,
                                  int32_t* n_pool);

/* csa2_topk_pool: the second level: a layer's own top-k inside the pool, from
 * csa2_index_score_pool's scores, written as entry indices (ascending, ties
 * to the lower entry, -1 padded), bit-exact on given scores.
 *   workspace: csa2_topk_workspace_size(ctx, n_query, cand_keep * B) bytes */
csa2_status csa2_topk_pool(csa2_ctx* ctx, void* stream, int32_t n_query, const float* scores_pool,
                           const int32_t* n_pool, const int32_t* cand, int32_t k, int32_t* out_idx,
                           void* workspace, size_t workspace_bytes);

/* ------------------------------------------------------------------------
 * csa2_attend: step 3 ("Reading Notes ...", section 3a attention formula and
 * 3f C2 step 3; WASTE item 1: the sink in the denominator only and the
 * de-rotation of the output's rope channels). For query q at t = q_pos[q] of
 * sequence b = seq_of_q[q], per head h:
 *   q~ = RoPE_t(q[q,h,:]);  rows R = window positions [max(lo_b, t-w+1), t]
 *   (row win_off[b] + p % (win_off[b+1]-win_off[b]) of win_kv) followed by
 *   the pool rows pool_off[b] + j for j in topk_idx[q, :], j != -1;
 *   s_r = softmax_scale * q~ . row_r;  o = sum_r e^{s_r} row_r /
 *   (sum_r e^{s_r} + e^{sink[h]});  out[q,h,:] = o with its rope channels
 *   rotated by -t. The same row is key and value.
 *   q        [n_query, 64, 512] bf16 (unrotated); q_pos [n_query] int64
 *   win_kv   stored window rows in kv_format, win_scale their scales
 *   win_off  [n_seq+1] int64 (capacity of sequence b's buffer = difference)
 *   win_lo   [n_seq] int64 window cut positions (nullable: 0)
 *   pool_kv  stored compressed rows in kv_format, pool_scale their scales
 *   topk_idx [n_query, topk] int32 (-1 = none); NULL: window only
 *   sink     [64] fp32; out [n_query, 64, 512] bf16; lse [n_query, 64] fp32
 *            natural-log denominator (nullable)
 * QK^T and PV run on tcgen05 tensor cores with bf16 operands (P rounded to
 * bf16) and fp32 accumulation in tensor memory.
 *   workspace of csa2_attend_workspace_size(ctx, n_query) bytes
 * q, win_kv, pool_kv and out must be 16-byte aligned (CSA2_ERR_INVALID_ARG). */
size_t csa2_attend_workspace_size(const csa2_ctx* ctx, int32_t n_query);
csa2_status csa2_attend(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query,
                        const uint16_t* q, const int64_t* q_pos, const int32_t* seq_of_q,
                        const void* win_kv, const uint8_t* win_scale, const int64_t* win_off,
                        const int64_t* win_lo, const void* pool_kv, const uint8_t* pool_scale,
                        const int64_t* pool_off, const int32_t* topk_idx, const float* sink,
                        uint16_t* out, float* lse, void* workspace, size_t workspace_bytes);

/* ------------------------------------------------------------------------
 * csa2_step: one layer step in one of the three modes ("Reading Notes ...",
 * 3f C2 step 4): Full = compress (when n_tokens > 0) + index_score + topk +
 * attend; Reindex = index_score + topk + attend on the borrowed pool and
 * keys; Reuse = attend with the borrowed selection in topk_idx. Every mode
 * uses its own q, window and sink. Field meanings are those of the
 * single-step calls above.
 * For few queries (2 * n_query <= SMs) the window tile of the attention runs
 * on a stream the context owns, forked from `stream` after the index launch
 * and joined back into it before the final merge; all work still orders
 * after what precedes the call on `stream`, and work enqueued on `stream`
 * after it orders after all of it (also under stream capture). Two steps on
 * one context must not run at the same time on different streams, as they
 * share that side stream. */
typedef struct csa2_step_args {
  int32_t mode;      /* csa2_mode */
  int32_t n_seq;
  int32_t n_query;
  int64_t max_vis;   /* host bound of n_vis */
  /* queries */
  const uint16_t* q;
  const int64_t* q_pos;
  const int32_t* seq_of_q;
  const int32_t* n_vis;
  const uint16_t* q_idx;   /* Full / Reindex */
  const float* w_heads;    /* Full / Reindex */
  const float* sink;
  /* window */
  const void* win_kv;
  const uint8_t* win_scale;
  const int64_t* win_off;
  const int64_t* win_lo;
  /* compressed pool and index keys (written by Full's compress) */
  void* pool_kv;
  uint8_t* pool_scale;
  void* idx_keys;
  uint8_t* idx_key_scale;
  const int64_t* pool_off;
  /* compressor inputs (Full only) */
  int64_t n_tokens;
  const uint16_t* raw;
  const float* gate;
  const int64_t* tok_off;
  const int64_t* first_pos;
  const float* norm_w;
  const uint16_t* w_idx;
  const float* k_norm_w;
  /* selection: written by Full / Reindex, read by Reuse */
  int32_t* topk_idx;
  /* outputs */
  uint16_t* out;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  /* compressor state (Full only): append != 0 makes the step's compress
   * follow csa2_compress_append, raw/gate/tok_off/first_pos being this
   * step's new tokens and the open groups waiting in state_raw/state_gate;
   * append == 0 keeps csa2_compress (whole groups only) */
  int32_t append;
  uint16_t* state_raw;
  float* state_gate;
  /* hierarchical indexer: cand_role 1 = this Full / Reindex step is the
   * candidate source and writes the pool of its queries to cand [n_query,
   * cand_keep] after its own selection (on the side stream, beside the
   * attention); 2 = this Reindex step scores and selects only inside the
   * pool in cand; 0 = neither */
  int32_t cand_role;
  int32_t* cand;
} csa2_step_args;

/* Two steps of one context must not overlap on the GPU: they share the
 * context's scan counters, side stream and events (see csa2_create). */
size_t csa2_step_workspace_size(const csa2_ctx* ctx, int32_t n_query, int64_t max_vis);
csa2_status csa2_step(csa2_ctx* ctx, void* stream, const csa2_step_args* args);

/* csa2_step_host: csa2_step with the step's inputs and output in host memory
 * (pinned, so that the transfers are asynchronous). The device buffers in
 * args are the staging buffers; the caches stay resident. A host buffer is
 * "mapped" below when it is page-locked memory that the device can address
 * (cudaHostAlloc, cudaMallocHost, or cudaHostRegister with mapping) and
 * 16-byte aligned.
 *   - io->q (n_query x 64 x 512 bf16) lands in args->q on the context's copy
 *     stream, which starts after the work already on `stream` and runs beside
 *     compress and the index scan: a mapped q by a small staging kernel (SM
 *     loads over the host link), any other by a copy-engine copy. Every
 *     attention launch of the step waits for it; nothing before reads q.
 *   - io->raw (n_tokens x 512 bf16) and io->gate (n_tokens x 512 fp32): when
 *     both are mapped, compress reads them where they lie and args->raw and
 *     args->gate are left untouched; otherwise they are copied there on the
 *     stream that runs compress, just before it.
 *   - io->out (n_query x 64 x 512 bf16): when mapped, the step's last launch
 *     writes the output into it directly over the host link and args->out is
 *     left untouched. Otherwise the step writes args->out and one copy on
 *     `stream` brings it into io->out.
 * A NULL host pointer skips that transfer. Returns after enqueueing; io->out
 * is valid once `stream` has completed, which orders after all of the step's
 * streams. Errors are those of csa2_step, plus CSA2_ERR_INVALID_ARG for a
 * host buffer whose device buffer in args is NULL. */
typedef struct csa2_host_io {
  const void* q;
  const void* raw;
  const void* gate;
  void* out;
} csa2_host_io;
csa2_status csa2_step_host(csa2_ctx* ctx, void* stream, const csa2_step_args* args, const csa2_host_io* io);

/* A csa2_step_host call captured once into a CUDA graph (its copies, its
 * launches on `stream` and on the context's side stream) and replayed by
 * csa2_step_graph_launch: each launch copies the same host buffers in, runs
 * the same step and copies the output back, in one driver call. Every buffer
 * that args and io name must stay valid while the graph exists; launches of
 * one context's graphs must not overlap in time (they share the context's
 * work counters), which holds when they go to one stream. */
typedef struct csa2_step_graph csa2_step_graph;
csa2_status csa2_step_graph_create(csa2_ctx* ctx, const csa2_step_args* args, const csa2_host_io* io,
                                   csa2_step_graph** out);
csa2_status csa2_step_graph_launch(csa2_step_graph* graph, void* stream);
void csa2_step_graph_destroy(csa2_step_graph* graph);

/* ------------------------------------------------------------------------
 * Pool sharding: one sequence's compressed pool split over G shards (devices
 * or launches), shard g holding entries [lo_g, hi_g) of every sequence. The
 * selection semantics are those of the unsharded step ("Reading Notes ...",
 * 3f C2 step 2, S_t = TopK sigma_t); the pages' own multi-rank form splits
 * heads and all-reduces the indexer's scores (PocketLLM "The CSA2 attention
 * layers"), this one splits the pool and exchanges 512 (score, entry) pairs
 * and one (m, l, O) partial per shard instead. Per shard:
 *   1. csa2_shard_visible: the shard's visible count;
 *   2. csa2_index_score + csa2_topk over the shard's own keys (entry j of the
 *      shard is global entry lo + j): its local top-k;
 *   3. csa2_topk_pairs: that selection as (score, global entry) pairs;
 *   4. exchange (all-gather) of the G pair lists; csa2_topk_merge: the global
 *      top-k, equal to the unsharded selection on the same scores;
 *   5. csa2_attend_partial over the global selection's entries that lie in
 *      the shard (the window on one shard only): an unnormalised partial;
 *   6. exchange of the G partials; csa2_attend_combine: the output, with the
 *      sink counted once.
 *
 * csa2_shard_visible: n_vis_shard[q] = clamp(n_vis[q] - shard_lo, 0,
 * shard_hi - shard_lo) for q < n_query; n_vis and n_vis_shard are [n_query]
 * int32 device arrays; 0 <= shard_lo <= shard_hi (host). */
csa2_status csa2_shard_visible(csa2_ctx* ctx, void* stream, int32_t n_query, const int32_t* n_vis, int64_t shard_lo,
                               int64_t shard_hi, int32_t* n_vis_shard);

/* csa2_topk_pairs: a local selection sel [n_query, k] int32 (ascending, -1
 * padded, entries relative to the shard) as pairs: pair_score[q, i] =
 * scores[q, sel[q, i]] and pair_idx[q, i] = index_base + sel[q, i]; a -1
 * entry gives (-inf, -1). scores [n_query, scores_ld] fp32 (the local scan's
 * rows); pair_score [n_query, k] fp32 and pair_idx [n_query, k] int32. */
csa2_status csa2_topk_pairs(csa2_ctx* ctx, void* stream, int32_t n_query, const float* scores, int64_t scores_ld,
                            const int32_t* sel, int32_t k, int64_t index_base, float* pair_score, int32_t* pair_idx);

/* csa2_topk_merge: the k best of n_lists pair lists, list-major as an
 * all-gather leaves them: pair_score / pair_idx [n_lists, n_query, list_len]
 * (fp32 / int32; entries with idx -1 are padding; each entry index appears
 * in at most one list). out_idx [n_query, k] int32 receives the k pairs of
 * largest score, ties to the lower entry index, -0.0 equal to +0.0, as
 * entry indices in ascending order, -1 padded: exactly csa2_topk's selection
 * over the same scores. n_lists * list_len must be at most 8,192 (else
 * CSA2_ERR_UNSUPPORTED); scores must not be NaN. One launch. */
csa2_status csa2_topk_merge(csa2_ctx* ctx, void* stream, int32_t n_query, int32_t n_lists, int32_t list_len,
                            const float* pair_score, const int32_t* pair_idx, int32_t k, int32_t* out_idx);

/* csa2_attend_partial: csa2_attend's softmax restricted to one shard's rows,
 * left unnormalised and without the sink, for csa2_attend_combine. The rows
 * are the window [max(lo, t-w+1), t] when with_window != 0 (one shard only),
 * and the entries j of topk_idx [n_query, topk] (global indices; NULL for
 * none) with shard_lo <= j < shard_hi, read from row pool_off[b] + j -
 * shard_lo of this shard's pool. For each query and head, with s_r = scale *
 * RoPE_t(q) . row_r and m a reference at least max_r s_r - 8 ln 2:
 *   part_o [n_query, 64, 512] fp32 = sum_r exp(s_r - m) row_r (rope
 *          channels not rotated back), 16-byte aligned
 *   part_m [n_query, 64] fp32 = m (natural-log units; -inf when the shard
 *          holds no row of that query)
 *   part_l [n_query, 64] fp32 = sum_r exp(s_r - m)
 * Window arguments are read only when with_window != 0. No workspace: one
 * CTA per query. Entries outside the shard are skipped; an entry inside it
 * but past the shard's pool is recorded as CSA2_FLAG_BAD_TOPK_INDEX. When a
 * query's entries inside the shard fill one run of columns (a selection in
 * ascending order, as csa2_topk_merge writes it), only that run is read, 128
 * entries a tile; any other order gives the same rows, tile by tile over
 * every column. */
csa2_status csa2_attend_partial(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query, const uint16_t* q,
                                const int64_t* q_pos, const int32_t* seq_of_q, int32_t with_window,
                                const void* win_kv, const uint8_t* win_scale, const int64_t* win_off,
                                const int64_t* win_lo, const void* pool_kv, const uint8_t* pool_scale,
                                const int64_t* pool_off, const int32_t* topk_idx, int64_t shard_lo, int64_t shard_hi,
                                float* part_o, float* part_m, float* part_l);

/* csa2_attend_combine: the log-sum-exp combine of n_parts (1..16) partials
 * laid out part-major as an all-gather leaves them: part_o [n_parts, n_query,
 * 64, 512], part_m and part_l [n_parts, n_query, 64] (fp32). With M =
 * max(max_g m_g, sink_h): out = sum_g e^(m_g - M) O_g / (sum_g e^(m_g - M) l_g
 * + e^(sink_h - M)), its rope channels rotated back by -t (q_pos [n_query]
 * int64), written as bf16 to out [n_query, 64, 512]; lse [n_query, 64] fp32
 * (nullable) = M + log(den). sink [64] fp32. */
csa2_status csa2_attend_combine(csa2_ctx* ctx, void* stream, int32_t n_query, int32_t n_parts, const float* part_o,
                                const float* part_m, const float* part_l, const int64_t* q_pos, const float* sink,
                                uint16_t* out, float* lse);

/* ------------------------------------------------------------------------
 * csa2_attend_noalloc: csa2_attend for callers that cannot allocate device
 * memory themselves (a host that owns all device memory through its own pool
 * and forbids outside allocations, or a loop that must never trigger the
 * allocator's implicit synchronisation). This entry point is an engineering
 * addition with no counterpart in the method's description; it computes
 * exactly what csa2_attend computes, with the same arguments minus the
 * workspace.
 *   - It allocates nothing and calls no allocating routine. Its split-K scratch
 *     is a library-owned device array of CSA2_NOALLOC_SCRATCH_BYTES, placed on
 *     each device that loads the library's module and held until exit.
 *   - Calls needing more scratch than that (csa2_attend_workspace_size(ctx,
 *     n_query) > CSA2_NOALLOC_SCRATCH_BYTES) are rejected with
 *     CSA2_ERR_WORKSPACE and a message; nothing is enqueued.
 *   - The first call made with a context looks up the array's device
 *     address on that context's device (which must be current) and keeps it
 *     in the context; make that first call before any stream capture begins.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents; calls whose work overlaps on the GPU race on it, so
 *     order them on one stream. */
#define CSA2_NOALLOC_SCRATCH_BYTES (32u << 20)
csa2_status csa2_attend_noalloc(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query, const uint16_t* q,
                                const int64_t* q_pos, const int32_t* seq_of_q, const void* win_kv,
                                const uint8_t* win_scale, const int64_t* win_off, const int64_t* win_lo,
                                const void* pool_kv, const uint8_t* pool_scale, const int64_t* pool_off,
                                const int32_t* topk_idx, const float* sink, uint16_t* out, float* lse);

/* Number of kernel launches the last entry point call on this context
 * enqueued (host). */
int32_t csa2_last_launch_count(const csa2_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H_ */
