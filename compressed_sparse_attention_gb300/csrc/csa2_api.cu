// Host side of the CSA2 C ABI: context, argument validation, workspace
// carving, kernel launches and the Full / Reindex / Reuse step dispatch.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

#include "ctx.cuh"
#include "launchers.cuh"

namespace {

constexpr size_t kAlign = 256;
inline size_t al(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

csa2_status fail(csa2_ctx* c, csa2_status s, const std::string& msg) {
  if (c) c->err = msg;
  return s;
}

csa2_status cuda_fail(csa2_ctx* c, cudaError_t e, const char* where) {
  return fail(c, CSA2_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

// YaRN ("NTK-by-parts", DeepSeek-V3 ramp) frequencies of the rotated pairs.
void rope_frequencies(const csa2_config& c, double* f) {
  const int half = c.rope_dim / 2;
  for (int i = 0; i < half; ++i) f[i] = std::pow(c.rope_theta, -(2.0 * i) / c.rope_dim);
  if (!(c.yarn_factor > 1.0)) return;
  auto boundary = [&](double turns) {
    return c.rope_dim * std::log(c.yarn_orig_len / (turns * 2.0 * M_PI)) / (2.0 * std::log(c.rope_theta));
  };
  double lo = std::floor(boundary(c.yarn_beta_fast));
  double hi = std::ceil(boundary(c.yarn_beta_slow));
  if (lo < 0) lo = 0;
  if (hi > c.rope_dim - 1) hi = c.rope_dim - 1;
  if (hi == lo) hi += 0.001;
  for (int i = 0; i < half; ++i) {
    double ramp = (i - lo) / (hi - lo);
    ramp = ramp < 0 ? 0 : (ramp > 1 ? 1 : ramp);
    // ramp 0 keeps the frequency, 1 divides it by the factor
    f[i] = f[i] * (1.0 - ramp) + f[i] / c.yarn_factor * ramp;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa2_status check_ws(csa2_ctx* c, const void* ws, size_t have, size_t need) {
  if (need == 0) return CSA2_OK;
  if (ws == nullptr || have < need)
    return fail(c, CSA2_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes");
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return fail(c, CSA2_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return CSA2_OK;
}

}  // namespace

extern "C" {

void csa2_default_config(csa2_config* c) {
  if (!c) return;
  std::memset(c, 0, sizeof(*c));
  c->n_heads = 64;
  c->head_dim = 512;
  c->rope_dim = 64;
  c->window = 128;
  c->compress_ratio = 4;
  c->idx_heads = 8;
  c->idx_dim = 128;
  c->topk = 512;
  c->kv_format = CSA2_KV_BF16;
  c->idx_key_format = CSA2_KV_BF16;
  c->softmax_scale = 1.0f / std::sqrt(512.0f);
  c->norm_eps = 1e-20f;
  c->rope_theta = 160000.0;
  c->yarn_factor = 16.0;
  c->yarn_orig_len = 65536.0;
  c->yarn_beta_fast = 32.0;
  c->yarn_beta_slow = 1.0;
  c->cand_block = 8;
  c->cand_keep = 2048;
}

// log2 of the candidate block size (a power of two)
static int cand_shift(const csa2_config& c) {
  int sh = 0;
  while ((1 << sh) < c.cand_block) ++sh;
  return sh;
}

const char* csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported geometry";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_DEVICE_FLAG: return "bad input recorded on the device";
    case CSA2_ERR_TIMEOUT: return "device wait timed out";
    case CSA2_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

static void release(csa2_ctx* ctx) {
  if (ctx->d_flags) cudaFree(ctx->d_flags);
  if (ctx->d_work) cudaFree(ctx->d_work);
  if (ctx->side) cudaStreamDestroy(ctx->side);
  if (ctx->copy) cudaStreamDestroy(ctx->copy);
  for (cudaEvent_t ev : {ctx->ev_join, ctx->ev_topk, ctx->ev_copy, ctx->ev_q})
    if (ev) cudaEventDestroy(ev);
  delete ctx;
}

csa2_status csa2_create(const csa2_config* cfg, csa2_ctx** out) {
  if (!cfg || !out) return CSA2_ERR_INVALID_ARG;
  *out = nullptr;
  const csa2_config& c = *cfg;
  if (c.n_heads != 64 || c.head_dim != 512 || c.idx_dim != 128) return CSA2_ERR_UNSUPPORTED;
  if (!(c.rope_dim == 0 || c.rope_dim == 64)) return CSA2_ERR_UNSUPPORTED;
  if (c.window < 1 || c.window > 128) return CSA2_ERR_UNSUPPORTED;
  if (c.compress_ratio < 1 || c.compress_ratio > 16) return CSA2_ERR_UNSUPPORTED;
  if (!(c.idx_heads == 8 || c.idx_heads == 16 || c.idx_heads == 32)) return CSA2_ERR_UNSUPPORTED;
  if (c.topk < 1 || c.topk > 2048) return CSA2_ERR_UNSUPPORTED;
  // pools must fit one top-k row of 16,384 entries
  if (c.cand_block < 1 || c.cand_block > 64 || (c.cand_block & (c.cand_block - 1)) != 0 || c.cand_keep < 1 ||
      c.cand_keep > 2048 || (int64_t)c.cand_keep * c.cand_block > 16384)
    return CSA2_ERR_UNSUPPORTED;
  if ((c.kv_format != CSA2_KV_BF16 && c.kv_format != CSA2_KV_FP8_E4M3_B32 && c.kv_format != CSA2_KV_FP4_E4M3_B16) ||
      (c.idx_key_format != CSA2_KV_BF16 && c.idx_key_format != CSA2_KV_FP8_E4M3_B32 &&
       c.idx_key_format != CSA2_KV_MXFP4_B32))
    return CSA2_ERR_UNSUPPORTED;
  if (!(c.rope_theta > 0) || !(c.yarn_orig_len > 0) || !(c.yarn_beta_fast > 0) || !(c.yarn_beta_slow > 0) ||
      !std::isfinite(c.softmax_scale) || !(c.norm_eps >= 0))
    return CSA2_ERR_INVALID_ARG;
  csa2_ctx* ctx = new csa2_ctx();
  ctx->cfg = c;
  cudaError_t e = cudaGetDevice(&ctx->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
  if (e == cudaSuccess) e = cudaMalloc(&ctx->d_flags, sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(ctx->d_flags, 0, sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMalloc(&ctx->d_work, 2 * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(ctx->d_work, 0, 2 * sizeof(unsigned long long));
  int prio_low = 0;
  if (e == cudaSuccess) e = cudaDeviceGetStreamPriorityRange(&prio_low, &ctx->prio_high);
  // the side stream carries the work that runs beside the caller's stream (a
  // candidate source's pool beside its attention): it goes first when both wait for SMs
  if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&ctx->side, cudaStreamNonBlocking, ctx->prio_high);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_join, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_topk, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ctx->copy, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_copy, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_q, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cudaGetLastError();
    release(ctx);
    return CSA2_ERR_CUDA;
  }
  std::memset(&ctx->rope, 0, sizeof(ctx->rope));
  ctx->rope.pairs = c.rope_dim / 2;
  rope_frequencies(c, ctx->rope.freq);
  *out = ctx;
  return CSA2_OK;
}

void csa2_destroy(csa2_ctx* ctx) {
  if (!ctx) return;
  release(ctx);
}

const char* csa2_last_error(const csa2_ctx* ctx) { return ctx ? ctx->err.c_str() : "no context"; }

int32_t csa2_last_launch_count(const csa2_ctx* ctx) { return ctx ? ctx->last_launches : 0; }

csa2_status csa2_rope_frequencies(const csa2_ctx* ctx, double* out, int32_t n) {
  if (!ctx || !out || n < ctx->rope.pairs) return CSA2_ERR_INVALID_ARG;
  for (int i = 0; i < ctx->rope.pairs; ++i) out[i] = ctx->rope.freq[i];
  return CSA2_OK;
}

csa2_status csa2_check(csa2_ctx* ctx, void* stream, uint32_t* flags_out) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t h = 0;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(&h, ctx->d_flags, sizeof(h), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(ctx->d_flags, 0, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "csa2_check");
  if (flags_out) *flags_out = h;
  if (h & CSA2_FLAG_WAIT_TIMEOUT) return fail(ctx, CSA2_ERR_TIMEOUT, "a device wait timed out");
  if (h) {
    char buf[96];
    std::snprintf(buf, sizeof(buf), "device error word 0x%x", h);
    return fail(ctx, CSA2_ERR_DEVICE_FLAG, buf);
  }
  return CSA2_OK;
}

csa2_status csa2_debug_wait_timeout(csa2_ctx* ctx, void* stream, uint64_t limit_ns) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (limit_ns < 1 || limit_ns > 1000000000ull)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "debug_wait_timeout: limit_ns must be 1 .. 1e9");
  const cudaError_t e = csa2::launch_wait_probe(reinterpret_cast<cudaStream_t>(stream), ctx->d_flags, limit_ns);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "debug_wait_timeout");
  ctx->last_launches = 1;
  return CSA2_OK;
}

csa2_status csa2_store_rows(csa2_ctx* ctx, void* stream, const float* rows, int64_t n_rows, int32_t dim,
                            const int64_t* pos, int32_t format, void* out, uint8_t* out_scale) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (n_rows < 0 || !(dim == 512 || dim == 128)) return fail(ctx, CSA2_ERR_INVALID_ARG, "dim must be 128 or 512");
  if (format < CSA2_KV_BF16 || format > CSA2_KV_MXFP4_B32) return fail(ctx, CSA2_ERR_INVALID_ARG, "format");
  if (n_rows == 0) return CSA2_OK;
  if (!rows || !out || (format != CSA2_KV_BF16 && !out_scale) || !aligned16(rows) || !aligned16(out))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "store_rows: null or misaligned buffer");
  cudaError_t e = csa2::launch_store_rows(reinterpret_cast<cudaStream_t>(stream), rows, n_rows, dim, pos,
                                          ctx->rope, format, out, out_scale);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "store_rows");
  ctx->last_launches = 1;
  return CSA2_OK;
}

static csa2_status do_compress(csa2_ctx* ctx, cudaStream_t st, const uint16_t* raw, const float* gate, int32_t n_seq,
                               int64_t n_tokens, const int64_t* tok_off, const int64_t* first_pos,
                               const int64_t* pool_off, const float* norm_w, const uint16_t* w_idx,
                               const float* k_norm_w, void* pool_kv, uint8_t* pool_kv_scale, void* idx_keys,
                               uint8_t* idx_key_scale, bool append = false, uint16_t* state_raw = nullptr,
                               float* state_gate = nullptr, const csa2::CompressTail* tail = nullptr,
                               bool pdl = false) {
  const csa2_config& c = ctx->cfg;
  const int m = c.compress_ratio;
  if (n_tokens < 0 || n_seq < 1) return fail(ctx, CSA2_ERR_INVALID_ARG, "compress: n_seq / n_tokens");
  if (n_tokens == 0) return CSA2_OK;
  if (!append && n_tokens % m) return fail(ctx, CSA2_ERR_INVALID_ARG, "compress: n_tokens must be whole groups");
  if (append && m > 1 && (!state_raw || !state_gate || !aligned16(state_raw) || !aligned16(state_gate)))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "compress_append: the state must be given and 16-byte aligned");
  if (!raw || !tok_off || !first_pos || !pool_off || !norm_w || !pool_kv || (m > 1 && !gate))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "compress: null pointer");
  if (c.kv_format != CSA2_KV_BF16 && !pool_kv_scale)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "compress: an fp8 / fp4 pool needs its scale array");
  if (w_idx && (!k_norm_w || !idx_keys || (c.idx_key_format != CSA2_KV_BF16 && !idx_key_scale)))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "compress: index key outputs missing");
  if (!aligned16(raw) || (gate && !aligned16(gate)) || !aligned16(norm_w) || (w_idx && !aligned16(w_idx)))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "compress: inputs must be 16-byte aligned");
  csa2::AppendArgs app;
  app.n_tokens = n_tokens;
  app.state_raw = state_raw;
  app.state_gate = state_gate;
  // append form: each sequence closes at most floor(n_b / m) + 1 groups
  const int64_t n_groups = append ? n_tokens / m + n_seq : n_tokens / m;
  int nl = 0;
  cudaError_t e = csa2::launch_compress(st, n_groups, raw, gate, m, n_seq, tok_off, first_pos, pool_off, norm_w,
                                        w_idx, k_norm_w, c.idx_dim, c.norm_eps, ctx->rope,
                                        c.kv_format, c.idx_key_format,
                                        pool_kv, pool_kv_scale, idx_keys, idx_key_scale, ctx->d_flags,
                                        append ? &app : nullptr, &nl, tail, pdl, ctx->num_sms);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "compress");
  ctx->last_launches += nl;
  return CSA2_OK;
}

csa2_status csa2_compress(csa2_ctx* ctx, void* stream, const uint16_t* raw, const float* gate, int32_t n_seq,
                          int64_t n_tokens, const int64_t* tok_off, const int64_t* first_pos, const int64_t* pool_off,
                          const float* norm_w, const uint16_t* w_idx, const float* k_norm_w, void* pool_kv,
                          uint8_t* pool_kv_scale, void* idx_keys, uint8_t* idx_key_scale) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  return do_compress(ctx, reinterpret_cast<cudaStream_t>(stream), raw, gate, n_seq, n_tokens, tok_off, first_pos,
                     pool_off, norm_w, w_idx, k_norm_w, pool_kv, pool_kv_scale, idx_keys, idx_key_scale);
}

csa2_status csa2_compress_append(csa2_ctx* ctx, void* stream, const uint16_t* raw, const float* gate, int32_t n_seq,
                                 int64_t n_tokens, const int64_t* tok_off, const int64_t* first_pos,
                                 const int64_t* pool_off, const float* norm_w, const uint16_t* w_idx,
                                 const float* k_norm_w, void* pool_kv, uint8_t* pool_kv_scale, void* idx_keys,
                                 uint8_t* idx_key_scale, uint16_t* state_raw, float* state_gate) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  return do_compress(ctx, reinterpret_cast<cudaStream_t>(stream), raw, gate, n_seq, n_tokens, tok_off, first_pos,
                     pool_off, norm_w, w_idx, k_norm_w, pool_kv, pool_kv_scale, idx_keys, idx_key_scale, true,
                     state_raw, state_gate);
}

// new_first / new_tok set: the scan leaves out the entries that this step's
// compress writes (see IdxArgs); the compress kernel scores them
static csa2_status do_index(csa2_ctx* ctx, cudaStream_t st, int32_t n_seq, int32_t n_query, const uint16_t* q_idx,
                            const float* w_heads, const void* idx_keys, const uint8_t* idx_key_scale,
                            const int64_t* pool_off, const int32_t* seq_of_q, const int32_t* n_vis, int64_t max_vis,
                            float* scores, int64_t ld, const int64_t* new_first = nullptr,
                            const int64_t* new_tok = nullptr, const int32_t* cand = nullptr,
                            int32_t* n_pool = nullptr, bool pdl = false, bool wait_first = false) {
  const csa2_config& c = ctx->cfg;
  // a pool row holds at most cand_keep blocks of entries
  const int64_t row_need = cand != nullptr ? std::min(max_vis, (int64_t)c.cand_keep * c.cand_block) : max_vis;
  if (n_query < 0 || n_seq < 1 || max_vis < 0 || ld < row_need)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "index_score: sizes");
  if (n_query == 0 || max_vis == 0) return CSA2_OK;
  if (!q_idx || !w_heads || !idx_keys || !pool_off || !seq_of_q || !n_vis || !scores)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "index_score: null pointer");
  if (c.idx_key_format != CSA2_KV_BF16 && !idx_key_scale)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "index_score: fp8 / mxfp4 keys need their scales");
  if (!aligned16(q_idx) || !aligned16(idx_keys) || (idx_key_scale && (reinterpret_cast<uintptr_t>(idx_key_scale) & 3)))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "index_score: misaligned buffer");
  const int kf = c.idx_key_format;
  csa2::IdxArgs ia;
  ia.n_query = n_query;
  ia.n_seq = n_seq;
  ia.max_vis = max_vis;
  ia.q_idx = q_idx;
  ia.w_heads = w_heads;
  ia.keys = idx_keys;
  ia.key_scale = idx_key_scale;
  ia.pool_off = pool_off;
  ia.seq_of_q = seq_of_q;
  ia.n_vis = n_vis;
  ia.scores = scores;
  ia.ld = ld;
  ia.flags = ctx->d_flags;
  ia.new_first = new_first;
  ia.new_tok = new_tok;
  ia.m = c.compress_ratio;
  ia.work = ctx->d_work;
  ia.cand = cand;
  ia.cand_ld = c.cand_keep;
  ia.cand_shift = cand_shift(c);
  ia.n_pool = n_pool;
  ia.wait_first = wait_first ? 1 : 0;
  cudaError_t e;
  if (new_first == nullptr && cand == nullptr &&
             csa2::index_tc_suited(kf != CSA2_KV_BF16, n_query, n_seq, c.idx_heads)) {
    e = csa2::launch_index_score_tc(st, ctx->num_sms, c.idx_heads, n_query, n_seq, max_vis, q_idx, w_heads,
                                    reinterpret_cast<const uint16_t*>(idx_keys), pool_off, seq_of_q, n_vis, scores,
                                    ld, ctx->d_flags);
  } else {
    e = csa2::launch_index_score(st, ctx->num_sms, c.idx_heads, kf, ia, pdl);
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "index_score");
  ctx->last_launches += 1;
  return CSA2_OK;
}

csa2_status csa2_index_score(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query, const uint16_t* q_idx,
                             const float* w_heads, const void* idx_keys, const uint8_t* idx_key_scale,
                             const int64_t* pool_off, const int32_t* seq_of_q, const int32_t* n_vis, int64_t max_vis,
                             float* scores, int64_t scores_ld) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  return do_index(ctx, reinterpret_cast<cudaStream_t>(stream), n_seq, n_query, q_idx, w_heads, idx_keys,
                  idx_key_scale, pool_off, seq_of_q, n_vis, max_vis, scores, scores_ld);
}

size_t csa2_topk_workspace_size(const csa2_ctx* ctx, int32_t n_query, int64_t max_vis) {
  if (!ctx || n_query < 0 || max_vis < 0) return 0;
  return csa2::topk_workspace_bytes(n_query, max_vis);
}

// pdl: launched inside csa2_step right after the library's own index scan,
// the top-k may start programmatically before the scan ends (it waits for it)
static csa2_status do_topk(csa2_ctx* ctx, cudaStream_t st, int32_t n_query, const float* scores, int64_t ld,
                           const int32_t* n_vis, int64_t max_vis, int32_t k, int32_t* out_idx, void* ws,
                           size_t ws_bytes, const int32_t* map = nullptr, bool pdl = false) {
  if (n_query < 0 || max_vis < 0 || ld < max_vis || k < 1 || k > 2048)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "topk: sizes (k must be 1..2048)");
  if (max_vis > 0xFFFFFFFEll) return fail(ctx, CSA2_ERR_UNSUPPORTED, "topk: rows longer than 2^32-2");
  if (n_query == 0) return CSA2_OK;
  if (!n_vis || !out_idx || (max_vis > 0 && !scores)) return fail(ctx, CSA2_ERR_INVALID_ARG, "topk: null pointer");
  csa2_status s = check_ws(ctx, ws, ws_bytes, csa2::topk_workspace_bytes(n_query, max_vis));
  if (s != CSA2_OK) return s;
  int nl = 0;
  cudaError_t e = map == nullptr
                      ? csa2::launch_topk(st, n_query, scores, ld, n_vis, max_vis, k, out_idx, ws, &nl, nullptr, 0, 0,
                                          pdl)
                      : csa2::launch_topk(st, n_query, scores, ld, n_vis, max_vis, k, out_idx, ws, &nl, map,
                                          ctx->cfg.cand_keep, cand_shift(ctx->cfg), pdl);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "topk");
  ctx->last_launches += nl;
  return CSA2_OK;
}

csa2_status csa2_topk(csa2_ctx* ctx, void* stream, int32_t n_query, const float* scores, int64_t scores_ld,
                      const int32_t* n_vis, int64_t max_vis, int32_t k, int32_t* out_idx, void* workspace,
                      size_t workspace_bytes) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  return do_topk(ctx, reinterpret_cast<cudaStream_t>(stream), n_query, scores, scores_ld, n_vis, max_vis, k, out_idx,
                 workspace, workspace_bytes);
}

size_t csa2_candidate_pool_workspace_size(const csa2_ctx* ctx, int32_t n_query, int64_t max_vis) {
  if (!ctx || n_query < 0 || max_vis < 0) return 0;
  return csa2::candidate_pool_workspace_bytes(n_query, max_vis, cand_shift(ctx->cfg));
}

static csa2_status do_candidate_pool(csa2_ctx* ctx, cudaStream_t st, int32_t n_query, const float* scores,
                                     int64_t ld, const int32_t* n_vis, int64_t max_vis, int32_t* cand, void* ws,
                                     size_t ws_bytes) {
  if (n_query < 0 || max_vis < 0 || ld < max_vis) return fail(ctx, CSA2_ERR_INVALID_ARG, "candidate_pool: sizes");
  if (max_vis > 0xFFFFFFFEll) return fail(ctx, CSA2_ERR_UNSUPPORTED, "candidate_pool: rows longer than 2^32-2");
  if (n_query == 0) return CSA2_OK;
  if (!n_vis || !cand || (max_vis > 0 && !scores)) return fail(ctx, CSA2_ERR_INVALID_ARG, "candidate_pool: null");
  csa2_status s = check_ws(ctx, ws, ws_bytes, csa2_candidate_pool_workspace_size(ctx, n_query, max_vis));
  if (s != CSA2_OK) return s;
  int nl = 0;
  cudaError_t e = csa2::launch_candidate_pool(st, n_query, scores, ld, n_vis, max_vis, cand_shift(ctx->cfg),
                                              ctx->cfg.cand_keep, cand, ws, &nl);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "candidate_pool");
  ctx->last_launches += nl;
  return CSA2_OK;
}

csa2_status csa2_candidate_pool(csa2_ctx* ctx, void* stream, int32_t n_query, const float* scores,
                                int64_t scores_ld, const int32_t* n_vis, int64_t max_vis, int32_t* cand,
                                void* workspace, size_t workspace_bytes) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  return do_candidate_pool(ctx, reinterpret_cast<cudaStream_t>(stream), n_query, scores, scores_ld, n_vis, max_vis,
                           cand, workspace, workspace_bytes);
}

csa2_status csa2_index_score_pool(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query,
                                  const uint16_t* q_idx, const float* w_heads, const void* idx_keys,
                                  const uint8_t* idx_key_scale, const int64_t* pool_off, const int32_t* seq_of_q,
                                  const int32_t* n_vis, int64_t max_vis, const int32_t* cand, float* scores_pool,
                                  int32_t* n_pool) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (!cand || !n_pool) return fail(ctx, CSA2_ERR_INVALID_ARG, "index_score_pool: null pool");
  const int64_t ld = (int64_t)ctx->cfg.cand_keep * ctx->cfg.cand_block;
  return do_index(ctx, reinterpret_cast<cudaStream_t>(stream), n_seq, n_query, q_idx, w_heads, idx_keys,
                  idx_key_scale, pool_off, seq_of_q, n_vis, max_vis, scores_pool, ld, nullptr, nullptr, cand, n_pool);
}

csa2_status csa2_topk_pool(csa2_ctx* ctx, void* stream, int32_t n_query, const float* scores_pool,
                           const int32_t* n_pool, const int32_t* cand, int32_t k, int32_t* out_idx, void* workspace,
                           size_t workspace_bytes) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (!cand) return fail(ctx, CSA2_ERR_INVALID_ARG, "topk_pool: null pool");
  const int64_t ld = (int64_t)ctx->cfg.cand_keep * ctx->cfg.cand_block;
  return do_topk(ctx, reinterpret_cast<cudaStream_t>(stream), n_query, scores_pool, ld, n_pool, ld, k, out_idx,
                 workspace, workspace_bytes, cand);
}

size_t csa2_attend_workspace_size(const csa2_ctx* ctx, int32_t n_query) {
  if (!ctx || n_query < 0) return 0;
  return csa2::attend_workspace_bytes(n_query, csa2::attend_plan(n_query, ctx->cfg.topk, true, ctx->num_sms));
}

// validates the attend arguments and fills the kernel parameters
static csa2_status attend_params(csa2_ctx* ctx, int32_t n_seq, int32_t n_query, const uint16_t* q,
                                 const int64_t* q_pos, const int32_t* seq_of_q, const void* win_kv,
                                 const uint8_t* win_scale, const int64_t* win_off, const int64_t* win_lo,
                                 const void* pool_kv, const uint8_t* pool_scale, const int64_t* pool_off,
                                 const int32_t* topk_idx, const float* sink, uint16_t* out, float* lse, void* ws,
                                 size_t ws_bytes, csa2::AttendParams* pp) {
  const csa2_config& c = ctx->cfg;
  const bool scaled = c.kv_format != CSA2_KV_BF16;  // fp8 window (fp8 or fp4 pool): scale arrays
  if (n_query < 0 || n_seq < 1) return fail(ctx, CSA2_ERR_INVALID_ARG, "attend: sizes");
  if (!q || !q_pos || !seq_of_q || !win_kv || !win_off || !sink || !out ||
      (topk_idx && (!pool_kv || !pool_off)) || (scaled && (!win_scale || (topk_idx && !pool_scale))))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "attend: null pointer");
  if (!aligned16(q) || !aligned16(win_kv) || (pool_kv && !aligned16(pool_kv)) || !aligned16(out))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "attend: misaligned buffer");
  const size_t need = csa2_attend_workspace_size(ctx, n_query);
  csa2_status s = check_ws(ctx, ws, ws_bytes, topk_idx ? need : 0);
  if (s != CSA2_OK) return s;
  if (n_query == 0) return CSA2_OK;
  csa2::AttendParams& p = *pp;
  std::memset(&p, 0, sizeof(p));
  p.q = q; p.q_pos = q_pos; p.seq_of_q = seq_of_q;
  p.win_kv = win_kv; p.win_scale = win_scale; p.win_off = win_off; p.win_lo = win_lo;
  p.pool_kv = pool_kv; p.pool_scale = pool_scale; p.pool_off = pool_off;
  p.topk_idx = topk_idx; p.sink = sink; p.out = out; p.lse = lse;
  p.flags = ctx->d_flags;
  p.n_seq = n_seq; p.n_query = n_query; p.topk = c.topk; p.window = c.window;
  p.scale_log2 = c.softmax_scale * 1.4426950408889634f;
  p.rp = ctx->rope;
  p.shard_lo = 0;
  p.shard_hi = INT64_MAX;
  return CSA2_OK;
}

static csa2_status do_attend(csa2_ctx* ctx, cudaStream_t st, int32_t n_seq, int32_t n_query, const uint16_t* q,
                             const int64_t* q_pos, const int32_t* seq_of_q, const void* win_kv,
                             const uint8_t* win_scale, const int64_t* win_off, const int64_t* win_lo,
                             const void* pool_kv, const uint8_t* pool_scale, const int64_t* pool_off,
                             const int32_t* topk_idx, const float* sink, uint16_t* out, float* lse, void* ws,
                             size_t ws_bytes) {
  csa2::AttendParams p;
  csa2_status s = attend_params(ctx, n_seq, n_query, q, q_pos, seq_of_q, win_kv, win_scale, win_off, win_lo, pool_kv,
                                pool_scale, pool_off, topk_idx, sink, out, lse, ws, ws_bytes, &p);
  if (s != CSA2_OK || n_query == 0) return s;
  int nl = 0;
  cudaError_t e = csa2::launch_attend(st, ctx->num_sms, ctx->cfg.kv_format, p, ws, &nl);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "attend");
  ctx->last_launches += nl;
  return CSA2_OK;
}

csa2_status csa2_attend(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query, const uint16_t* q,
                        const int64_t* q_pos, const int32_t* seq_of_q, const void* win_kv, const uint8_t* win_scale,
                        const int64_t* win_off, const int64_t* win_lo, const void* pool_kv, const uint8_t* pool_scale,
                        const int64_t* pool_off, const int32_t* topk_idx, const float* sink, uint16_t* out, float* lse,
                        void* workspace, size_t workspace_bytes) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  return do_attend(ctx, reinterpret_cast<cudaStream_t>(stream), n_seq, n_query, q, q_pos, seq_of_q, win_kv, win_scale,
                   win_off, win_lo, pool_kv, pool_scale, pool_off, topk_idx, sink, out, lse, workspace,
                   workspace_bytes);
}

// ---------------------------------------------------------------------------
// Pool sharding of one sequence's compressed pool over several devices or
// launches: per shard the visible count, the local selection's (score,
// entry) pairs, the merge of all shards' pairs, the shard's partial
// attention and the log-sum-exp combine of the partials.
// ---------------------------------------------------------------------------
csa2_status csa2_shard_visible(csa2_ctx* ctx, void* stream, int32_t n_query, const int32_t* n_vis, int64_t shard_lo,
                               int64_t shard_hi, int32_t* n_vis_shard) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (n_query < 0 || shard_lo < 0 || shard_hi < shard_lo || shard_hi - shard_lo > 0x7FFFFFFFll)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "shard_visible: sizes");
  if (n_query == 0) return CSA2_OK;
  if (!n_vis || !n_vis_shard) return fail(ctx, CSA2_ERR_INVALID_ARG, "shard_visible: null pointer");
  int nl = 0;
  const cudaError_t e = csa2::launch_shard_visible(reinterpret_cast<cudaStream_t>(stream), n_query, n_vis, shard_lo,
                                                   shard_hi, n_vis_shard, &nl);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "shard_visible");
  ctx->last_launches = nl;
  return CSA2_OK;
}

csa2_status csa2_topk_pairs(csa2_ctx* ctx, void* stream, int32_t n_query, const float* scores, int64_t scores_ld,
                            const int32_t* sel, int32_t k, int64_t index_base, float* pair_score, int32_t* pair_idx) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (n_query < 0 || k < 1 || k > 2048 || scores_ld < 1 || index_base < 0)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "topk_pairs: sizes");
  if (n_query == 0) return CSA2_OK;
  if (!scores || !sel || !pair_score || !pair_idx) return fail(ctx, CSA2_ERR_INVALID_ARG, "topk_pairs: null pointer");
  int nl = 0;
  const cudaError_t e = csa2::launch_topk_pairs(reinterpret_cast<cudaStream_t>(stream), n_query, scores, scores_ld, sel,
                                                k, index_base, pair_score, pair_idx, &nl);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "topk_pairs");
  ctx->last_launches = nl;
  return CSA2_OK;
}

csa2_status csa2_topk_merge(csa2_ctx* ctx, void* stream, int32_t n_query, int32_t n_lists, int32_t list_len,
                            const float* pair_score, const int32_t* pair_idx, int32_t k, int32_t* out_idx) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (n_query < 0 || n_lists < 1 || list_len < 1 || k < 1 || k > 2048)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "topk_merge: sizes");
  if ((int64_t)n_lists * list_len > 8192)
    return fail(ctx, CSA2_ERR_UNSUPPORTED, "topk_merge: n_lists * list_len must be at most 8192");
  if (n_query == 0) return CSA2_OK;
  if (!pair_score || !pair_idx || !out_idx) return fail(ctx, CSA2_ERR_INVALID_ARG, "topk_merge: null pointer");
  int nl = 0;
  const cudaError_t e = csa2::launch_topk_merge(reinterpret_cast<cudaStream_t>(stream), n_query, n_lists, list_len,
                                                pair_score, pair_idx, k, out_idx, &nl);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "topk_merge");
  ctx->last_launches = nl;
  return CSA2_OK;
}

csa2_status csa2_attend_partial(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query, const uint16_t* q,
                                const int64_t* q_pos, const int32_t* seq_of_q, int32_t with_window,
                                const void* win_kv, const uint8_t* win_scale, const int64_t* win_off,
                                const int64_t* win_lo, const void* pool_kv, const uint8_t* pool_scale,
                                const int64_t* pool_off, const int32_t* topk_idx, int64_t shard_lo, int64_t shard_hi,
                                float* part_o, float* part_m, float* part_l) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  const csa2_config& c = ctx->cfg;
  const bool scaled = c.kv_format != CSA2_KV_BF16;
  if (n_query < 0 || n_seq < 1 || shard_lo < 0 || shard_hi < shard_lo)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "attend_partial: sizes or shard range");
  if (!with_window && !topk_idx) return fail(ctx, CSA2_ERR_INVALID_ARG, "attend_partial: neither window nor selection");
  if (n_query == 0) return CSA2_OK;
  if (!q || !q_pos || !seq_of_q || !part_o || !part_m || !part_l ||
      (with_window && (!win_kv || !win_off || (scaled && !win_scale))) ||
      (topk_idx && (!pool_kv || !pool_off || (scaled && !pool_scale))))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "attend_partial: null pointer");
  if (!aligned16(q) || !aligned16(part_o) || (with_window && !aligned16(win_kv)) || (pool_kv && !aligned16(pool_kv)))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "attend_partial: misaligned buffer");
  csa2::AttendParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q; p.q_pos = q_pos; p.seq_of_q = seq_of_q;
  // a shard without the window never reads it; win_off must still index
  // sequences, so the pool offsets stand in for it
  p.win_kv = with_window ? win_kv : pool_kv;
  p.win_scale = with_window ? win_scale : pool_scale;
  p.win_off = with_window ? win_off : pool_off;
  p.win_lo = with_window ? win_lo : nullptr;
  p.pool_kv = pool_kv; p.pool_scale = pool_scale; p.pool_off = pool_off;
  p.topk_idx = topk_idx;
  p.flags = ctx->d_flags;
  p.n_seq = n_seq; p.n_query = n_query; p.topk = c.topk; p.window = c.window;
  p.scale_log2 = c.softmax_scale * 1.4426950408889634f;
  p.rp = ctx->rope;
  p.shard_lo = shard_lo;
  p.shard_hi = shard_hi;
  p.part_o = part_o;
  p.part_m = part_m;
  p.part_l = part_l;
  int nl = 0;
  const cudaError_t e = csa2::launch_attend_partial(reinterpret_cast<cudaStream_t>(stream), c.kv_format, p,
                                                    with_window ? 1 : 0, &nl);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "attend_partial");
  ctx->last_launches = nl;
  return CSA2_OK;
}

csa2_status csa2_attend_combine(csa2_ctx* ctx, void* stream, int32_t n_query, int32_t n_parts, const float* part_o,
                                const float* part_m, const float* part_l, const int64_t* q_pos, const float* sink,
                                uint16_t* out, float* lse) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (n_query < 0 || n_parts < 1 || n_parts > 16) return fail(ctx, CSA2_ERR_INVALID_ARG, "attend_combine: n_parts 1..16");
  if (n_query == 0) return CSA2_OK;
  if (!part_o || !part_m || !part_l || !q_pos || !sink || !out || !aligned16(part_o) || !aligned16(out))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "attend_combine: null or misaligned buffer");
  int nl = 0;
  const cudaError_t e = csa2::launch_attend_combine(reinterpret_cast<cudaStream_t>(stream), n_query, n_parts, part_o,
                                                    part_m, part_l, q_pos, sink, ctx->rope, out, lse, &nl);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "attend_combine");
  ctx->last_launches = nl;
  return CSA2_OK;
}

// The step's workspace: index scores (full rows of max_vis, or pool rows of
// cand_keep * cand_block for a pool reader), the pool sizes, the top-k
// scratch, the candidate-pool scratch (a candidate source builds its pool
// beside the attention) and the attention partials, side by side.
struct StepWs {
  size_t scores, n_pool, tk, cand, at;
};
static StepWs step_ws(const csa2_ctx* ctx, int32_t n_query, int64_t max_vis) {
  const int64_t ld = max_vis > 0 ? max_vis : 1;
  const int64_t ldc = (int64_t)ctx->cfg.cand_keep * ctx->cfg.cand_block;
  StepWs w;
  w.scores = al((size_t)n_query * (size_t)std::max(ld, ldc) * 4);
  w.n_pool = al((size_t)n_query * 4);
  w.tk = al(csa2_topk_workspace_size(ctx, n_query, max_vis));
  w.cand = al(csa2_candidate_pool_workspace_size(ctx, n_query, max_vis));
  w.at = al(csa2_attend_workspace_size(ctx, n_query));
  return w;
}

size_t csa2_step_workspace_size(const csa2_ctx* ctx, int32_t n_query, int64_t max_vis) {
  if (!ctx || n_query < 0 || max_vis < 0) return 0;
  const StepWs w = step_ws(ctx, n_query, max_vis);
  return w.scores + w.n_pool + w.tk + w.cand + w.at;
}

// Host buffers of a step's inputs (csa2_step_host). A *_dev pointer is the
// same buffer's device address, set when it is page-locked, mapped and 16-byte
// aligned: then q is staged by a kernel and compress reads the raw tokens and
// gates in place; otherwise the copy engines move them.
struct StepHostIn {
  const void* q = nullptr;
  const void* raw = nullptr;
  const void* gate = nullptr;
  const void* q_dev = nullptr;
  const void* raw_dev = nullptr;
  const void* gate_dev = nullptr;
};

static csa2_status step_impl(csa2_ctx* ctx, cudaStream_t st, const csa2_step_args* a, const StepHostIn* hin);

csa2_status csa2_step(csa2_ctx* ctx, void* stream, const csa2_step_args* a) {
  return step_impl(ctx, reinterpret_cast<cudaStream_t>(stream), a, nullptr);
}

static csa2_status step_impl(csa2_ctx* ctx, cudaStream_t st, const csa2_step_args* a, const StepHostIn* hin) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (!a) return fail(ctx, CSA2_ERR_INVALID_ARG, "step: null args");
  if (a->mode != CSA2_MODE_FULL && a->mode != CSA2_MODE_REINDEX && a->mode != CSA2_MODE_REUSE)
    return fail(ctx, CSA2_ERR_INVALID_ARG, "step: unknown mode");
  if (!a->topk_idx) return fail(ctx, CSA2_ERR_INVALID_ARG, "step: topk_idx is required");
  const size_t need = csa2_step_workspace_size(ctx, a->n_query, a->max_vis);
  csa2_status s = check_ws(ctx, a->workspace, a->workspace_bytes, need);
  if (s != CSA2_OK) return s;
  if (a->cand_role < 0 || a->cand_role > 2 || (a->cand_role != 0 && !a->cand) ||
      (a->cand_role != 0 && a->mode == CSA2_MODE_REUSE))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "step: cand_role needs cand and a Full or Reindex step");
  const bool pool_src = a->cand_role == 1, pool_read = a->cand_role == 2;
  char* ws = reinterpret_cast<char*>(a->workspace);
  const int64_t ld = a->max_vis > 0 ? a->max_vis : 1;
  const int64_t ldc = (int64_t)ctx->cfg.cand_keep * ctx->cfg.cand_block;
  const StepWs wl = step_ws(ctx, a->n_query, a->max_vis);
  float* scores = reinterpret_cast<float*>(ws);
  int32_t* n_pool = reinterpret_cast<int32_t*>(ws + wl.scores);
  char* tk_ws = ws + wl.scores + wl.n_pool;
  const size_t tk_bytes = wl.tk;
  char* cand_ws = tk_ws + wl.tk;
  char* at_ws = cand_ws + wl.cand;
  const size_t at_bytes = a->workspace_bytes - (size_t)(at_ws - ws);
  // the attention arguments are checked before anything is enqueued
  csa2::AttendParams ap;
  s = attend_params(ctx, a->n_seq, a->n_query, a->q, a->q_pos, a->seq_of_q, a->win_kv, a->win_scale, a->win_off,
                    a->win_lo, a->pool_kv, a->pool_scale, a->pool_off, a->topk_idx, a->sink, a->out, a->lse, at_ws,
                    at_bytes, &ap);
  if (s != CSA2_OK) return s;
  const int kvf = ctx->cfg.kv_format;
  const int m = ctx->cfg.compress_ratio;
  int launches = 0;
  // Every exit after a fork makes the caller's stream wait for the side
  // stream's last launch, so that a capture of the step stays well formed and
  // the caller's stream orders after all of it.
  // The same holds for the copy stream that brings q in from host memory.
  bool side_open = false, q_pending = false;
  auto join = [&](csa2_status so) -> csa2_status {
    cudaError_t je = cudaSuccess;
    if (side_open) {
      side_open = false;
      je = cudaEventRecord(ctx->ev_join, ctx->side);
      if (je == cudaSuccess) je = cudaStreamWaitEvent(st, ctx->ev_join, 0);
    }
    if (q_pending) {
      q_pending = false;
      const cudaError_t qe = cudaStreamWaitEvent(st, ctx->ev_q, 0);
      if (je == cudaSuccess) je = qe;
    }
    if (je != cudaSuccess && so == CSA2_OK) return cuda_fail(ctx, je, "step: join");
    return so;
  };
  // Host inputs. Nothing before the attention reads q, so it moves on the
  // copy stream beside compress and the index scan (a staging kernel, placed
  // first so that its CTAs start before the scan's fill the SMs), and every
  // attention launch waits for it. Compress reads mapped raw tokens and gates
  // where they lie; others are copied just before it on its stream.
  const size_t q_bytes = hin && hin->q ? (size_t)a->n_query * csa2::kHeads * csa2::kDim * 2 : 0;
  const bool tok_direct = hin && hin->raw_dev && (hin->gate_dev || !hin->gate);
  const size_t raw_bytes = hin && hin->raw && !tok_direct ? (size_t)a->n_tokens * csa2::kDim * 2 : 0;
  const size_t gate_bytes = hin && hin->gate && !tok_direct ? (size_t)a->n_tokens * csa2::kDim * 4 : 0;
  const uint16_t* raw_in = tok_direct ? static_cast<const uint16_t*>(hin->raw_dev) : a->raw;
  const float* gate_in = tok_direct && hin->gate_dev ? static_cast<const float*>(hin->gate_dev) : a->gate;
  auto wait_q = [&](cudaStream_t sw) -> cudaError_t {
    if (!q_pending) return cudaSuccess;
    const cudaError_t we = cudaStreamWaitEvent(sw, ctx->ev_q, 0);
    if (we == cudaSuccess && sw == st) q_pending = false;
    return we;
  };
  auto copy_tokens = [&](cudaStream_t sc) -> cudaError_t {
    cudaError_t ce = cudaSuccess;
    if (raw_bytes)
      ce = cudaMemcpyAsync(const_cast<uint16_t*>(a->raw), hin->raw, raw_bytes, cudaMemcpyHostToDevice, sc);
    if (ce == cudaSuccess && gate_bytes)
      ce = cudaMemcpyAsync(const_cast<float*>(a->gate), hin->gate, gate_bytes, cudaMemcpyHostToDevice, sc);
    return ce;
  };
  if (q_bytes) {
    const cudaError_t e = cudaEventRecord(ctx->ev_copy, st);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "step: copy of q");
  }
  // enqueued after the launches it must not delay (the scan's, whose CTAs then
  // hold every SM: the staging runs as they retire, before top-k ends)
  bool q_staged = false;
  auto stage_q = [&]() -> cudaError_t {
    if (!q_bytes || q_staged) return cudaSuccess;
    q_staged = true;
    cudaError_t e = cudaStreamWaitEvent(ctx->copy, ctx->ev_copy, 0);
    if (e == cudaSuccess) {
      q_pending = true;
      if (hin->q_dev)
        e = csa2::launch_stage_copy(ctx->copy, ctx->num_sms, hin->q_dev, const_cast<uint16_t*>(a->q),
                                    (int64_t)q_bytes, &launches);
      else
        e = cudaMemcpyAsync(const_cast<uint16_t*>(a->q), hin->q, q_bytes, cudaMemcpyHostToDevice, ctx->copy);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_q, ctx->copy);
    return e;
  };
  // A decode-shaped Full step (at most two closing groups per sequence, the
  // scan in its CUDA-core form): compress runs first on the caller's stream
  // and scores the entries it writes itself, from the keys it stores. The
  // scan over the entries that existed before the step starts
  // programmatically beside it (its CTAs take the SMs compress leaves, and
  // wait for compress only before they exit), so that every kernel of the
  // step after compress has a single predecessor and can start early.
  const bool full = a->mode == CSA2_MODE_FULL;
  const bool overlap = full && !pool_read && a->n_query > 0 && a->max_vis > 0 && a->n_tokens <= 2LL * m * a->n_seq &&
                       !csa2::index_tc_suited(ctx->cfg.idx_key_format != CSA2_KV_BF16, a->n_query, a->n_seq,
                                              ctx->cfg.idx_heads);
  const bool tail = overlap && a->w_idx != nullptr;  // compress writes index keys: it scores the new ones
  if (full) {
    cudaError_t ce = copy_tokens(st);
    if (ce != cudaSuccess) return join(cuda_fail(ctx, ce, "step: copy of the raw tokens"));
    ctx->last_launches = 0;
    csa2::CompressTail ct;
    if (tail) {
      if (!a->q_idx || !a->w_heads || !a->seq_of_q || !a->n_vis || !aligned16(a->q_idx))
        return join(fail(ctx, CSA2_ERR_INVALID_ARG, "step: index arguments missing or misaligned"));
      ct.n_query = a->n_query;
      ct.idx_heads = ctx->cfg.idx_heads;
      ct.max_vis = a->max_vis;
      ct.ld = ld;
      ct.seq_of_q = a->seq_of_q;
      ct.n_vis = a->n_vis;
      ct.q_idx = a->q_idx;
      ct.w_heads = a->w_heads;
      ct.scores = scores;
    }
    // the step's first kernel: launched programmatically, it waits for the
    // previous kernel of the stream before it reads anything (this hides the
    // launch latency only; its inputs are complete once the wait returns)
    s = do_compress(ctx, st, raw_in, gate_in, a->n_seq, a->n_tokens, a->tok_off, a->first_pos, a->pool_off,
                    a->norm_w, a->w_idx, a->k_norm_w, a->pool_kv, a->pool_scale, a->idx_keys, a->idx_key_scale,
                    a->append != 0, a->state_raw, a->state_gate, tail ? &ct : nullptr, true);
    if (s != CSA2_OK) return join(s);
    launches += ctx->last_launches;
  }
  if (!full) {
    const cudaError_t ce = copy_tokens(st);
    if (ce != cudaSuccess) return join(cuda_fail(ctx, ce, "step: copy of the raw tokens"));
  }
  if (a->n_query == 0) {
    ctx->last_launches = launches;
    return join(CSA2_OK);
  }
  if (a->mode == CSA2_MODE_REUSE) {
    // nothing to overlap with: window and selected tiles share one launch
    ctx->last_launches = 0;
    cudaError_t e = stage_q();
    if (e == cudaSuccess) e = wait_q(st);
    if (e == cudaSuccess) e = csa2::launch_attend(st, ctx->num_sms, kvf, ap, at_ws, &ctx->last_launches);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "step: attend");
    ctx->last_launches += launches;
    return CSA2_OK;
  }
  ctx->last_launches = 0;
  // the scan follows compress programmatically (waiting for it at its end),
  // or is the step's first kernel (waiting for the stream's previous kernel
  // at its start); with a compress that is not the overlap form it waits at
  // its start too
  const bool scan_first = !full;
  const bool scan_pdl = scan_first || (overlap && a->n_tokens > 0) || (full && a->n_tokens > 0);
  const bool scan_wait_first = scan_first || !(overlap && a->n_tokens > 0);
  if (pool_read)  // the hierarchical indexer's second level: score inside the pool only
    s = do_index(ctx, st, a->n_seq, a->n_query, a->q_idx, a->w_heads, a->idx_keys, a->idx_key_scale, a->pool_off,
                 a->seq_of_q, a->n_vis, a->max_vis, scores, ldc, nullptr, nullptr, a->cand, n_pool, scan_pdl,
                 scan_wait_first);
  else
    s = do_index(ctx, st, a->n_seq, a->n_query, a->q_idx, a->w_heads, a->idx_keys, a->idx_key_scale, a->pool_off,
                 a->seq_of_q, a->n_vis, a->max_vis, scores, ld, tail ? a->first_pos : nullptr,
                 tail ? a->tok_off : nullptr, nullptr, nullptr, scan_pdl, scan_wait_first);
  if (s != CSA2_OK) return join(s);
  launches += ctx->last_launches;
  cudaError_t e = stage_q();
  if (e != cudaSuccess) return join(cuda_fail(ctx, e, "step: copy of q"));
  // top-k follows the library's own scan on this stream: it starts
  // programmatically and waits for the scan before reading the scores
  ctx->last_launches = 0;
  if (pool_read)
    s = do_topk(ctx, st, a->n_query, scores, ldc, n_pool, ldc, ctx->cfg.topk, a->topk_idx, tk_ws, tk_bytes, a->cand,
                true);
  else
    s = do_topk(ctx, st, a->n_query, scores, ld, a->n_vis, a->max_vis, ctx->cfg.topk, a->topk_idx, tk_ws, tk_bytes,
                nullptr, true);
  if (s != CSA2_OK) return join(s);
  launches += ctx->last_launches;
  if (pool_src) {
    e = cudaEventRecord(ctx->ev_topk, st);
    if (e != cudaSuccess) return join(cuda_fail(ctx, e, "step: record top-k"));
  }
  e = wait_q(st);
  if (e != cudaSuccess) return join(cuda_fail(ctx, e, "step: wait for q"));
  // The attention follows the library's own top-k on this stream: its CTAs
  // start programmatically, the window tiles (the first CTA of each query)
  // run beside top-k, and the selection is read after waiting for it. Its
  // other inputs are the step's, complete before the step began or ordered
  // by events. The merge follows the attention the same way.
  ap.pdl = 1;
  // rows of up to 16,384 entries take a one-CTA top-k, short enough that a
  // CTA holding the window tile and a selected tile would run them in series
  e = csa2::launch_attend(st, ctx->num_sms, kvf, ap, at_ws, &launches, pool_read || a->max_vis <= 16384);
  if (e != cudaSuccess) return join(cuda_fail(ctx, e, "step: attend"));
  if (pool_src) {
    // the candidate source's pool, for the layers after it, on the side
    // stream beside the attention; the caller's stream waits for it last
    e = cudaStreamWaitEvent(ctx->side, ctx->ev_topk, 0);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "step: candidate pool");
    side_open = true;
    ctx->last_launches = 0;
    s = do_candidate_pool(ctx, ctx->side, a->n_query, scores, ld, a->n_vis, a->max_vis, a->cand, cand_ws, wl.cand);
    launches += ctx->last_launches;
    s = join(s);
    if (s != CSA2_OK) return s;
  }
  ctx->last_launches = launches;
  return CSA2_OK;
}

csa2_status csa2_step_host(csa2_ctx* ctx, void* stream, const csa2_step_args* a, const csa2_host_io* io) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  if (!a || !io) return fail(ctx, CSA2_ERR_INVALID_ARG, "step_host: null args");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t q_bytes = (size_t)a->n_query * csa2::kHeads * csa2::kDim * 2;
  if ((io->q && !a->q) || (io->raw && !a->raw) || (io->gate && !a->gate) || (io->out && !a->out))
    return fail(ctx, CSA2_ERR_INVALID_ARG, "step_host: a host buffer without its device buffer");
  // An output buffer in page-locked host memory that the device addresses
  // (16-byte aligned) is written by the step's last launch directly, over the
  // host link; any other is filled by one copy from args->out after the step.
  auto dev_addr = [](const void* h) -> void* {
    if (!h) return nullptr;
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, h) != cudaSuccess) {
      cudaGetLastError();  // an address CUDA does not know: the copy engines move it
      return nullptr;
    }
    if (pa.type != cudaMemoryTypeHost || !pa.devicePointer || (reinterpret_cast<uintptr_t>(pa.devicePointer) & 15))
      return nullptr;
    return pa.devicePointer;
  };
  csa2_step_args da = *a;
  bool direct_out = false;
  if (io->out && q_bytes) {
    if (void* d = dev_addr(io->out)) {
      da.out = static_cast<uint16_t*>(d);
      direct_out = true;
    }
  }
  StepHostIn hin;
  hin.q = io->q;
  hin.raw = io->raw;
  hin.gate = io->gate;
  hin.q_dev = dev_addr(io->q);
  hin.raw_dev = dev_addr(io->raw);
  hin.gate_dev = dev_addr(io->gate);
  csa2_status s = step_impl(ctx, st, &da, &hin);
  if (s != CSA2_OK) return s;
  if (io->out && q_bytes && !direct_out) {
    const cudaError_t e = cudaMemcpyAsync(io->out, a->out, q_bytes, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "step_host: copy out");
  }
  return CSA2_OK;
}

struct csa2_step_graph {
  csa2_ctx* ctx = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

csa2_status csa2_step_graph_create(csa2_ctx* ctx, const csa2_step_args* a, const csa2_host_io* io,
                                   csa2_step_graph** out) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  if (!a || !io || !out) return fail(ctx, CSA2_ERR_INVALID_ARG, "step_graph_create: null argument");
  *out = nullptr;
  cudaStream_t cs = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "step_graph_create: stream");
  csa2_step_graph* g = new csa2_step_graph();
  g->ctx = ctx;
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  csa2_status s = CSA2_OK;
  if (e == cudaSuccess) {
    s = csa2_step_host(ctx, cs, a, io);
    // end the capture whatever happened, so that the stream is usable again
    const cudaError_t ee = cudaStreamEndCapture(cs, &g->graph);
    if (s == CSA2_OK && ee != cudaSuccess) s = cuda_fail(ctx, ee, "step_graph_create: capture");
  } else {
    s = cuda_fail(ctx, e, "step_graph_create: begin capture");
  }
  if (s == CSA2_OK) {
    e = cudaGraphInstantiate(&g->exec, g->graph, 0);
    if (e != cudaSuccess) s = cuda_fail(ctx, e, "step_graph_create: instantiate");
  }
  cudaStreamDestroy(cs);
  if (s != CSA2_OK) {
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    return s;
  }
  *out = g;
  return CSA2_OK;
}

csa2_status csa2_step_graph_launch(csa2_step_graph* g, void* stream) {
  if (!g) return CSA2_ERR_INVALID_ARG;
  const cudaError_t e = cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(g->ctx, e, "step_graph_launch");
  return CSA2_OK;
}

void csa2_step_graph_destroy(csa2_step_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

}  // extern "C"
