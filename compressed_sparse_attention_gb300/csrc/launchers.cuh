// Internal launcher declarations shared by the kernel files and the C-ABI host
// code (not part of the public interface).
#pragma once
#include "common.cuh"

namespace csa2 {

// Launch on `st` with programmatic stream serialization when `pdl` is set:
// the kernel may start before the previous kernel of the stream ends and
// waits for it with pdl_wait() before reading what it wrote. `priority`
// (when nonzero) is the launch's scheduling priority.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      int priority, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (priority != 0) {
    attr[na].id = cudaLaunchAttributePriority;
    attr[na].val.priority = priority;
    ++na;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct AttendParams {
  const uint16_t* q;
  const int64_t* q_pos;
  const int32_t* seq_of_q;
  const void* win_kv;
  const uint8_t* win_scale;
  const int64_t* win_off;
  const int64_t* win_lo;
  const void* pool_kv;
  const uint8_t* pool_scale;
  const int64_t* pool_off;
  const int32_t* topk_idx;
  const float* sink;
  uint16_t* out;
  float* lse;
  uint16_t* ws_o; // [n_query][n_slots][64][512] unnormalised partial outputs, bf16
  float2* ws_ml;  // [n_query][n_split][64] running (max, sum) per head
  uint32_t* flags;
  int n_seq;
  int n_query;
  int topk;
  int window;
  int n_tiles;          // tiles of one query: window + ceil(topk / 128)
  int tile_base;        // first tile this launch covers
  int tile_count;       // tiles this launch covers
  int n_split;          // CTAs per query in this launch
  int tiles_per_split;
  int lead_tiles;       // tiles of split 0 (the others take tiles_per_split each)
  int n_slots;          // partial slots per query in the workspace
  int slot_base;        // slot of this launch's first split
  int direct;           // 1: write the normalised output, no partials; 2: write the
                        // unnormalised partial (part_o, part_m, part_l) of csa2_attend_partial
  float scale_log2;  // softmax_scale * log2(e)
  RopeParams rp;
  // pool sharding (csa2_attend_partial): selected entries j outside
  // [shard_lo, shard_hi) are skipped, the others read pool row j - shard_lo;
  // the defaults 0 and INT64_MAX read every entry
  int64_t shard_lo;
  int64_t shard_hi;
  float* part_o;  // [n_query][64][512] fp32, rope channels not rotated back
  float* part_m;  // [n_query][64] reference max, natural-log units (-inf: no rows)
  float* part_l;  // [n_query][64] sum of exp(s_r - m)
  // launch settings (host only): pdl = programmatic launch after the previous
  // kernel of the stream (csa2_step's top-k, or its selected tiles for the
  // merge); the kernel reads the selection only after pdl_wait(). priority:
  // the launch's scheduling priority (0: the stream's)
  int pdl;
  int priority;
};

cudaError_t launch_store_rows(cudaStream_t st, const float* rows, int64_t n_rows, int dim, const int64_t* pos,
                              const RopeParams& rp, int fmt, void* out, uint8_t* out_scale);
// the append form of the compressor (csa2_compress_append); NULL: whole groups
struct AppendArgs {
  int64_t n_tokens = 0;
  uint16_t* state_raw = nullptr;
  float* state_gate = nullptr;
};
// Scores of the entries a decode step compresses, taken by the compress
// kernel itself from the index keys it stores (the index scan of that step
// leaves those entries out): for each query q of the group's sequence whose
// visible count covers entry j, scores[q * ld + j] = sum_h w_heads[q, h] *
// relu(q_idx[q, h] . key_j) with the stored key's exact values, fp32.
struct CompressTail {
  int n_query = 0;
  int idx_heads = 0;
  int64_t max_vis = 0;
  int64_t ld = 0;
  const int32_t* seq_of_q = nullptr;
  const int32_t* n_vis = nullptr;
  const uint16_t* q_idx = nullptr;
  const float* w_heads = nullptr;
  float* scores = nullptr;  // NULL: no scoring
};
// n_groups: the closing groups (whole-group form) or a bound of them (append
// form: n_tokens / m + n_seq); n_launch counts the launches made
// bytes (a multiple of 16, both pointers 16-byte aligned) from device-addressable
// host memory to device memory, by a few CTAs
cudaError_t launch_stage_copy(cudaStream_t st, int num_sms, const void* src, void* dst, int64_t bytes,
                              int* n_launch);
cudaError_t launch_compress(cudaStream_t st, int64_t n_groups, const uint16_t* raw, const float* gate, int m,
                            int n_seq, const int64_t* tok_off, const int64_t* first_pos, const int64_t* pool_off,
                            const float* norm_w, const uint16_t* w_idx, const float* k_norm_w, int idx_dim,
                            float eps, const RopeParams& rp, int kv_fmt, int idx_fmt, void* pool_kv,
                            uint8_t* pool_kv_scale, void* idx_keys, uint8_t* idx_key_scale, uint32_t* flags,
                            const AppendArgs* app, int* n_launch, const CompressTail* tail = nullptr,
                            bool pdl = false, int num_sms = 0);
// arguments of the index scan (csa2_index_score)
struct IdxArgs {
  int n_query = 0, n_seq = 0;
  int64_t n_chunks = 0, max_vis = 0;
  const uint16_t* q_idx = nullptr;
  const float* w_heads = nullptr;
  const void* keys = nullptr;
  const uint8_t* key_scale = nullptr;
  const int64_t* pool_off = nullptr;
  const int32_t* seq_of_q = nullptr;
  const int32_t* n_vis = nullptr;
  float* scores = nullptr;
  int64_t ld = 0;
  uint32_t* flags = nullptr;
  // set: the scan leaves out the entries this step compresses (entries at or
  // above first_pos[b] / m of a sequence with tok_off[b+1] > tok_off[b]) and
  // the compress kernel scores them (CompressTail)
  const int64_t* new_first = nullptr;
  const int64_t* new_tok = nullptr;
  int m = 1;
  // 1: launched programmatically as a step's first kernel: wait for the
  // previous kernel of the stream before reading anything
  int wait_first = 0;
  unsigned long long* work = nullptr;  // [2] ticket counters, zero between launches
  // set: the hierarchical indexer's pool form. Row position p of query q is
  // entry (cand[q * cand_ld + (p >> cand_shift)] << cand_shift) | low bits;
  // n_pool[q] receives the number of pool entries below n_vis
  const int32_t* cand = nullptr;
  int cand_ld = 0;
  int cand_shift = 0;
  int32_t* n_pool = nullptr;
};
// pdl: launched programmatically after the step's compress kernel, which
// it waits for only before its CTAs exit (it reads nothing compress writes)
cudaError_t launch_index_score(cudaStream_t st, int num_sms, int idx_heads, int idx_fmt, IdxArgs a,
                               bool pdl = false);
// tensor-core form of the indexer for many queries per sequence (bf16 keys)
bool index_tc_suited(int idx_fp8, int n_query, int n_seq, int idx_heads);
cudaError_t launch_index_score_tc(cudaStream_t st, int num_sms, int idx_heads, int n_query, int n_seq,
                                  int64_t max_vis, const uint16_t* q_idx, const float* w_heads, const uint16_t* keys,
                                  const int64_t* pool_off, const int32_t* seq_of_q, const int32_t* n_vis,
                                  float* scores, int64_t ld, uint32_t* flags);
size_t topk_workspace_bytes(int n_query, int64_t max_vis);
// map_blocks set (rows of at most 16,384): row entry e is written as the
// entry index (map_blocks[q * map_ld + (e >> map_shift)] << map_shift) | low bits
// pdl: the one-launch forms start programmatically after the previous kernel
// of the stream (csa2_step's index scan) and wait for it before reading
cudaError_t launch_topk(cudaStream_t st, int n_query, const float* scores, int64_t ld, const int32_t* n_vis,
                        int64_t max_vis, int k, int32_t* out_idx, void* ws, int* n_launch,
                        const int32_t* map_blocks = nullptr, int map_ld = 0, int map_shift = 0, bool pdl = false);
size_t candidate_pool_workspace_bytes(int n_query, int64_t max_vis, int shift);
cudaError_t launch_candidate_pool(cudaStream_t st, int n_query, const float* scores, int64_t ld,
                                  const int32_t* n_vis, int64_t max_vis, int shift, int keep, int32_t* cand,
                                  void* ws, int* n_launch);
struct AttendPlan {
  int n_tiles;
  int ns;       // CTAs per query
  int tps;      // selected tiles per CTA
  int lead;     // tiles of a query's first CTA (the window tile and its tps selected tiles)
  int n_slots;  // partial slots per query (0: direct output)
  int ctas;     // CTAs of the persistent launch for many queries (one per SM)
};
int attend_num_tiles(int topk, bool has_idx);
// own_window: the window tile may take a CTA of its own (the workspace is
// sized for it, the larger plan)
AttendPlan attend_plan(int n_query, int topk, bool has_idx, int num_sms, bool own_window = true);
size_t attend_workspace_bytes(int n_query, const AttendPlan& pl);
cudaError_t launch_attend_main(cudaStream_t st, int kv_fmt, AttendParams p, const AttendPlan& pl, void* ws,
                               int* n_launch);
cudaError_t launch_attend_merge(cudaStream_t st, AttendParams p, const AttendPlan& pl, void* ws, int* n_launch);
cudaError_t launch_attend(cudaStream_t st, int num_sms, int kv_fmt, AttendParams p, void* ws, int* n_launch,
                          bool own_window = true);
// one CTA per query over the window tile (when with_window) and the selected
// tiles, writing the unnormalised partial (direct = 2)
cudaError_t launch_attend_partial(cudaStream_t st, int kv_fmt, AttendParams p, int with_window, int* n_launch);
// log-sum-exp combine of n_parts partials [n_parts][n_query] with the sink
cudaError_t launch_attend_combine(cudaStream_t st, int n_query, int n_parts, const float* part_o, const float* part_m,
                                  const float* part_l, const int64_t* q_pos, const float* sink, const RopeParams& rp,
                                  uint16_t* out, float* lse, int* n_launch);
// n_vis_shard[q] = clamp(n_vis[q] - lo, 0, hi - lo)
cudaError_t launch_shard_visible(cudaStream_t st, int n_query, const int32_t* n_vis, int64_t lo, int64_t hi,
                                 int32_t* n_vis_shard, int* n_launch);
// (score, lo + j) pairs of a shard's local selection; -1 entries give (-inf, -1)
cudaError_t launch_topk_pairs(cudaStream_t st, int n_query, const float* scores, int64_t ld, const int32_t* sel, int k,
                              int64_t index_base, float* pair_score, int32_t* pair_idx, int* n_launch);
// the k best of n_lists lists of (score, index) pairs [n_lists][n_query][k_in]
cudaError_t launch_topk_merge(cudaStream_t st, int n_query, int n_lists, int k_in, const float* pair_score,
                              const int32_t* pair_idx, int k, int32_t* out_idx, int* n_launch);
// one CTA waiting on an mbarrier nothing arrives at, for limit_ns (csa2_debug_wait_timeout)
cudaError_t launch_wait_probe(cudaStream_t st, uint32_t* flags, uint64_t limit_ns);

}  // namespace csa2
